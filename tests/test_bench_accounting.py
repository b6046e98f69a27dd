"""The bench's algorithmic work (the numerators of its roofline fractions) against values
worked out by hand on tiny problems."""
import bench
from paged_attention_relative_gqa_gb300 import workloads as W


def test_decode_bytes_by_hand():
    # B 2, Hq 4, Hkv 2, D 8, E 5, window 3, page 4; lengths 6 and 2, one new token each.
    # p = 5 sees keys 3..5 (3 keys, pages 0 and 1); p = 1 sees keys 0..1 (2 keys, page 0).
    prob = W.make_problem(num_q_heads=4, num_kv_heads=2, head_dim=8, page_size=4, rel_extent=5, window=3,
                          q_lens=[1, 1], seq_lens=[6, 2], seed=0)
    kv = (3 + 2) * 2 * 8 * 2 * 2            # visible keys x Hkv x D x bf16 x (K and V)
    bias = 4 * 3 * 4 + 4 * 2 * 4            # Hq x min(|Vis|, E) x fp32
    pages = (2 + 1) * 4                     # block-table entries read
    q_out = 2 * 4 * 8 * 2 * 2               # q and out rows
    lens = 2 * 4                            # seq_lens
    assert bench.decode_bytes(prob) == kv + bias + pages + q_out + lens == 676


def test_prefill_work_by_hand():
    # one sequence of 3 new tokens (positions 0..2), causal, E 2: visible keys 1, 2, 3
    prob = W.make_problem(num_q_heads=2, num_kv_heads=1, head_dim=8, page_size=8, rel_extent=2, window=-1,
                          q_lens=[3], seq_lens=[3], seed=0)
    flops, nbytes, bias_flops = bench.prefill_work(prob)
    assert flops == (1 + 2 + 3) * 4 * 8 * 2          # 4 D per visible (row, key, head)
    bias = (1 + 2 + 2) * 2 * 4                        # min(|Vis|, E) buckets x Hq x fp32
    kv = 3 * 1 * 8 * 2 * 2
    qo = 3 * 2 * 8 * 2 * 2
    assert nbytes == bias + kv + qo and bias_flops == 0
    # the same shape with the bias in low-rank form (d_rel 16): r and the projection are read
    # once, and every bias bucket used costs 2 d_rel FLOPs
    lr = W.make_problem(num_q_heads=2, num_kv_heads=1, head_dim=8, page_size=8, rel_extent=2, window=-1,
                        q_lens=[3], seq_lens=[3], seed=0, lowrank_d=16)
    flops2, nbytes2, bias_flops2 = bench.prefill_work(lr)
    assert flops2 == flops
    assert nbytes2 == 3 * 2 * 16 * 2 + 2 * 16 * 2 + kv + qo
    assert bias_flops2 == (1 + 2 + 2) * 2 * 2 * 16


def test_kv_write_bytes_by_hand():
    # two requests: 5 new rows at positions 3..7 (pages 0 and 1 of page size 4), and one
    # decode row at position 9 (page 2); Hkv 2, D 8, kernel size 3
    step = W.make_kv_step(num_kv_heads=2, head_dim=8, page_size=4, kernel_size=3, q_lens=[5, 1],
                          seq_lens=[8, 10], seed=0)
    row = 2 * 8 * 2
    expect = 2 * 6 * row * 2                 # new rows read, cache rows written (K and V)
    expect += 2 * 2 * 2 * 2 * row            # state rows read and written: K/V x in/out x B x (ks - 1)
    expect += 2 * 2 * 8 * 3 * 4              # filters
    expect += (2 * 2 + 1) * 4                # cu_q_lens and seq_lens
    expect += (2 + 1) * 4                    # table entries of the pages written
    assert bench.kv_write_bytes(step) == expect
