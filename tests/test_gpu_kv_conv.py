"""GPU parity of the K/V short convolution and paged write (inkling_attn_kv_conv_write)
against the fp64 oracle ``oracle/kv_conv.py``, through the C ABI.

Bar: every slot the step writes holds a value within  ulp_bf16(|y|) + ks * 2^-24 * mag
of the oracle's exact fp64 value y, where mag = sum_j |w_j x_j|: the kernel sums the ks
products in fp32 (at most ks roundings, each below 2^-24 of a partial sum bounded by mag)
and rounds once to bf16 (half an ulp of a value at most one binade above |y|).  Every
other slot of the pools keeps its bits (NaN pages included), and the carried state is
bit-exact (it is a copy).  Most slots also equal the oracle's own bf16 rounding; where
the products cancel, the fp32 error can move the result by more than one bf16 ulp of the
small result.
"""
import numpy as np
import pytest
import torch

import oracle.kv_conv as okc
from paged_attention_relative_gqa_gb300 import binding
from paged_attention_relative_gqa_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    yield
    torch.cuda.empty_cache()


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def run_gpu(step, ws=None):
    """One call; returns (k_cache, v_cache, state_k_out, state_v_out, device error)."""
    params = binding.make_params(num_seqs=step.num_seqs, num_q_heads=step.num_kv_heads,
                                 num_kv_heads=step.num_kv_heads, head_dim=step.head_dim,
                                 page_size=step.page_size, max_pages_per_seq=step.max_pages,
                                 num_pages=step.num_pages, rel_extent=1, window=-1, sm_scale=1.0)
    if ws is None:
        ws = binding.alloc_workspace(params, False, DEV)
    kc, vc = step.k_cache.clone(), step.v_cache.clone()
    sk, sv = torch.empty_like(step.state_k), torch.empty_like(step.state_v)
    has_state = step.kernel_size > 1
    binding.inkling_attn_kv_conv_write(params, step.k_new, step.v_new, step.cu_q_lens, step.seq_lens,
                                       step.block_table, step.w_k, step.w_v,
                                       step.state_k if has_state else None, step.state_v if has_state else None,
                                       sk if has_state else None, sv if has_state else None, kc, vc, ws)
    err = binding.inkling_attn_read_device_error(ws)
    return kc, vc, sk, sv, err


def written_mask(step, only=None):
    """[num_pages, Hkv, P] mask of the slots the step writes (requests in `only`, or all)."""
    P = step.page_size
    m = np.zeros((step.num_pages, P), bool)
    bt = step.block_table.cpu().numpy()
    for b, (n, L) in enumerate(zip(step.q_lens, step.seq_lens_list)):
        if only is not None and b not in only:
            continue
        for p in range(L - n, L):
            m[bt[b, p // P], p % P] = True
    return np.broadcast_to(m[:, None, :], (step.num_pages, step.num_kv_heads, P))


def bf16_ulp(y):
    e = np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -133)))
    return 2.0 ** (e - 7)


def check(step, got, label):
    kc, vc, sk, sv, err = got
    assert err == 0, f"{label}: device error {err:#x}"
    kw = step.oracle_kwargs()
    ref = okc.kv_conv_write(**kw)
    mask = written_mask(step)
    ks = step.kernel_size
    for name, ours_t, before, x, st, w, st_ours, st_ref in (
            ("k", kc, kw["k_cache_bits"], kw["k_new_bits"], kw["state_k_bits"], kw["w_k"], sk, ref[2]),
            ("v", vc, kw["v_cache_bits"], kw["v_new_bits"], kw["state_v_bits"], kw["w_v"], sv, ref[3])):
        ours = bits(ours_t)
        # untouched slots: exactly the old bits
        assert np.array_equal(ours[~mask], before[~mask]), f"{label} {name}: stray write"
        y, mag, page, slot, _ = okc.kv_conv_rows(x_bits=x, cu_q=kw["cu_q"], seq_lens=kw["seq_lens"],
                                                 block_table=kw["block_table"], page_size=kw["page_size"],
                                                 w=w, ks=ks, state_bits=st)
        rows = page >= 0
        got_v = okc.bf16_bits_to_f64(ours[page[rows], :, slot[rows], :])
        tol = bf16_ulp(y[rows]) + ks * 2.0 ** -24 * mag[rows]
        bad = ~(np.abs(got_v - y[rows]) <= tol)
        assert not bad.any(), (f"{label} {name}: {int(bad.sum())} slots outside the fp32 bound; worst excess "
                               f"{np.nanmax(np.abs(got_v - y[rows]) - tol):.3e}")
        want_bits = ref[0] if name == "k" else ref[1]
        same = (ours[mask] == want_bits[mask]).mean() if mask.any() else 1.0
        assert same > 0.99, f"{label} {name}: only {same:.4f} of slots equal the oracle's bf16 rounding"
        if ks > 1:
            assert np.array_equal(bits(st_ours), st_ref), f"{label}: state_{name} differs"


# (Hkv, D, P, ks, q_lens, seq_lens)
CASES = [
    (2, 64, 8, 4, [5, 1, 0, 9], [5, 20, 3, 30]),                  # empty request, decode row, P8
    (2, 128, 16, 1, [17, 3], [40, 3]),                            # ks 1: plain write, no state
    (1, 64, 8, 2, [1], [1]),                                      # one token, fresh request
    (4, 128, 64, 3, [130, 64, 1, 2], [200, 64, 900, 2]),          # runs crossing requests
    (16, 128, 64, 8, [7, 2, 33], [7, 500, 40]),                   # ks 8, n < ks - 1 (state shifts)
    (8, 64, 32, 5, [1] * 40, list(range(1, 41))),                 # decode-shaped: 40 one-token requests
    (3, 128, 256, 4, [600, 3, 1000], [600, 1000, 3000]),          # P256, long prompts (runs of 8)
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_kv_conv_write_matches_oracle(case):
    Hkv, D, P, ks, ql, sl = CASES[case]
    step = W.make_kv_step(num_kv_heads=Hkv, head_dim=D, page_size=P, kernel_size=ks, q_lens=ql,
                          seq_lens=sl, seed=400 + case, device=DEV)
    check(step, run_gpu(step), f"kv case {CASES[case]}")


# Steps with enough new rows for the staged (shared-memory ring) kernel: at least one
# tile of K and one of V per SM (tiles hold about 32 KB of new rows, at most 32 tokens).
STAGED = [
    (8, 128, 64, 4, [1500, 1, 2, 700, 1], [1500, 5000, 3, 900, 64]),   # tiles cut requests, n < ks - 1
    (16, 128, 64, 8, [3000, 5, 1], [3000, 40, 100]),                    # 8-token tiles, ks 8
    (32, 128, 16, 2, [2000, 300], [2100, 300]),                         # 512 vectors per row, 4-token tiles
    (4, 64, 8, 1, [5000], [5000]),                                      # ks 1
    (2, 64, 32, 3, [1] * 300 + [4000], list(range(50, 350)) + [4000]),  # 300 one-row requests, then a prompt
]


@pytest.mark.parametrize("case", range(len(STAGED)))
def test_kv_conv_write_staged_matches_oracle(case):
    Hkv, D, P, ks, ql, sl = STAGED[case]
    step = W.make_kv_step(num_kv_heads=Hkv, head_dim=D, page_size=P, kernel_size=ks, q_lens=ql,
                          seq_lens=sl, seed=500 + case, device=DEV)
    check(step, run_gpu(step), f"kv staged case {case}")


def test_kv_conv_write_staged_reports_bad_pages():
    step = W.make_kv_step(num_kv_heads=8, head_dim=128, page_size=64, kernel_size=4, q_lens=[2000, 1500],
                          seq_lens=[2000, 1600], seed=9, device=DEV)
    bt = step.block_table.clone()
    bt[1, 10] = -3                           # positions 640..703 of request 1
    step.block_table = bt
    kc, vc, sk, sv, err = run_gpu(step)
    assert err == binding.DEVERR_PAGE_OUT_OF_RANGE
    keep = ~written_mask(step, only=(0,))
    # request 0 is written in full; request 1 everywhere but page slot 10
    m1 = np.zeros_like(keep)
    P = step.page_size
    bt_np = bt.cpu().numpy()
    for p in range(100, 1600):
        if p // P != 10:
            m1[bt_np[1, p // P], :, p % P] = True
    keep &= ~m1
    assert np.array_equal(bits(kc)[keep], bits(step.k_cache)[keep])
    assert np.array_equal(bits(vc)[keep], bits(step.v_cache)[keep])


def test_kv_conv_write_global_prefill_full_size():
    """4 x 8192 fresh prompts, 8 KV heads, ks 4: every written slot and the state."""
    step = W.kv_prefill_global(DEV)
    check(step, run_gpu(step), "kv_prefill_global")


def test_kv_conv_write_swa_decode_full_size():
    step = W.kv_decode_swa(DEV)
    check(step, run_gpu(step), "kv_decode_swa")


def test_kv_conv_two_steps_equal_one():
    """A prompt written in two steps, the state of the first fed to the second, leaves
    the pools and the final state bit-identical to one step over all of it."""
    Hkv, D, P, ks = 4, 128, 16, 4
    n = [37, 5, 64]
    m = [20, 1, 60]
    whole = W.make_kv_step(num_kv_heads=Hkv, head_dim=D, page_size=P, kernel_size=ks, q_lens=n,
                           seq_lens=[40, 5, 200], seed=77, device=DEV)
    kc_w, vc_w, sk_w, sv_w, err = run_gpu(whole)
    assert err == 0
    cu = whole.cu_q_lens.cpu().tolist()
    idx1 = torch.cat([torch.arange(cu[b], cu[b] + m[b]) for b in range(3)]).to(DEV)
    idx2 = torch.cat([torch.arange(cu[b] + m[b], cu[b + 1]) for b in range(3)]).to(DEV)

    def cu_of(lens):
        c = torch.zeros(len(lens) + 1, dtype=torch.int32)
        c[1:] = torch.cumsum(torch.tensor(lens), 0)
        return c.to(DEV)

    import dataclasses
    s1 = dataclasses.replace(whole, q_lens=m, k_new=whole.k_new[idx1].contiguous(),
                             v_new=whole.v_new[idx1].contiguous(), cu_q_lens=cu_of(m),
                             seq_lens_list=[L - a + b for L, a, b in zip(whole.seq_lens_list, n, m)])
    s1.seq_lens = torch.tensor(s1.seq_lens_list, dtype=torch.int32, device=DEV)
    k1, v1, sk1, sv1, err = run_gpu(s1)
    assert err == 0
    rest = [a - b for a, b in zip(n, m)]
    s2 = dataclasses.replace(whole, q_lens=rest, k_new=whole.k_new[idx2].contiguous(),
                             v_new=whole.v_new[idx2].contiguous(), cu_q_lens=cu_of(rest),
                             state_k=sk1, state_v=sv1, k_cache=k1, v_cache=v1)
    k2, v2, sk2, sv2, err = run_gpu(s2)
    assert err == 0
    for a, b in ((k2, kc_w), (v2, vc_w), (sk2, sk_w), (sv2, sv_w)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_kv_conv_write_repeat_is_bitwise_stable():
    step = W.make_kv_step(num_kv_heads=8, head_dim=128, page_size=64, kernel_size=4, q_lens=[300, 1, 77],
                          seq_lens=[300, 1000, 100], seed=91, device=DEV)
    a = run_gpu(step)
    b = run_gpu(step)
    for x, y in zip(a[:4], b[:4]):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_kv_conv_write_reports_bad_pages_and_lengths_without_writing():
    """A block-table entry outside the pool and a request with more new rows than history
    set their error bits; their rows are skipped and nothing else changes."""
    step = W.make_kv_step(num_kv_heads=2, head_dim=64, page_size=8, kernel_size=4, q_lens=[4, 3, 6],
                          seq_lens=[20, 9, 6], seed=5, device=DEV)
    bt = step.block_table.clone()
    bt[0, 2] = step.num_pages + 100          # positions 16..19 of request 0 (its 4 new rows)
    step.block_table = bt
    kc, vc, sk, sv, err = run_gpu(step)
    assert err == binding.DEVERR_PAGE_OUT_OF_RANGE
    keep = ~written_mask(step, only=(1, 2))      # request 0 writes nothing
    assert np.array_equal(bits(kc)[keep], bits(step.k_cache)[keep])
    assert np.array_equal(bits(vc)[keep], bits(step.v_cache)[keep])
    # request 1: claim 3 new rows over a history of 2
    step2 = W.make_kv_step(num_kv_heads=2, head_dim=64, page_size=8, kernel_size=4, q_lens=[4, 3, 6],
                           seq_lens=[20, 9, 6], seed=6, device=DEV)
    step2.seq_lens = torch.tensor([20, 2, 6], dtype=torch.int32, device=DEV)
    kc2, vc2, _, _, err2 = run_gpu(step2)
    assert err2 == binding.DEVERR_QLEN_EXCEEDS_KV
    keep = ~written_mask(step2, only=(0, 2))     # request 1 writes nothing
    assert np.array_equal(bits(kc2)[keep], bits(step2.k_cache)[keep])


def test_kv_conv_write_captures_in_a_cuda_graph():
    step = W.kv_decode_swa(DEV)
    params = binding.make_params(num_seqs=step.num_seqs, num_q_heads=step.num_kv_heads,
                                 num_kv_heads=step.num_kv_heads, head_dim=step.head_dim,
                                 page_size=step.page_size, max_pages_per_seq=step.max_pages,
                                 num_pages=step.num_pages, rel_extent=1, window=-1, sm_scale=1.0)
    ws = binding.alloc_workspace(params, False, DEV)
    kc, vc = step.k_cache.clone(), step.v_cache.clone()
    sk, sv = torch.empty_like(step.state_k), torch.empty_like(step.state_v)

    def call():
        binding.inkling_attn_kv_conv_write(params, step.k_new, step.v_new, step.cu_q_lens, step.seq_lens,
                                           step.block_table, step.w_k, step.w_v, step.state_k, step.state_v,
                                           sk, sv, kc, vc, ws)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    kc.copy_(step.k_cache)
    vc.copy_(step.v_cache)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    g.replay()
    torch.cuda.synchronize()
    assert binding.inkling_attn_read_device_error(ws) == 0
    check(step, (kc, vc, sk, sv, 0), "graph replay")
