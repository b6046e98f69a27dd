"""GPU parity of the prefill with the bias in low-rank form
(inkling_attn_prefill_lowrank_bias): the kernel computes every bias tile from r and the
transposed projection; the oracle builds the whole bias tensor in fp64 (``oracle/lowrank.py``)
and runs the attention oracle on it.  Tolerances are those of every prefill."""
import pytest
import torch

from paged_attention_relative_gqa_gb300 import binding
from paged_attention_relative_gqa_gb300 import workloads as W
from tests.parity import compare, gpu_rows, oracle_full, oracle_rows, run_gpu, sampled_check

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    yield
    torch.cuda.empty_cache()


def test_lowrank_bias_swa_prefill_tiny_every_row():
    prob = W.make_problem(num_q_heads=8, num_kv_heads=2, head_dim=64, page_size=16, rel_extent=512,
                          window=512, q_lens=[1024], seq_lens=[1024], seed=0, device=DEV, lowrank_d=64)
    out, err = run_gpu(prob)
    assert err == 0
    compare(out.float().cpu().numpy(), oracle_full(prob), "low-rank bias swa_prefill_tiny")


# (Hq, Hkv, D, P, W, E, q_lens, seq_lens, d_rel)
# (the last two include items whose bias tiles are their last few tiles: long prefixes, E 7,
# and 4096 with a 5000-key history)
EDGE_LR = [
    (8, 8, 128, 16, 5, 16, [33, 1, 64], [33, 2, 300], 64),        # MHA, tiny window, cached prefix
    (16, 1, 128, 32, 64, 600, [65, 129], [100, 129], 64),         # G16, window == tile
    (8, 2, 128, 256, 512, 512, [300, 1], [1500, 777], 64),        # P256, SWA
    (8, 2, 64, 8, -1, 7, [1, 5, 70], [1, 40, 200], 64),           # P8, D64, E7 (clamp)
    (4, 4, 128, 64, -1, 1, [200], [300], 64),                     # E1: every key clamped
    (8, 2, 128, 64, -1, 4096, [700, 0, 130], [5000, 3, 130], 64), # long cached prefix, empty row
    (8, 2, 128, 64, 512, 512, [300, 1], [1500, 777], 32),         # d_rel 32 (zero columns 32-63)
    (8, 4, 64, 16, -1, 100, [150, 40], [150, 300], 16),           # d_rel 16, D64, P16
    (16, 2, 128, 64, -1, 1024, [257], [900], 48),                 # d_rel 48
]


@pytest.mark.parametrize("case", range(len(EDGE_LR)))
def test_lowrank_bias_edge_shapes(case):
    Hq, Hkv, D, P, Wn, E, ql, sl, d = EDGE_LR[case]
    prob = W.make_problem(num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=P, rel_extent=E,
                          window=Wn, q_lens=ql, seq_lens=sl, seed=600 + case, device=DEV,
                          max_pages=max(-(-L // P) for L in sl) + 3, lowrank_d=d)
    out, err = run_gpu(prob)
    assert err == 0
    compare(out.float().cpu().numpy(), oracle_full(prob), f"low-rank bias edge prefill {EDGE_LR[case]}")


@pytest.mark.parametrize("d_rel", [64, 32])
def test_lowrank_bias_with_std4_bias(d_rel):
    """A bias of standard deviation 4 (the scores are dominated by it): the tile's bias is
    held in fp16 on its way to the fp32 score, so this is where that rounding would show."""
    prob = W.make_problem(num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=64, rel_extent=1024,
                          window=-1, q_lens=[700, 300], seq_lens=[700, 900], seed=88 + d_rel, device=DEV,
                          rel_std=4.0, lowrank_d=d_rel)
    out, err = run_gpu(prob)
    assert err == 0
    compare(out.float().cpu().numpy(), oracle_full(prob), f"low-rank bias, std 4, d_rel {d_rel}")


@pytest.mark.parametrize("std,d_rel", [(4.0, 64), (0.5, 64), (4.0, 32)])
def test_lowrank_bias_error_is_that_of_the_fp32_bias(std, d_rel):
    """The bias tile passes through fp16 in the low-rank path (fp32 products, rounded to fp16
    in the ring, back to fp32 for the score).  Against the fp64 oracle its error must be no
    larger than the fp32-bias entry's on the same bias (built in fp64, rounded to fp32): the
    budget goes to the bf16 P and output, which both paths share, not to the fp16 step."""
    import numpy as np
    prob = W.make_problem(num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=64, rel_extent=1024,
                          window=-1, q_lens=[700, 300], seq_lens=[700, 900], seed=88 + d_rel, device=DEV,
                          rel_std=std, lowrank_d=d_rel)
    ref = oracle_full(prob)
    a, err_a = run_gpu(prob)
    mat = (prob.r.double().reshape(-1, d_rel) @ prob.rel_proj_t.double().t()).float()
    prob.r, prob.rel_proj_t, prob.rel_logits = None, None, mat.reshape(prob.total_q, prob.num_q_heads, -1).contiguous()
    b, err_b = run_gpu(prob)
    assert err_a == 0 and err_b == 0
    ea, eb = a.float().cpu().numpy() - ref, b.float().cpu().numpy() - ref
    ma, mb = float(np.abs(ea).max()), float(np.abs(eb).max())
    ra, rb = float(np.linalg.norm(ea) / np.linalg.norm(ref)), float(np.linalg.norm(eb) / np.linalg.norm(ref))
    print(f"std {std} d_rel {d_rel}: low-rank max_abs {ma:.3e} rel_rms {ra:.3e}; fp32 bias max_abs {mb:.3e} rel_rms {rb:.3e}")
    assert ma <= 1.1 * mb + 1e-3 and ra <= 1.1 * rb + 1e-4


def test_lowrank_bias_matches_the_materialised_bias_entry():
    """The low-rank entry against the fp32 entry fed rel = r x proj (built in fp32 by a
    library GEMM): the same attention up to the rounding of the bias (fp16 in the low-rank
    path), the summation order of each kernel and the bf16 output."""
    prob = W.mixed_layer("swa", 0, DEV)[0]
    lr = W.make_problem(num_q_heads=prob.num_q_heads, num_kv_heads=prob.num_kv_heads, head_dim=prob.head_dim,
                        page_size=prob.page_size, rel_extent=prob.rel_extent, window=prob.window,
                        q_lens=prob.q_lens, seq_lens=prob.seq_lens_list, seed=77, device=DEV, lowrank_d=64)
    a, err_a = run_gpu(lr)
    mat = (lr.r.float().reshape(-1, 64) @ lr.rel_proj_t.float().t()).reshape(lr.total_q, lr.num_q_heads, -1)
    r_saved, p_saved = lr.r, lr.rel_proj_t
    lr.r, lr.rel_proj_t, lr.rel_logits = None, None, mat.contiguous()
    b, err_b = run_gpu(lr)
    assert err_a == 0 and err_b == 0
    d = a.float() - b.float()
    diff = d.abs().max().item()
    rel = (d.norm() / b.float().norm()).item()
    # Two kernels with different fp32 summation orders (the materialised bias runs the
    # head-pair prefill), each within max-abs 2e-2 and relative RMS 5e-3 of the fp64 oracle:
    # their difference is held to the same bounds.
    assert diff <= 2e-2 and rel <= 5e-3, f"low-rank vs materialised bias: max diff {diff}, rel RMS {rel}"
    lr.r, lr.rel_proj_t = r_saved, p_saved


def test_lowrank_bias_global_prefill_sampled_rows_and_repeats():
    prob = W.global_prefill_lowrank(DEV)
    out, err = run_gpu(prob)
    assert err == 0
    sampled_check(prob, out, 46, "low-rank bias global_prefill (4x8192, sampled)")
    again, _ = run_gpu(prob)
    assert torch.equal(out, again)
    del prob, out, again
    torch.cuda.empty_cache()


def test_lowrank_bias_with_q_and_out_only_16_byte_aligned():
    """q and out 16-byte aligned but not 32 (the C ABI asks 16): the output rows then go out
    in 128-bit stores instead of 256-bit ones, with the same bits."""
    from tests.test_gpu_parity import _at_16_byte_offset
    from tests.parity import bits
    import numpy as np
    prob = W.make_problem(num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=64, rel_extent=512,
                          window=-1, q_lens=[300, 129], seq_lens=[700, 129], seed=41, device=DEV, lowrank_d=64)
    ref, _ = run_gpu(prob)
    q_aligned = prob.q
    prob.q = _at_16_byte_offset(q_aligned)
    params = binding.params_of(prob)
    ws = binding.alloc_workspace(params, True, prob.q.device)
    out = _at_16_byte_offset(torch.full_like(prob.q, float("nan")))
    binding.run(prob, out=out, workspace=ws)
    assert binding.inkling_attn_read_device_error(ws) == 0
    assert np.array_equal(bits(out), bits(ref))
    prob.q = q_aligned
