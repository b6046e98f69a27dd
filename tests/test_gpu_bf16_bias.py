"""GPU parity of the bf16-bias prefill (inkling_attn_prefill_bf16bias).

The problems carry the same seeded bias rounded to bf16; the oracle reads those rounded
values (widened exactly), so the tolerances are the ones of the fp32-bias path.  The
bf16 and fp32 entry points fed the same bias values must agree bit for bit: only the
element type of the staged bias differs between them.
"""
import pytest
import torch

from paged_attention_relative_gqa_gb300 import binding
from paged_attention_relative_gqa_gb300 import workloads as W
from tests.parity import compare, gpu_rows, oracle_full, oracle_rows, run_gpu, sampled_check

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF16 = torch.bfloat16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    yield
    torch.cuda.empty_cache()


def test_bf16_bias_swa_prefill_tiny_every_row():
    prob = W.make_problem(num_q_heads=8, num_kv_heads=2, head_dim=64, page_size=16, rel_extent=512,
                          window=512, q_lens=[1024], seq_lens=[1024], seed=0, device=DEV, bias_dtype=BF16)
    assert prob.rel_logits.dtype == BF16
    out, err = run_gpu(prob)
    assert err == 0
    compare(out.float().cpu().numpy(), oracle_full(prob), "bf16 bias swa_prefill_tiny")


# (Hq, Hkv, D, P, W, E, q_lens, seq_lens): E a multiple of 8
EDGE_BF16 = [
    (8, 8, 128, 16, 5, 16, [33, 1, 64], [33, 2, 300]),        # MHA, tiny window, cached prefix
    (16, 1, 128, 32, 64, 600, [65, 129], [100, 129]),         # G16, window == tile
    (8, 2, 128, 256, 512, 512, [300, 1], [1500, 777]),        # P256, SWA
    (8, 2, 64, 8, -1, 8, [1, 5, 70], [1, 40, 200]),           # P8, D64, E8 (clamp)
]


@pytest.mark.parametrize("case", range(len(EDGE_BF16)))
def test_bf16_bias_edge_shapes(case):
    Hq, Hkv, D, P, Wn, E, ql, sl = EDGE_BF16[case]
    prob = W.make_problem(num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=P, rel_extent=E,
                          window=Wn, q_lens=ql, seq_lens=sl, seed=300 + case, device=DEV,
                          max_pages=max(-(-L // P) for L in sl) + 3, bias_dtype=BF16)
    out, err = run_gpu(prob)
    assert err == 0
    compare(out.float().cpu().numpy(), oracle_full(prob), f"bf16 bias edge prefill {EDGE_BF16[case]}")


def test_bf16_bias_equals_fp32_bias_with_the_same_values():
    prob = W.mixed_layer("swa", 0, DEV)[0]
    prob.rel_logits = prob.rel_logits.to(BF16)
    a, err_a = run_gpu(prob)
    prob.rel_logits = prob.rel_logits.float()   # the same values, fp32 entry point
    b, err_b = run_gpu(prob)
    assert err_a == 0 and err_b == 0
    assert torch.equal(a, b)


def test_bf16_bias_global_prefill_sampled_rows_and_repeats():
    prob = W.global_prefill(DEV, bias_dtype=BF16)
    out, err = run_gpu(prob)
    assert err == 0
    sampled_check(prob, out, 45, "bf16 bias global_prefill (4x8192, sampled)")
    again, _ = run_gpu(prob)
    assert torch.equal(out, again)
    del prob, out, again
    torch.cuda.empty_cache()
