"""Failure detection by status, not by fault: a pipeline wait that runs out.

Every mbarrier wait in the kernels is bounded.  inkling_attn_set_wait_limit_ns(0) makes any
wait that finds its data not yet ready give up at once, which is the timeout path with no
fault and no hang: the kernel records INK_DEVERR_WAIT_TIMEOUT in the workspace error word,
stops issuing copies and tensor-core operations, waits for those already issued, and
returns.  Rows it did not finish are left as they were (here: zeros), so the output stays
finite.  With the limit restored, the same calls on the same device pass parity, i.e. the
context is still usable.  (The failure detection of "Inkling attn backend cleanup fake
registry", TensorRT-LLM PR #17860: the epoch-checked ready flag detects stale decode metadata
rather than reading it; here the kernels report a stalled pipeline rather than hanging.)
"""
import numpy as np
import pytest
import torch

from paged_attention_relative_gqa_gb300 import binding
from paged_attention_relative_gqa_gb300 import workloads as W
from tests.parity import compare, oracle_full
from tests.test_gpu_kv_conv import check as kv_check, run_gpu as run_kv

pytestmark = pytest.mark.gpu
DEV = "cuda"
DEFAULT_LIMIT_NS = 2_000_000_000


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    yield
    binding.inkling_attn_set_wait_limit_ns(DEFAULT_LIMIT_NS)
    torch.cuda.empty_cache()


def attention_cases():
    """Problems large enough that their pipelines certainly wait: a decode, the head-pair
    prefill with fp32 and with bf16 bias, and the low-rank-bias prefill."""
    dec = W.make_problem(num_q_heads=16, num_kv_heads=4, head_dim=128, page_size=64, rel_extent=512, window=512,
                         q_lens=[1] * 24, seq_lens=[1500 + 97 * i for i in range(24)], seed=31, device=DEV)
    pre = W.make_problem(num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=64, rel_extent=1024, window=-1,
                         q_lens=[700, 300], seq_lens=[700, 900], seed=32, device=DEV)
    pre_bf = W.make_problem(num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=64, rel_extent=1024, window=-1,
                            q_lens=[700, 300], seq_lens=[700, 900], seed=33, device=DEV, bias_dtype=torch.bfloat16)
    pre_lr = W.make_problem(num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=64, rel_extent=1024, window=-1,
                            q_lens=[700, 300], seq_lens=[700, 900], seed=34, device=DEV, lowrank_d=64)
    return [("decode", dec), ("prefill fp32 bias", pre), ("prefill bf16 bias", pre_bf), ("prefill low-rank bias", pre_lr)]


def run_once(prob):
    params = binding.params_of(prob)
    ws = binding.alloc_workspace(params, True, prob.q.device)
    out = torch.zeros_like(prob.q)
    binding.run(prob, out=out, workspace=ws)
    err = binding.inkling_attn_read_device_error(ws)
    return out, err


def kv_step():
    # prefill-sized: the staged K/V kernel (its bulk copies and stage rings) runs
    return W.make_kv_step(num_kv_heads=8, head_dim=128, page_size=64, kernel_size=4, q_lens=[1024] * 4,
                          seq_lens=[1024] * 4, seed=35, device=DEV)


def test_waits_that_run_out_report_a_timeout_and_the_device_recovers():
    cases = attention_cases()
    step = kv_step()
    binding.inkling_attn_set_wait_limit_ns(0)
    try:
        for label, prob in cases:
            out, err = run_once(prob)
            print(f"{label}: error word {err:#x} with a zero wait limit")
            assert err & binding.DEVERR_WAIT_TIMEOUT, f"{label}: no timeout recorded"
            assert torch.isfinite(out.float()).all(), f"{label}: non-finite output after the timeout"
        err = run_kv(step)[4]
        print(f"K/V write: error word {err:#x} with a zero wait limit")
        assert err & binding.DEVERR_WAIT_TIMEOUT, "K/V write: no timeout recorded"
    finally:
        binding.inkling_attn_set_wait_limit_ns(DEFAULT_LIMIT_NS)
    torch.cuda.synchronize()
    # the same calls on the same device, with the default limit: no error, oracle parity
    for label, prob in cases:
        out, err = run_once(prob)
        assert err == 0, f"{label}: error word {err:#x} after the limit was restored"
        compare(out.float().cpu().numpy(), oracle_full(prob), f"{label} after the timeout test")
    kv_check(step, run_kv(step), "K/V write after the timeout test")
