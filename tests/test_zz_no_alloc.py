"""The allocation-free decode entry point (inkling_attn_decode_noalloc).

It exists for callers that cannot allocate device memory and therefore cannot pass the
workspace inkling_attn_decode needs; it uses a fixed 64 MiB device array inside the
library instead.  This file is collected last so that a run stopping at the first
failure has already run every other test; it passes alone in a fresh process too.
"""
import ctypes

import pytest
import torch

from paged_attention_relative_gqa_gb300 import binding, build
from paged_attention_relative_gqa_gb300 import workloads as W
from tests.parity import TOL_MAX_ABS, TOL_REL_RMS


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_rejects_a_workspace_need_beyond_its_scratch_without_launching():
    build.build()
    lib = binding.load_library()
    # 4096 sequences x 64 heads x many splits: far more than 64 MiB of partials
    params = binding.make_params(num_seqs=4096, num_q_heads=64, num_kv_heads=8, head_dim=128,
                                 page_size=64, max_pages_per_seq=4096, num_pages=1 << 20,
                                 rel_extent=4096, window=-1, sm_scale=0.088)
    assert binding.inkling_attn_workspace_bytes(params, True) > (64 << 20)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    r = lib.inkling_attn_decode_noalloc(ctypes.byref(params), fake, fake, fake, fake, fake, fake,
                                        fake, None)
    assert r == 4  # INK_ERR_WORKSPACE
    bad = binding.make_params(num_seqs=1, num_q_heads=12, num_kv_heads=8, head_dim=128, page_size=64,
                              max_pages_per_seq=4, num_pages=8, rel_extent=8, window=-1, sm_scale=1.0)
    r = lib.inkling_attn_decode_noalloc(ctypes.byref(bad), fake, fake, fake, fake, fake, fake, fake, None)
    assert r == 2  # INK_ERR_BAD_SHAPE


def _compare(a, b, label):
    diff = (a.float() - b.float())
    max_abs = diff.abs().max().item()
    rel_rms = (diff.norm() / b.float().norm()).item()
    print(f"{label}: {a.shape[0] * a.shape[1]} rows compared, max_abs {max_abs:.3e}, rel_rms {rel_rms:.3e}")
    assert torch.isfinite(a.float()).all()
    assert max_abs <= TOL_MAX_ABS and rel_rms <= TOL_REL_RMS


@pytest.mark.gpu
def test_noalloc_decode_matches_workspace_decode_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    lib = binding.load_library()
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev).cuda_stream
    problems = [W.swa_decode(dev, seed=2),
                W.make_problem(num_q_heads=16, num_kv_heads=2, head_dim=128, page_size=64,
                               rel_extent=4096, window=-1, q_lens=[1, 1, 1], seq_lens=[20000, 3, 9000],
                               seed=4, device=dev)]
    for i, prob in enumerate(problems):  # two calls in a row, different shapes
        params = binding.params_of(prob)
        ws = binding.alloc_workspace(params, True, dev)
        ref = torch.empty_like(prob.q)
        binding.inkling_attn_decode(params, prob.q, prob.k_cache, prob.v_cache, prob.block_table,
                                    prob.seq_lens, prob.rel_logits, ref, ws)
        got = torch.full_like(prob.q, float("nan"))
        r = lib.inkling_attn_decode_noalloc(ctypes.byref(params), _ptr(prob.q), _ptr(prob.k_cache),
                                            _ptr(prob.v_cache), _ptr(prob.block_table),
                                            _ptr(prob.seq_lens), _ptr(prob.rel_logits), _ptr(got),
                                            ctypes.c_void_p(stream))
        assert r == 0
        torch.cuda.synchronize()
        _compare(got, ref, f"noalloc call {i + 1} vs workspace decode")
