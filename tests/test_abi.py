"""Host-side checks of the C ABI: the library builds, loads, exports every symbol the
header declares, and rejects bad arguments before touching the GPU.  No compute call
is made, so these run without a GPU."""
import ctypes
import os
import re

import pytest

from paged_attention_relative_gqa_gb300 import binding, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "inkling_attn.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(inkling_attn_\w+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_expected_entry_points():
    names = declared_functions()
    for n in ("inkling_attn_prefill", "inkling_attn_decode", "inkling_attn_workspace_bytes",
              "inkling_attn_workspace_init", "inkling_attn_read_device_error",
              "inkling_attn_status_string", "inkling_attn_version"):
        assert n in names
    assert set(names) <= set(binding.EXPORTED_SYMBOLS) | set(names)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in the header but not exported"
    assert lib.inkling_attn_version() >= 100


def test_status_strings(lib):
    for code in range(0, 8):
        s = binding.status_string(code)
        assert isinstance(s, str) and s
    assert binding.status_string(0) == "ok"


def good_params(**kw):
    base = dict(num_seqs=4, num_q_heads=64, num_kv_heads=8, head_dim=128, page_size=64,
                max_pages_per_seq=512, num_pages=2400, rel_extent=4096, window=-1,
                sm_scale=0.088)
    base.update(kw)
    return binding.make_params(**base)


def test_workspace_bytes_is_host_only_and_monotone(lib):
    a = binding.inkling_attn_workspace_bytes(good_params(), True)
    b = binding.inkling_attn_workspace_bytes(good_params(num_seqs=8), True)
    p = binding.inkling_attn_workspace_bytes(good_params(), False)
    assert a > 0 and b >= a and 0 < p <= a
    # decode partials: at least B * Hq * splits * D floats
    assert a >= 4 * 64 * 128 * 4


@pytest.mark.parametrize("bad,code", [
    (dict(num_q_heads=12, num_kv_heads=8), 2),     # non-divisible GQA: an error, not a mis-map
    (dict(head_dim=96), 2),
    (dict(page_size=48), 3),
    (dict(page_size=4), 3),
    (dict(rel_extent=0), 2),
    (dict(num_pages=0), 2),
])
def test_invalid_params_are_rejected_without_launch(lib, bad, code):
    params = good_params(**bad)
    assert binding.inkling_attn_workspace_bytes(params, True) == 0
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first
    r = lib.inkling_attn_decode(ctypes.byref(params), fake, fake, fake, fake, fake, fake, fake,
                                fake, 1 << 30, None)
    assert r == code
    r = lib.inkling_attn_prefill(ctypes.byref(params), fake, fake, 16, 64, fake, fake, fake, fake, fake,
                                 fake, fake, 1 << 30, None)
    assert r == code
    r = lib.inkling_attn_prefill_bf16bias(ctypes.byref(params), fake, fake, 16, 64, fake, fake, fake, fake,
                                          fake, fake, fake, 1 << 30, None)
    assert r == code


def test_bf16_bias_prefill_needs_16_byte_bias_rows(lib):
    ok = ctypes.c_void_p(1 << 20)
    # E a multiple of 4 but not of 8: bf16 rows are not 16-byte multiples
    params = good_params(rel_extent=4092)
    r = lib.inkling_attn_prefill_bf16bias(ctypes.byref(params), ok, ok, 16, 64, ok, ok, ok, ok, ok,
                                          ok, ok, 1 << 30, None)
    assert r == 2
    # bias base 8-byte but not 16-byte aligned (the fp32 entry only needs 4 bytes)
    params = good_params()
    odd = ctypes.c_void_p((1 << 20) + 8)
    r = lib.inkling_attn_prefill_bf16bias(ctypes.byref(params), ok, ok, 16, 64, ok, ok, ok, ok, odd,
                                          ok, ok, 1 << 30, None)
    assert r == 5


def test_null_and_misaligned_pointers_are_rejected(lib):
    params = good_params()
    ok = ctypes.c_void_p(1 << 20)
    r = lib.inkling_attn_decode(ctypes.byref(params), None, ok, ok, ok, ok, ok, ok, ok, 1 << 30, None)
    assert r == 1
    odd = ctypes.c_void_p((1 << 20) + 2)
    r = lib.inkling_attn_decode(ctypes.byref(params), odd, ok, ok, ok, ok, ok, ok, ok, 1 << 30, None)
    assert r == 5


def test_small_workspace_is_rejected(lib):
    params = good_params()
    ok = ctypes.c_void_p(1 << 20)
    need = binding.inkling_attn_workspace_bytes(params, True)
    r = lib.inkling_attn_decode(ctypes.byref(params), ok, ok, ok, ok, ok, ok, ok, ok, need - 256, None)
    assert r == 4
    r = lib.inkling_attn_read_device_error(ok, 16, None, ctypes.byref(ctypes.c_uint32()), 0)
    assert r == 4


def test_binding_refuses_cpu_tensors(lib):
    import torch
    from paged_attention_relative_gqa_gb300 import workloads as W
    prob = W.make_problem(num_q_heads=2, num_kv_heads=1, head_dim=64, page_size=16, rel_extent=8,
                          window=-1, q_lens=[1], seq_lens=[5], seed=0)
    with pytest.raises(ValueError):
        binding.inkling_attn_decode(binding.params_of(prob), prob.q, prob.k_cache, prob.v_cache,
                                    prob.block_table, prob.seq_lens, prob.rel_logits,
                                    torch.empty_like(prob.q), torch.empty(256, dtype=torch.uint8))


def _kv_call(lib, params, ks=4, *, k_new=None, w=None, st=None, ws_bytes=1 << 30, total_q=64):
    ok = ctypes.c_void_p(1 << 20)
    k_new = ok if k_new is None else k_new
    w = ok if w is None else w
    st = ok if st is None else st
    return lib.inkling_attn_kv_conv_write(ctypes.byref(params), k_new, ok, ok, total_q, ok, ok, w, ok, ks,
                                          st, ok, ok, ok, ok, ok, ok, ws_bytes, None)


def test_kv_conv_write_rejects_bad_arguments_without_launch(lib):
    params = good_params()
    assert _kv_call(lib, params, ks=0) == 2                      # kernel size below 1
    assert _kv_call(lib, params, ks=9) == 2                      # kernel size above 8
    assert _kv_call(lib, params, total_q=-1) == 2
    assert _kv_call(lib, params, k_new=ctypes.c_void_p(0)) == 1  # NULL input rows
    assert _kv_call(lib, params, st=ctypes.c_void_p(0)) == 1     # NULL state with ks > 1
    assert _kv_call(lib, params, k_new=ctypes.c_void_p((1 << 20) + 2)) == 5
    assert _kv_call(lib, params, w=ctypes.c_void_p((1 << 20) + 4)) == 5    # filters need 16 bytes
    assert _kv_call(lib, params, st=ctypes.c_void_p((1 << 20) + 8)) == 5
    assert _kv_call(lib, params, ws_bytes=16) == 4
    assert _kv_call(lib, good_params(head_dim=96)) == 2
    assert _kv_call(lib, good_params(page_size=12)) == 3


def test_kv_conv_write_kernel_size_one_needs_no_state(lib):
    """ks == 1 has no state: NULL state pointers pass validation; total_q == 0 launches
    nothing (B = 0 rows of state are also nothing), so the call returns without a GPU."""
    params = good_params(num_seqs=0)
    assert _kv_call(lib, params, ks=1, st=ctypes.c_void_p(0), total_q=0) == 0


def test_lowrank_bias_prefill_rejects_bad_rank_and_alignment(lib):
    ok = ctypes.c_void_p(1 << 20)
    params = good_params()
    for d in (0, 4, 12, 36, 72, 128):
        r = lib.inkling_attn_prefill_lowrank_bias(ctypes.byref(params), ok, ok, 16, 64, ok, ok, ok, ok, ok, ok, d,
                                                  ok, ok, 1 << 30, None)
        assert r == 2, d
    odd = ctypes.c_void_p((1 << 20) + 4)
    r = lib.inkling_attn_prefill_lowrank_bias(ctypes.byref(params), ok, ok, 16, 64, ok, ok, ok, ok, odd, ok, 64,
                                              ok, ok, 1 << 30, None)
    assert r == 5
    r = lib.inkling_attn_prefill_lowrank_bias(ctypes.byref(params), ok, ok, 16, 64, ok, ok, ok, ok, None, ok, 64,
                                              ok, ok, 1 << 30, None)
    assert r == 1
