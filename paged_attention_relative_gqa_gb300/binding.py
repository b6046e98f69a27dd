"""ctypes binding of ``libinkling_attn.so`` (the C ABI in ``include/inkling_attn.h``).

Argument marshalling only: every step of the attention runs in the library's CUDA
kernels.  Functions keep the C names and argument order; tensors are passed by device
pointer after checking device, dtype, contiguity and shape.  There is no fallback: if
the library is missing or a call returns an error status, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

_lib = None

INK_OK = 0
STATUS_NAMES = {0: "INK_OK", 1: "INK_ERR_NULL_PTR", 2: "INK_ERR_BAD_SHAPE",
                3: "INK_ERR_BAD_PAGE_SIZE", 4: "INK_ERR_WORKSPACE", 5: "INK_ERR_ALIGNMENT",
                6: "INK_ERR_CUDA", 7: "INK_ERR_TOO_LARGE"}
DEVERR_PAGE_OUT_OF_RANGE = 0x1
DEVERR_QLEN_EXCEEDS_KV = 0x2
DEVERR_WAIT_TIMEOUT = 0x4
DEVERR_QLEN_EXCEEDS_MAX = 0x8
DEVERR_BAD_ROWS = 0x10

EXPORTED_SYMBOLS = ("inkling_attn_workspace_bytes", "inkling_attn_workspace_init",
                    "inkling_attn_prefill", "inkling_attn_prefill_bf16bias",
                    "inkling_attn_prefill_lowrank_bias", "inkling_attn_decode",
                    "inkling_attn_decode_noalloc", "inkling_attn_kv_conv_write",
                    "inkling_attn_read_device_error", "inkling_attn_status_string",
                    "inkling_attn_version", "inkling_attn_set_wait_limit_ns")


class InkError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} ({status_string(code)})")


class ink_attn_params_t(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("max_pages_per_seq", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("rel_extent", ctypes.c_int32),
                ("window", ctypes.c_int32), ("sm_scale", ctypes.c_float)]


def library_path() -> str:
    return _build.LIB


def load_library(path: Optional[str] = None):
    """Load the CUDA library (no build, no fallback: a missing library is an error)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or library_path()
    if not os.path.exists(p):
        raise RuntimeError(f"libinkling_attn.so not found at {p}; build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(p)
    V, S, I32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32
    PP = ctypes.POINTER(ink_attn_params_t)
    lib.inkling_attn_workspace_bytes.argtypes = [PP, ctypes.c_int]
    lib.inkling_attn_workspace_bytes.restype = S
    lib.inkling_attn_workspace_init.argtypes = [V, S, V]
    lib.inkling_attn_workspace_init.restype = ctypes.c_int
    lib.inkling_attn_prefill.argtypes = [PP, V, V, I32, I32, V, V, V, V, V, V, V, S, V]
    lib.inkling_attn_prefill.restype = ctypes.c_int
    lib.inkling_attn_prefill_bf16bias.argtypes = [PP, V, V, I32, I32, V, V, V, V, V, V, V, S, V]
    lib.inkling_attn_prefill_bf16bias.restype = ctypes.c_int
    lib.inkling_attn_prefill_lowrank_bias.argtypes = [PP, V, V, I32, I32, V, V, V, V, V, V, I32, V, V, S, V]
    lib.inkling_attn_prefill_lowrank_bias.restype = ctypes.c_int
    lib.inkling_attn_decode.argtypes = [PP, V, V, V, V, V, V, V, V, S, V]
    lib.inkling_attn_decode.restype = ctypes.c_int
    lib.inkling_attn_decode_noalloc.argtypes = [PP, V, V, V, V, V, V, V, V]
    lib.inkling_attn_decode_noalloc.restype = ctypes.c_int
    lib.inkling_attn_kv_conv_write.argtypes = [PP, V, V, V, I32, V, V, V, V, I32, V, V, V, V, V, V, V, S, V]
    lib.inkling_attn_kv_conv_write.restype = ctypes.c_int
    lib.inkling_attn_read_device_error.argtypes = [V, S, V, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]
    lib.inkling_attn_read_device_error.restype = ctypes.c_int
    lib.inkling_attn_status_string.argtypes = [ctypes.c_int]
    lib.inkling_attn_status_string.restype = ctypes.c_char_p
    lib.inkling_attn_version.argtypes = []
    lib.inkling_attn_version.restype = I32
    lib.inkling_attn_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.inkling_attn_set_wait_limit_ns.restype = None
    if path is None:
        _lib = lib
    return lib


def status_string(code: int) -> str:
    return load_library().inkling_attn_status_string(int(code)).decode()


def make_params(*, num_seqs, num_q_heads, num_kv_heads, head_dim, page_size,
                max_pages_per_seq, num_pages, rel_extent, window, sm_scale) -> ink_attn_params_t:
    return ink_attn_params_t(int(num_seqs), int(num_q_heads), int(num_kv_heads), int(head_dim),
                             int(page_size), int(max_pages_per_seq), int(num_pages),
                             int(rel_extent), int(window), float(sm_scale))


def params_of(prob) -> ink_attn_params_t:
    """Params for a ``workloads.Problem``."""
    return make_params(num_seqs=prob.num_seqs, num_q_heads=prob.num_q_heads,
                       num_kv_heads=prob.num_kv_heads, head_dim=prob.head_dim,
                       page_size=prob.page_size, max_pages_per_seq=prob.max_pages,
                       num_pages=prob.num_pages, rel_extent=prob.rel_extent,
                       window=prob.window, sm_scale=prob.sm_scale)


def _stream_handle(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, name: str, dtype) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _check(code: int, where: str):
    if code != INK_OK:
        raise InkError(code, where)


def inkling_attn_workspace_bytes(params: ink_attn_params_t, is_decode: bool) -> int:
    return int(load_library().inkling_attn_workspace_bytes(ctypes.byref(params), int(bool(is_decode))))


def inkling_attn_workspace_init(workspace: torch.Tensor, stream=None):
    _check(load_library().inkling_attn_workspace_init(
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream_handle(stream)),
        "inkling_attn_workspace_init")


def alloc_workspace(params: ink_attn_params_t, is_decode: bool = True, device="cuda") -> torch.Tensor:
    """Allocate (through PyTorch) and initialise a workspace for ``params``."""
    n = inkling_attn_workspace_bytes(params, is_decode)
    if n == 0:
        raise InkError(2, "inkling_attn_workspace_bytes")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    inkling_attn_workspace_init(ws)
    return ws


def inkling_attn_prefill(params, q, cu_q_lens, max_q_len, k_cache, v_cache, block_table,
                         seq_lens, rel_logits, out, workspace, stream=None):
    """Paged prefill; a bf16 ``rel_logits`` goes to inkling_attn_prefill_bf16bias."""
    lib = load_library()
    bf16 = isinstance(rel_logits, torch.Tensor) and rel_logits.dtype == torch.bfloat16
    fn = lib.inkling_attn_prefill_bf16bias if bf16 else lib.inkling_attn_prefill
    code = fn(
        ctypes.byref(params), _dev(q, "q", torch.bfloat16), _dev(cu_q_lens, "cu_q_lens", torch.int32),
        int(max_q_len), int(q.shape[0]), _dev(k_cache, "k_cache", torch.bfloat16),
        _dev(v_cache, "v_cache", torch.bfloat16),
        _dev(block_table, "block_table", torch.int32), _dev(seq_lens, "seq_lens", torch.int32),
        _dev(rel_logits, "rel_logits", torch.bfloat16 if bf16 else torch.float32),
        _dev(out, "out", torch.bfloat16),
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream_handle(stream))
    _check(code, "inkling_attn_prefill_bf16bias" if bf16 else "inkling_attn_prefill")
    return out


def inkling_attn_prefill_lowrank_bias(params, q, cu_q_lens, max_q_len, k_cache, v_cache, block_table,
                                      seq_lens, r, rel_proj_t, out, workspace, stream=None):
    """Paged prefill with the bias given as r [T, Hq, d_rel] and rel_proj_t [E, d_rel]."""
    lib = load_library()
    if r.dim() != 3 or rel_proj_t.dim() != 2 or rel_proj_t.shape[1] != r.shape[2]:
        raise ValueError("r must be [T, Hq, d_rel] and rel_proj_t [E, d_rel]")
    code = lib.inkling_attn_prefill_lowrank_bias(
        ctypes.byref(params), _dev(q, "q", torch.bfloat16), _dev(cu_q_lens, "cu_q_lens", torch.int32),
        int(max_q_len), int(q.shape[0]), _dev(k_cache, "k_cache", torch.bfloat16),
        _dev(v_cache, "v_cache", torch.bfloat16), _dev(block_table, "block_table", torch.int32),
        _dev(seq_lens, "seq_lens", torch.int32), _dev(r, "r", torch.bfloat16),
        _dev(rel_proj_t, "rel_proj_t", torch.bfloat16), int(r.shape[2]), _dev(out, "out", torch.bfloat16),
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream_handle(stream))
    _check(code, "inkling_attn_prefill_lowrank_bias")
    return out


def inkling_attn_decode(params, q, k_cache, v_cache, block_table, seq_lens, rel_logits, out,
                        workspace, stream=None):
    lib = load_library()
    code = lib.inkling_attn_decode(
        ctypes.byref(params), _dev(q, "q", torch.bfloat16), _dev(k_cache, "k_cache", torch.bfloat16),
        _dev(v_cache, "v_cache", torch.bfloat16), _dev(block_table, "block_table", torch.int32),
        _dev(seq_lens, "seq_lens", torch.int32), _dev(rel_logits, "rel_logits", torch.float32),
        _dev(out, "out", torch.bfloat16), _dev(workspace, "workspace", torch.uint8),
        workspace.numel(), _stream_handle(stream))
    _check(code, "inkling_attn_decode")
    return out


def inkling_attn_decode_noalloc(params, q, k_cache, v_cache, block_table, seq_lens, rel_logits,
                                out, stream=None):
    """Decode without a workspace (the library's own fixed device scratch is used)."""
    lib = load_library()
    code = lib.inkling_attn_decode_noalloc(
        ctypes.byref(params), _dev(q, "q", torch.bfloat16), _dev(k_cache, "k_cache", torch.bfloat16),
        _dev(v_cache, "v_cache", torch.bfloat16), _dev(block_table, "block_table", torch.int32),
        _dev(seq_lens, "seq_lens", torch.int32), _dev(rel_logits, "rel_logits", torch.float32),
        _dev(out, "out", torch.bfloat16), _stream_handle(stream))
    _check(code, "inkling_attn_decode_noalloc")
    return out


def inkling_attn_kv_conv_write(params, k_new, v_new, cu_q_lens, seq_lens, block_table, w_k, w_v,
                               state_k_in, state_v_in, state_k_out, state_v_out, k_cache, v_cache,
                               workspace, stream=None):
    """Causal short convolution of the step's K/V rows into the paged caches, and the
    carried state; ``kernel_size`` is the last dimension of ``w_k``.  With kernel size 1
    the state tensors may be None."""
    lib = load_library()
    ks = int(w_k.shape[-1])
    if tuple(w_v.shape) != tuple(w_k.shape):
        raise ValueError("w_k and w_v must have the same shape")

    def opt(t, name):
        return None if t is None else _dev(t, name, torch.bfloat16)

    code = lib.inkling_attn_kv_conv_write(
        ctypes.byref(params), _dev(k_new, "k_new", torch.bfloat16), _dev(v_new, "v_new", torch.bfloat16),
        _dev(cu_q_lens, "cu_q_lens", torch.int32), int(k_new.shape[0]),
        _dev(seq_lens, "seq_lens", torch.int32), _dev(block_table, "block_table", torch.int32),
        _dev(w_k, "w_k", torch.float32), _dev(w_v, "w_v", torch.float32), ks,
        opt(state_k_in, "state_k_in"), opt(state_v_in, "state_v_in"),
        opt(state_k_out, "state_k_out"), opt(state_v_out, "state_v_out"),
        _dev(k_cache, "k_cache", torch.bfloat16), _dev(v_cache, "v_cache", torch.bfloat16),
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream_handle(stream))
    _check(code, "inkling_attn_kv_conv_write")
    return k_cache, v_cache


def inkling_attn_set_wait_limit_ns(limit_ns: int) -> None:
    """Limit of one pipeline wait in kernels launched from now on (tests of the timeout path)."""
    load_library().inkling_attn_set_wait_limit_ns(int(limit_ns))


def inkling_attn_read_device_error(workspace: torch.Tensor, stream=None, clear: bool = True) -> int:
    v = ctypes.c_uint32(0)
    _check(load_library().inkling_attn_read_device_error(
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream_handle(stream),
        ctypes.byref(v), int(bool(clear))), "inkling_attn_read_device_error")
    return int(v.value)


def run(prob, out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
        stream=None) -> torch.Tensor:
    """One call over a device-resident ``workloads.Problem`` (decode if every n_b == 1)."""
    params = params_of(prob)
    if out is None:
        out = torch.empty_like(prob.q)
    if workspace is None:
        workspace = alloc_workspace(params, True, prob.q.device)
    if prob.r is not None:
        return inkling_attn_prefill_lowrank_bias(params, prob.q, prob.cu_q_lens, prob.max_q_len, prob.k_cache,
                                                 prob.v_cache, prob.block_table, prob.seq_lens, prob.r,
                                                 prob.rel_proj_t, out, workspace, stream)
    if prob.is_decode:
        return inkling_attn_decode(params, prob.q, prob.k_cache, prob.v_cache, prob.block_table,
                                   prob.seq_lens, prob.rel_logits, out, workspace, stream)
    return inkling_attn_prefill(params, prob.q, prob.cu_q_lens, prob.max_q_len, prob.k_cache,
                                prob.v_cache, prob.block_table, prob.seq_lens, prob.rel_logits,
                                out, workspace, stream)
