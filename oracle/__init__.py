"""fp64 CPU oracle for paged relative-bias GQA attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this package:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg use
it.  It shares no code with the CUDA library; the two meet only through the seeded
input generators, which hold none of the method's arithmetic.

Two independent restatements of the same definition live here:

* ``attn_ref.c`` (loaded through ctypes): per-row loops in fp64, OpenMP over rows.
  This is the oracle that parity tests compare against.
* ``brute.py``: numpy, materialises the whole masked score matrix per sequence.
  It is used only to pin the C oracle on tiny inputs.

Both follow "Support Inkling-NVFP4 model" (TensorRT-LLM PR #17062), section
"Architecture" (bias added pre-softmax per query token, head and distance; 512-key
windows on local layers, full causal on global ones) and the GQA / page-table /
seq-len rules of "Inkling attn backend cleanup fake registry" (TensorRT-LLM PR #17860).

Parity is pinned for every function here (see ``tests/test_oracle_pins.py``).
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_ref.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle_attn.so")
_lock = threading.Lock()
_lib = None


def build(src: str = _SRC, out: str = _LIB, extra_flags: tuple = ()) -> str:
    """Compile ``src`` into a shared library at ``out`` with gcc (OpenMP when available)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("oracle build needs gcc")
    base = [cc, "-O2", "-std=c11", "-shared", "-fPIC", *extra_flags, "-o", out, src, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    return out


def _needs_build() -> bool:
    return (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)


def load(path: str | None = None):
    """Return the ctypes handle of the compiled oracle (building it if stale)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _needs_build():
                build()
            _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def _bind(lib):
    P = ctypes.c_void_p
    i = ctypes.c_int
    lib.oracle_attention_rows.argtypes = [i, i, i, i, i, i, i, i, i, ctypes.c_double,
                                          P, P, P, P, P, P, P, ctypes.c_int64, P, P, P, P, P]
    lib.oracle_attention_rows.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    return lib


def num_threads() -> int:
    return int(load().oracle_num_threads())


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def attention_rows(*, num_q_heads: int, num_kv_heads: int, head_dim: int, page_size: int,
                   rel_extent: int, window: int, sm_scale: float,
                   cu_q, seq_lens, q_bits, k_bits, v_bits, block_table, rel,
                   rows_t, rows_h, q_rows_bits=None, rel_rows=None, lib=None) -> np.ndarray:
    """fp64 output rows ``[n_rows, D]`` for the (packed row, head) pairs given.

    ``q_bits``/``k_bits``/``v_bits`` are bf16 bit patterns (uint16 arrays) shaped
    ``[total_q, Hq, D]`` and ``[num_pages, Hkv, P, D]``; ``rel`` is fp32
    ``[total_q, Hq, E]``; ``block_table`` is int32 ``[B, max_pages]``.
    ``q_rows_bits`` ``[n_rows, D]`` and ``rel_rows`` ``[n_rows, E]``, when given, are the
    query vectors and bias rows of the requested rows (``q_bits``/``rel`` may then be
    empty placeholders).
    """
    lib = lib or load()
    cu_q = _c(cu_q, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    q_bits = _c(q_bits, np.uint16)
    k_bits = _c(k_bits, np.uint16)
    v_bits = _c(v_bits, np.uint16)
    block_table = _c(block_table, np.int32)
    rel = _c(rel, np.float32)
    rows_t = _c(rows_t, np.int32)
    rows_h = _c(rows_h, np.int32)
    if q_rows_bits is not None:
        q_rows_bits = _c(q_rows_bits, np.uint16)
        assert q_rows_bits.shape == (rows_t.shape[0], head_dim)
    if rel_rows is not None:
        rel_rows = _c(rel_rows, np.float32)
        assert rel_rows.shape == (rows_t.shape[0], rel_extent)
    num_seqs = seq_lens.shape[0]
    num_pages = k_bits.shape[0]
    max_pages = block_table.shape[1] if block_table.ndim == 2 else 0
    n = rows_t.shape[0]
    out = np.zeros((n, head_dim), dtype=np.float64)
    ptr = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    st = lib.oracle_attention_rows(num_seqs, num_q_heads, num_kv_heads, head_dim, page_size,
                                   max_pages, num_pages, rel_extent, window, float(sm_scale),
                                   ptr(cu_q), ptr(seq_lens), ptr(q_bits), ptr(k_bits),
                                   ptr(v_bits), ptr(block_table), ptr(rel), n, ptr(rows_t),
                                   ptr(rows_h), ptr(q_rows_bits), ptr(rel_rows), ptr(out))
    if st != 0:
        raise ValueError(f"oracle rejected the inputs (status {st})")
    return out


def attention(*, num_q_heads: int, head_dim: int, cu_q, **kw) -> np.ndarray:
    """Full fp64 output ``[total_q, Hq, D]`` (every row, every head)."""
    total_q = int(np.asarray(cu_q)[-1])
    t = np.repeat(np.arange(total_q, dtype=np.int32), num_q_heads)
    h = np.tile(np.arange(num_q_heads, dtype=np.int32), total_q)
    o = attention_rows(num_q_heads=num_q_heads, head_dim=head_dim, cu_q=cu_q,
                       rows_t=t, rows_h=h, **kw)
    return o.reshape(total_q, num_q_heads, head_dim)
