"""fp64 oracle for the step before attention: the causal K/V short convolution and the
paged K/V write.

TEST INFRASTRUCTURE ONLY (see the package docstring): only ``tests/``, ``__graft_entry__``
and ``bench.py``'s CPU-baseline leg may use it.  It shares no code with the CUDA library.

What it computes follows "Support Inkling-NVFP4 model" (TensorRT-LLM PR #17062):

* section "Architecture": each attention layer runs a causal short convolution on K and on
  V, carrying per-request state across decode steps;

and "Inkling attn backend cleanup fake registry" (TensorRT-LLM PR #17860):

* the commit about carrying the short-convolution state through a cache transfer: each
  convolution keeps a window of kernel_size - 1 past inputs per request (a fresh request
  starts from zeros);
* the commit that moves the KV write into the backend, and the page-table commits: the
  step's K/V rows go into the paged cache at the request's positions through its block
  table (key k in page block_table[b][k // P], slot k % P).

The pages give neither the kernel size nor any bias or activation; the plainest reading
is taken: a depthwise (per channel) convolution with no bias and no activation,

    y[p, g, d] = sum_{j=0}^{ks-1} w[g, d, j] * x[p - (ks - 1) + j, g, d]

where x is the raw projection of position p of the request, taken from this step's new
rows for the last n_b positions and from the carried state for the ks - 1 positions before
them.  y is rounded to bf16 (nearest even) when written to the cache; the new state is
the last ks - 1 raw inputs (rows of x), bf16 as given.
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float64 -> bf16 bit patterns, round to nearest even through fp32 first.

    The CUDA path rounds its fp32 sum to bf16; rounding the fp64 value straight to bf16
    can differ from that only when the fp32 rounding crosses a bf16 tie, which the parity
    tests allow for (1 bf16 ulp)."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    nan = np.isnan(f)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    out = rounded.astype(np.uint16)
    out[nan] = 0x7FC0
    return out


def kv_conv_rows(*, x_bits, cu_q, seq_lens, block_table, page_size, w, ks, state_bits):
    """The convolution of one of K or V, row by row, before any rounding.

    Returns (y, mag, page, slot, state_out): y[t] the fp64 value of new row t
    ([T, Hkv, D]); mag[t] = sum_j |w[., ., j] * x_j| of its terms (the scale of the
    rounding error of any finite-precision sum of them); page[t], slot[t] the cache slot it
    goes to (page -1 for rows of no request); state_out the carried state [B, ks - 1, Hkv, D]
    (bf16 bits).
    """
    T, Hkv, D = x_bits.shape
    B = len(seq_lens)
    w = np.asarray(w, np.float64)
    y_all = np.zeros((T, Hkv, D), np.float64)
    mag_all = np.zeros((T, Hkv, D), np.float64)
    page_of = np.full(T, -1, np.int64)
    slot_of = np.full(T, -1, np.int64)
    st_out = np.zeros((B, max(ks - 1, 0), Hkv, D), np.uint16)
    for b in range(B):
        t0, t1 = int(cu_q[b]), int(cu_q[b + 1])
        n, L = t1 - t0, int(seq_lens[b])
        x_new = bf16_bits_to_f64(x_bits[t0:t1])                       # [n, Hkv, D]
        st_bits = state_bits
        prev = bf16_bits_to_f64(st_bits[b]) if ks > 1 else np.zeros((0, Hkv, D))
        hist = np.concatenate([prev, x_new], axis=0)                  # [ks - 1 + n, Hkv, D]
        for i in range(n):
            p = L - n + i
            # window rows hist[i .. i + ks - 1] are positions p - (ks - 1) .. p
            y = np.zeros((Hkv, D), np.float64)
            mag = np.zeros((Hkv, D), np.float64)
            for j in range(ks):
                y += w[:, :, j] * hist[i + j]
                mag += np.abs(w[:, :, j] * hist[i + j])
            y_all[t0 + i], mag_all[t0 + i] = y, mag
            page_of[t0 + i] = int(block_table[b][p // page_size])
            slot_of[t0 + i] = p % page_size
        if ks > 1:
            st_out[b] = np.concatenate([np.asarray(st_bits[b], np.uint16), np.asarray(x_bits[t0:t1], np.uint16)],
                                       axis=0)[n:]
    return y_all, mag_all, page_of, slot_of, st_out


def kv_conv_write(*, k_new_bits, v_new_bits, cu_q, seq_lens, block_table, page_size,
                  w_k, w_v, ks, state_k_bits, state_v_bits, k_cache_bits, v_cache_bits):
    """The step's convolution and paged write, in fp64, rounded to bf16 when stored.

    Shapes: k_new/v_new bf16 bits [T, Hkv, D]; w_k/w_v float [Hkv, D, ks];
    state_k/state_v bf16 bits [B, ks - 1, Hkv, D] (oldest first); caches bf16 bits
    [num_pages, Hkv, P, D].  Returns (k_cache, v_cache, state_k_out, state_v_out) as bf16
    bits; slots the step does not write keep their input bits.
    """
    out = []
    states = []
    for x_bits, st_bits, w, cache_bits in ((k_new_bits, state_k_bits, w_k, k_cache_bits),
                                           (v_new_bits, state_v_bits, w_v, v_cache_bits)):
        cache = np.array(cache_bits, dtype=np.uint16, copy=True)
        y, _, page, slot, st_out = kv_conv_rows(x_bits=x_bits, cu_q=cu_q, seq_lens=seq_lens,
                                                block_table=block_table, page_size=page_size, w=w, ks=ks,
                                                state_bits=st_bits)
        rows = page >= 0
        cache[page[rows], :, slot[rows], :] = f64_to_bf16_bits(y[rows])
        out.append(cache)
        states.append(st_out)
    return out[0], out[1], states[0], states[1]
