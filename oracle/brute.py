"""Materialised-matrix restatement of the attention definition, for tiny inputs.

TEST INFRASTRUCTURE ONLY (it pins ``attn_ref.c``; nothing on the product path uses it).

Per sequence it gathers the logical K/V history through the block table, builds the
full ``[n_b, Hq, L_b]`` score matrix with an explicit boolean mask, adds the bias
gathered by clamped distance, and applies a max-subtracted softmax.  The order of
operations is deliberately different from the per-row C loops so that the two agree
only if both follow the definition:

* bias added pre-softmax per (query token, head, distance), "Support Inkling-NVFP4
  model" (TensorRT-LLM PR #17062), section "Architecture";
* GQA head map ``h // (Hq // Hkv)`` and positional paging ``k // P`` bounded by the
  sequence's own length, "Inkling attn backend cleanup fake registry"
  (TensorRT-LLM PR #17860).
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def attention(*, num_q_heads, num_kv_heads, head_dim, page_size, rel_extent, window,
              sm_scale, cu_q, seq_lens, q_bits, k_bits, v_bits, block_table, rel):
    """Full fp64 output ``[total_q, Hq, D]``."""
    cu_q = np.asarray(cu_q, dtype=np.int64)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    q = bf16_bits_to_f64(q_bits)
    kc = bf16_bits_to_f64(k_bits)
    vc = bf16_bits_to_f64(v_bits)
    rel = np.asarray(rel, dtype=np.float64)
    G = num_q_heads // num_kv_heads
    assert G * num_kv_heads == num_q_heads
    out = np.zeros((int(cu_q[-1]), num_q_heads, head_dim))
    for b in range(seq_lens.shape[0]):
        L = int(seq_lens[b])
        t0, t1 = int(cu_q[b]), int(cu_q[b + 1])
        n = t1 - t0
        if L == 0 or n == 0:
            continue
        assert n <= L
        n_pages = -(-L // page_size)
        pages = np.asarray(block_table[b, :n_pages], dtype=np.int64)
        # [n_pages, Hkv, P, D] -> [n_pages*P, Hkv, D] -> keep the first L logical keys
        K = kc[pages].transpose(0, 2, 1, 3).reshape(n_pages * page_size, num_kv_heads, head_dim)[:L]
        V = vc[pages].transpose(0, 2, 1, 3).reshape(n_pages * page_size, num_kv_heads, head_dim)[:L]
        K = np.repeat(K, G, axis=1)          # query head h reads KV head h // G
        V = np.repeat(V, G, axis=1)
        pos = L - n + np.arange(n)            # absolute positions of the new tokens
        dist = pos[:, None] - np.arange(L)[None, :]          # [n, L]
        visible = dist >= 0
        if window > 0:
            visible &= dist <= window - 1
        bucket = np.clip(dist, 0, rel_extent - 1)
        bias = np.take_along_axis(rel[t0:t1], np.broadcast_to(bucket[:, None, :], (n, num_q_heads, L)), axis=2)
        S = sm_scale * np.einsum("nhd,lhd->nhl", q[t0:t1], K) + bias
        S = np.where(visible[:, None, :], S, -np.inf)
        S = S - S.max(axis=2, keepdims=True)
        Wt = np.exp(S)
        Wt /= Wt.sum(axis=2, keepdims=True)
        out[t0:t1] = np.einsum("nhl,lhd->nhd", Wt, V)
    return out
