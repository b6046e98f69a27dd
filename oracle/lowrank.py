"""fp64 oracle for the low-rank form of the relative-position bias.

TEST INFRASTRUCTURE ONLY (see the package docstring): only ``tests/``, ``__graft_entry__``
and ``bench.py``'s CPU-baseline leg may use it.  It shares no code with the CUDA library.

"Support Inkling-NVFP4 model" (TensorRT-LLM PR #17062), review of ``_build_rel_logits``:
the bias tensor of a layer is built from a per-(token, head) vector ``r [T, H, d_rel]`` and
the layer's projection ``rel_logits_proj [d_rel, rel_extent]`` as their product over
``d_rel`` (there in fp32, from the two operands widened to fp32):

    rel[t, h, e] = sum_c r[t, h, c] * rel_logits_proj[c, e]

The library takes the projection transposed, bucket-major ``[E, d_rel]`` (``proj_t``), so
the oracle takes that layout too and uses its transpose.  Here the product is exact in
fp64 (bf16 operands, at most 64 terms); the attention oracle then takes the bias in fp32,
a rounding of relative size 2^-24.
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def rel_from_lowrank(r_bits, proj_t_bits) -> np.ndarray:
    """rel ``[T, H, E]`` (fp64) from r bits ``[T, H, d_rel]`` and proj_t bits ``[E, d_rel]``."""
    r = bf16_bits_to_f64(r_bits)
    proj = bf16_bits_to_f64(proj_t_bits).T            # rel_logits_proj [d_rel, E]
    T, H, d = r.shape
    assert proj.shape[0] == d, "d_rel of r and of the projection differ"
    return (r.reshape(T * H, d) @ proj).reshape(T, H, proj.shape[1])


def rel_rows_from_lowrank(r_rows_bits, proj_t_bits) -> np.ndarray:
    """Bias rows ``[n, E]`` (fp64) for r rows ``[n, d_rel]`` (bits)."""
    r = bf16_bits_to_f64(r_rows_bits)
    proj = bf16_bits_to_f64(proj_t_bits).T
    assert proj.shape[0] == r.shape[1], "d_rel of r and of the projection differ"
    return r @ proj
