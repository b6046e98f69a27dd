"""Shared helpers of the GPU parity tests: run the CUDA path, run the oracle on the same
inputs (whole or a seeded row sample), and compare with the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_attention_relative_gqa_gb300 import binding

# GPU (bf16 output) vs fp64 oracle, every config.
TOL_MAX_ABS = 2e-2
TOL_REL_RMS = 5e-3


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def run_gpu(prob, workspace=None, check_error=True):
    """Run the CUDA path on a device-resident problem; return (out, error word)."""
    params = binding.params_of(prob)
    ws = workspace if workspace is not None else binding.alloc_workspace(params, True, prob.q.device)
    out = torch.full_like(prob.q, float("nan"))
    binding.run(prob, out=out, workspace=ws)
    err = binding.inkling_attn_read_device_error(ws)
    if check_error:
        assert err == 0, f"device error word {err:#x}"
    return out, err


def oracle_full(prob) -> np.ndarray:
    kw = prob.oracle_kwargs()
    if prob.r is not None:
        import oracle.lowrank as lr
        kw["rel"] = lr.rel_from_lowrank(*prob.lowrank_bits())
    return oracle.attention(**kw)


def oracle_rows(prob, rows: np.ndarray) -> np.ndarray:
    """Oracle on sampled (t, h) rows of a device-resident problem (only those rows'
    query vectors and bias rows are copied to the host)."""
    dev = prob.q.device
    t = torch.from_numpy(rows[:, 0].astype(np.int64)).to(dev)
    h = torch.from_numpy(rows[:, 1].astype(np.int64)).to(dev)
    q_rows = bits(prob.q[t, h])
    if prob.r is not None:
        import oracle.lowrank as lr
        rel_rows = lr.rel_rows_from_lowrank(bits(prob.r[t, h]), bits(prob.rel_proj_t))
    else:
        rel_rows = prob.rel_logits[t, h].float().cpu().numpy()
    return oracle.attention_rows(
        num_q_heads=prob.num_q_heads, num_kv_heads=prob.num_kv_heads, head_dim=prob.head_dim,
        page_size=prob.page_size, rel_extent=prob.rel_extent, window=prob.window,
        sm_scale=prob.sm_scale, cu_q=prob.cu_q_lens.cpu().numpy(),
        seq_lens=prob.seq_lens.cpu().numpy(), q_bits=np.zeros(1, np.uint16),
        k_bits=bits(prob.k_cache), v_bits=bits(prob.v_cache),
        block_table=prob.block_table.cpu().numpy(), rel=np.zeros(1, np.float32),
        rows_t=rows[:, 0], rows_h=rows[:, 1], q_rows_bits=q_rows, rel_rows=rel_rows)


def compare(gpu: np.ndarray, ref: np.ndarray, label: str):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape
    nrows = int(np.prod(gpu.shape[:-1]))
    assert nrows > 0, f"{label}: nothing compared"
    assert np.all(np.isfinite(gpu)), f"{label}: non-finite GPU output"
    diff = gpu - ref
    max_abs = float(np.max(np.abs(diff)))
    rel_rms = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-30))
    print(f"{label}: {nrows} rows compared, max_abs {max_abs:.3e}, rel_rms {rel_rms:.3e}")
    assert max_abs <= TOL_MAX_ABS, f"{label}: max_abs {max_abs}"
    assert rel_rms <= TOL_REL_RMS, f"{label}: rel_rms {rel_rms}"
    return max_abs, rel_rms


# Rows compared per sequence when the oracle cannot take every row of a workload.
SAMPLE_PER_SEQ = 4096


def sampled_check(prob, out: torch.Tensor, seed: int, label: str, per_seq: int = SAMPLE_PER_SEQ):
    """Compare a seeded sample of at least ``per_seq`` (t, h) rows of every sequence (all of
    them when a sequence has fewer) with the oracle, and print the per-sequence counts."""
    from paged_attention_relative_gqa_gb300 import workloads as W
    rows = W.sample_rows(prob, per_seq=per_seq, seed=seed)
    counts = W.rows_per_sequence(prob, rows)
    for n, c in zip(prob.q_lens, counts):
        assert c >= min(per_seq, n * prob.num_q_heads), f"{label}: only {c} rows sampled"
    print(f"{label}: rows per sequence {counts}")
    return compare(gpu_rows(out, rows), oracle_rows(prob, rows), label)


def gpu_rows(out: torch.Tensor, rows: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(rows[:, 0].astype(np.int64)).to(out.device)
    h = torch.from_numpy(rows[:, 1].astype(np.int64)).to(out.device)
    return out[t, h].float().cpu().numpy()
