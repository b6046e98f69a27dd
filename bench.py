"""Benchmark of the paged relative-bias GQA attention path on GB300.

Default (N=1): the SWA-layer decode workload (batch 64, 64 query heads over 16 KV heads,
head_dim 128, window 512, contexts U{1024..8192}, page 64, fp32 bias [64, 64, 512]) is
the headline step: one decode call, i.e. one pass of every step of the hot path (page
walk, scores, bias gather, mask, online softmax, PV, split-K merge, store).  The same
run also reports the other workloads (global decode, SWA prefill tiny, global prefill,
mixed 5 SWA + 1 global serving step) under "workloads".

One JSON line is printed by rank 0.  `--impl reference` times the fp64 CPU oracle on
the same workload instead (a bounded row sample per step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import shutil
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_attention_relative_gqa_gb300 import workloads as W  # noqa: E402
from paged_attention_relative_gqa_gb300 import overlap  # noqa: E402

METRIC = "decode attn HBM GB/s (% of 8 TB/s); prefill attn TFLOP/s (% bf16 peak); tok/s"
HEADLINE = "swa_decode"
DATA = "synthetic (seeded; Q/K/V ~N(0,1) bf16, bias ~N(0,0.5) fp32)"


# ---------------------------------------------------------------- algorithmic work

def visible_ranges(prob):
    """Per new token: (p, lo) of its visible keys."""
    out = []
    for n, L in zip(prob.q_lens, prob.seq_lens_list):
        pos = np.arange(L - n, L, dtype=np.int64)
        lo = np.zeros_like(pos) if prob.window <= 0 else np.maximum(0, pos - prob.window + 1)
        out.append((pos, lo))
    return out


def decode_bytes(prob) -> int:
    """K+V of visible keys, bias buckets used, Q and out, table entries and lengths read."""
    D, Hq, Hkv, E, P = prob.head_dim, prob.num_q_heads, prob.num_kv_heads, prob.rel_extent, prob.page_size
    total = 0
    for (pos, lo) in visible_ranges(prob):
        for p, l in zip(pos.tolist(), lo.tolist()):
            vis = p - l + 1
            total += vis * Hkv * D * 2 * 2
            total += Hq * min(vis, E) * 4
            total += ((p // P) - (l // P) + 1) * 4
    total += prob.total_q * Hq * D * 2 * 2 + prob.num_seqs * 4
    return total


def prefill_work(prob):
    """(FLOPs, bytes, bias FLOPs): 4*D per visible (row, key, head); bias read once (or,
    in low-rank form, r and the projection read once, plus 2*d_rel FLOPs per bias bucket
    used), Q/out, K/V once."""
    D, Hq, Hkv, E = prob.head_dim, prob.num_q_heads, prob.num_kv_heads, prob.rel_extent
    flops = 0
    bias = 0
    buckets = 0
    for (pos, lo) in visible_ranges(prob):
        vis = pos - lo + 1
        flops += int(vis.sum()) * 4 * D * Hq
        buckets += int(np.minimum(vis, E).sum()) * Hq
    bias_flops = 0
    if prob.r is not None:
        d = prob.r.shape[-1]
        bias = prob.r.numel() * 2 + prob.rel_proj_t.numel() * 2
        bias_flops = buckets * 2 * d
    else:
        bias = buckets * prob.rel_logits.element_size()
    kv = sum(prob.seq_lens_list) * Hkv * D * 2 * 2
    qo = prob.total_q * Hq * D * 2 * 2
    return flops, bias + kv + qo, bias_flops


def kv_write_bytes(step) -> int:
    """K/V write: new K and V rows read, the same number of cache rows written, the
    carried state read and written, the filters, lengths, offsets and the table entries
    of the pages written."""
    row = step.num_kv_heads * step.head_dim * 2
    ks, B, P = step.kernel_size, step.num_seqs, step.page_size
    total = 2 * step.total_q * row * 2
    total += 2 * 2 * B * (ks - 1) * row
    total += 2 * step.num_kv_heads * step.head_dim * ks * 4
    total += (2 * B + 1) * 4
    for n, L in zip(step.q_lens, step.seq_lens_list):
        if n:
            total += ((L - 1) // P - (L - n) // P + 1) * 4
    return total


# ---------------------------------------------------------------- GPU timing helpers

class Clocks:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        smi = shutil.which("nvidia-smi")
        if not smi:
            return
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        self.proc = subprocess.Popen([smi, "-i", str(self.index), f"--query-gpu={self.Q}",
                                      "--format=csv,noheader,nounits", "-lms", "100"],
                                     stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        time.sleep(0.3)

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 9:
                rows.append(f)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def time_steps(fns, steps, warmup, stream):
    """Warm up, then time exactly `steps` calls (cycling through `fns`) with CUDA events
    on `stream`; returns ms per step."""
    with torch.cuda.stream(stream):
        for i in range(warmup):
            fns[i % len(fns)]()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for i in range(steps):
            fns[i % len(fns)]()
        end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


def time_flushed(fn, steps, warmup, stream, flush):
    """Per-call CUDA-event time of `fn` with L2 flushed (a write of `flush`, larger than
    L2) before every call; returns the mean ms of the calls alone."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            flush.zero_()
            fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in ev) / steps


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), float(m["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def kernel_source_hash(name: str) -> str:
    p = os.path.join(ROOT, "paged_attention_relative_gqa_gb300", "csrc", name)
    return hashlib.sha256(open(p, "rb").read()).hexdigest()[:16]


def profiled_traffic(kernel_file: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            t = json.load(f)
        e = t[workload]
        if e.get("source_sha256_16") == kernel_source_hash(kernel_file):
            return int(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ---------------------------------------------------------------- our arm

def make_call(binding, prob, out, ws):
    params = binding.params_of(prob)
    if prob.r is not None:
        return lambda: binding.inkling_attn_prefill_lowrank_bias(params, prob.q, prob.cu_q_lens, prob.max_q_len,
                                                                 prob.k_cache, prob.v_cache, prob.block_table,
                                                                 prob.seq_lens, prob.r, prob.rel_proj_t, out, ws)
    if prob.is_decode:
        return lambda: binding.inkling_attn_decode(params, prob.q, prob.k_cache, prob.v_cache,
                                                   prob.block_table, prob.seq_lens, prob.rel_logits,
                                                   out, ws)
    return lambda: binding.inkling_attn_prefill(params, prob.q, prob.cu_q_lens, prob.max_q_len,
                                                prob.k_cache, prob.v_cache, prob.block_table,
                                                prob.seq_lens, prob.rel_logits, out, ws)


def bench_workload(binding, probs, steps, warmup, stream):
    calls = []
    keep = []
    for prob in probs:
        params = binding.params_of(prob)
        ws = binding.alloc_workspace(params, True, prob.q.device)
        out = torch.empty_like(prob.q)
        keep.append((ws, out))
        calls.append(make_call(binding, prob, out, ws))
    ms = time_steps(calls, steps, warmup, stream)
    for (ws, _) in keep:
        assert binding.inkling_attn_read_device_error(ws) == 0
    return ms


def e2e_decode(binding, prob, steps, warmup, stream):
    """Through the C ABI with host buffers: each step copies the step's inputs (q, bias,
    block table, lengths) from pinned host memory, runs decode, and reads the output
    back.  The K/V pool is the resident cache."""
    dev = prob.q.device
    host = {k: getattr(prob, k).cpu().pin_memory() for k in ("q", "rel_logits", "block_table", "seq_lens")}
    dbuf = {k: torch.empty_like(getattr(prob, k)) for k in host}
    out = torch.empty_like(prob.q)
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    params = binding.params_of(prob)
    ws = binding.alloc_workspace(params, True, dev)

    def step():
        for k in host:
            dbuf[k].copy_(host[k], non_blocking=True)
        binding.inkling_attn_decode(params, dbuf["q"], prob.k_cache, prob.v_cache, dbuf["block_table"],
                                    dbuf["seq_lens"], dbuf["rel_logits"], out, ws)
        out_h.copy_(out, non_blocking=True)

    ms = time_steps([step], steps, warmup, stream)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * out_h.element_size()
    return ms, h2d, d2h


E2E_GRAPH_STEPS = 25


def e2e_decode_pipelined(binding, prob, steps, warmup, stream):
    """The same per-step work as `e2e_decode` (every step copies its inputs from pinned host
    memory, runs decode through the C ABI and reads its output back), issued as a serving
    loop issues it: two sets of device buffers, the inputs of step i + 1 copied on their own
    stream while step i computes, and the output of step i copied back on a third stream
    while step i + 1 computes.  E2E_GRAPH_STEPS such steps are captured once into a CUDA
    graph and replayed (the host would otherwise spend longer issuing a step's copies,
    events and call than the GPU spends on it).  Returns ms per step."""
    dev = prob.q.device
    keys = ("q", "rel_logits", "block_table", "seq_lens")
    host = {k: getattr(prob, k).cpu().pin_memory() for k in keys}
    dbuf = [{k: torch.empty_like(getattr(prob, k)) for k in keys} for _ in range(2)]
    outs = [torch.empty_like(prob.q) for _ in range(2)]
    out_h = [torch.empty(prob.q.shape, dtype=prob.q.dtype).pin_memory() for _ in range(2)]
    params = binding.params_of(prob)
    ws = binding.alloc_workspace(params, True, dev)
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: [torch.cuda.Event() for _ in range(2)]
    loaded, computed, read = ev(), ev(), ev()

    def run(n):
        def load(i):
            s = i & 1
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(computed[s])   # step i - 2 has read this set
                for k in keys:
                    dbuf[s][k].copy_(host[k], non_blocking=True)
                loaded[s].record(up)
        up.wait_stream(stream)
        down.wait_stream(stream)
        load(0)
        for i in range(n):
            s = i & 1
            if i + 1 < n:
                load(i + 1)
            with torch.cuda.stream(stream):
                stream.wait_event(loaded[s])
                if i >= 2:
                    stream.wait_event(read[s])   # step i - 2's output has been copied back
                b = dbuf[s]
                binding.inkling_attn_decode(params, b["q"], prob.k_cache, prob.v_cache, b["block_table"],
                                            b["seq_lens"], b["rel_logits"], outs[s], ws, stream)
                computed[s].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(computed[s])
                out_h[s].copy_(outs[s], non_blocking=True)
                read[s].record(down)
        stream.wait_stream(up)
        stream.wait_stream(down)

    run(2)   # eager once: the library's one-time per-device setup stays outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        run(E2E_GRAPH_STEPS)
    reps = max(1, steps // E2E_GRAPH_STEPS)
    with torch.cuda.stream(stream):
        for _ in range(max(1, warmup // E2E_GRAPH_STEPS)):
            graph.replay()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(reps):
            graph.replay()
        end.record(stream)
    torch.cuda.synchronize()
    assert binding.inkling_attn_read_device_error(ws) == 0
    del graph
    # every step decodes the same inputs: both host copies of the output hold the bits of a
    # plain device-resident call
    ref = torch.empty_like(prob.q)
    binding.inkling_attn_decode(params, prob.q, prob.k_cache, prob.v_cache, prob.block_table, prob.seq_lens,
                                prob.rel_logits, ref, ws, stream)
    torch.cuda.synchronize()
    ref_h = ref.cpu()
    assert all(torch.equal(o.view(torch.int16), ref_h.view(torch.int16)) for o in out_h), "e2e output differs"
    return start.elapsed_time(end) / (reps * E2E_GRAPH_STEPS)


def cpu_baseline_decode(prob_cpu, seconds: float = 10.0):
    """The fp64 oracle on whole passes of the workload, repeated for about `seconds`."""
    import oracle
    kw = prob_cpu.oracle_kwargs()
    nbytes = decode_bytes(prob_cpu)
    t_sum, passes = 0.0, 0
    while t_sum < seconds:
        t0 = time.perf_counter()
        oracle.attention(**kw)
        t_sum += time.perf_counter() - t0
        passes += 1
    gbs = nbytes * passes / t_sum / 1e9
    return gbs, t_sum, passes, oracle.num_threads()


WORKLOAD_DESC = {
    "swa_decode": "swa_decode: batch 64, 64 q heads / 16 kv heads, head_dim 128, window 512, "
                  "contexts U{1024..8192}, page 64, bias [64,64,512] fp32",
    "global_decode": "global_decode: batch 32, 64 q heads / 8 kv heads, head_dim 128, full causal, "
                     "contexts U{8192..32768}, page 64, bias [32,64,4096] fp32 (clamped)",
    "swa_prefill_tiny": "swa_prefill_tiny: 1 x 1024 tokens, 8 q heads / 2 kv heads, head_dim 64, "
                        "window 512, page 16, bias [1024,8,512] fp32",
    "global_prefill": "global_prefill: 4 x 8192 tokens, 64 q heads / 8 kv heads, head_dim 128, "
                      "full causal, page 64, bias [32768,64,4096] fp32 (clamped)",
    "global_prefill_bf16bias": "global_prefill with the bias in bf16 (inkling_attn_prefill_bf16bias): "
                               "4 x 8192 tokens, 64 q heads / 8 kv heads, head_dim 128, full causal, "
                               "page 64, bias [32768,64,4096] bf16 (clamped)",
    "global_prefill_lowrank": "global_prefill with the bias in low-rank form (inkling_attn_prefill_lowrank_bias): "
                              "4 x 8192 tokens, 64 q heads / 8 kv heads, head_dim 128, full causal, page 64, "
                              "E 4096 (clamped), r [32768,64,64] bf16, projection [4096,64] bf16",
    "global_prefill_lowrank_small": "global_prefill_lowrank_small (profiling size): 1 x 2048 tokens, 64 q heads / "
                                    "8 kv heads, head_dim 128, full causal, page 64, E 4096, r [2048,64,64] bf16",
    "global_prefill_small": "global_prefill_small (profiling size): 1 x 2048 tokens, 64 q heads / "
                            "8 kv heads, head_dim 128, full causal, page 64, bias [2048,64,4096] fp32",
    "global_prefill_bf16bias_small": "global_prefill_bf16bias_small (profiling size): 1 x 2048 tokens, 64 q "
                                     "heads / 8 kv heads, head_dim 128, full causal, page 64, bias "
                                     "[2048,64,4096] bf16",
    "kv_prefill_global": "K/V short convolution (ks 4) + paged write of a global-layer prefill step: "
                         "4 fresh prompts x 8192 tokens, 8 kv heads, head_dim 128, page 64",
    "kv_decode_swa": "K/V short convolution (ks 4) + paged write of an SWA-layer decode step: 64 requests, "
                     "16 kv heads, head_dim 128, contexts U{1024..8192}, page 64 (back-to-back steps over rotating "
                     "instances > L2; isolated_ms: one call with L2 flushed before it)",
    "mixed": "mixed serving step: 5 SWA + 1 global layer, each one prefill call (8 x 2048 tokens) "
             "and one decode call (128 requests, contexts log-uniform 512..16384)",
    "mixed_kv_graph": "mixed serving step with each layer's K/V write, replayed from one CUDA graph (24 calls): "
                      "5 SWA + 1 global layer, each: K/V short convolution (ks 4) + paged write of the prefill "
                      "rows (8 x 2048) and of the decode rows (128), then the prefill call and the decode call; "
                      "per layer the prefill side and the decode side on two streams (fork/join)",
    "mixed_graph": "mixed serving step replayed from one CUDA graph (its 12 calls captured once): 5 SWA + "
                   "1 global layer, each one prefill call (8 x 2048 tokens) and one decode call (128 "
                   "requests, contexts log-uniform 512..16384), the two on two streams (fork/join per layer)",
}


def workload_instances(name, dev):
    """Problems of one workload; decode workloads get two instances (each > L2) that
    alternate between steps so no step finds its inputs in L2."""
    if name == "swa_decode":
        return [W.swa_decode(dev, seed=2), W.swa_decode(dev, seed=1002)]
    if name == "global_decode":
        return [W.global_decode(dev, seed=3), W.global_decode(dev, seed=1003)]
    if name == "swa_prefill_tiny":
        return [W.swa_prefill_tiny(dev, seed=s) for s in range(8)]  # 8 x 17 MB > L2
    if name == "global_prefill":
        return [W.global_prefill(dev, seed=4)]                       # 36 GB > L2
    if name == "global_prefill_bf16bias":
        return [W.global_prefill(dev, seed=4, bias_dtype=torch.bfloat16)]   # 19 GB > L2
    if name == "global_prefill_lowrank":
        return [W.global_prefill_lowrank(dev, seed=4)]                # r 268 MB + Q/out 1 GB > L2
    if name == "global_prefill_lowrank_small":
        return [W.global_prefill_lowrank(dev, seed=4, batch=1, tokens=2048)]   # profiling size
    if name == "global_prefill_small":
        return [W.global_prefill(dev, seed=4, batch=1, tokens=2048)]  # 2.2 GB > L2
    if name == "global_prefill_bf16bias_small":
        return [W.global_prefill(dev, seed=4, batch=1, tokens=2048, bias_dtype=torch.bfloat16)]  # 1.1 GB > L2
    raise ValueError(name)


def kv_call(binding, step, dev):
    """A K/V-write call over `step` into copies of its pools; returns (fn, workspace)."""
    params = binding.make_params(num_seqs=step.num_seqs, num_q_heads=step.num_kv_heads,
                                 num_kv_heads=step.num_kv_heads, head_dim=step.head_dim,
                                 page_size=step.page_size, max_pages_per_seq=step.max_pages,
                                 num_pages=step.num_pages, rel_extent=1, window=-1, sm_scale=1.0)
    ws = binding.alloc_workspace(params, False, dev)
    sk, sv = torch.empty_like(step.state_k), torch.empty_like(step.state_v)

    def fn():
        binding.inkling_attn_kv_conv_write(params, step.k_new, step.v_new, step.cu_q_lens, step.seq_lens,
                                           step.block_table, step.w_k, step.w_v, step.state_k, step.state_v,
                                           sk, sv, step.k_cache, step.v_cache, ws)
    return fn, ws


def kv_instances(step, n, seed=11):
    """`n` K/V decode steps over the pools of `step`: each its own new rows and carried
    state, and its pages placed by its own permutation of the pool's pages, so that no two
    instances touch the same bytes."""
    import dataclasses
    g = torch.Generator()
    g.manual_seed(seed)
    npages = step.k_cache.shape[0]
    out = [step]
    for _ in range(n - 1):
        perm = torch.randperm(npages, generator=g).to(torch.int32).to(step.block_table.device)
        bt = step.block_table.clone()
        ok = (bt >= 0) & (bt < npages)
        bt[ok] = perm[bt[ok].long()]
        out.append(dataclasses.replace(step, k_new=step.k_new.clone(), v_new=step.v_new.clone(),
                                       state_k=step.state_k.clone(), state_v=step.state_v.clone(),
                                       block_table=bt))
    return out


def measure_kv(binding, name, dev, steps, warmup, stream, hbm_peak):
    step = W.kv_prefill_global(dev) if name == "kv_prefill_global" else W.kv_decode_swa(dev)
    fn, ws = kv_call(binding, step, dev)
    nbytes = kv_write_bytes(step)
    extra = {}
    if name == "kv_prefill_global":
        m = time_steps([fn], steps, warmup, stream)          # 268 MB read + 268 MB written per call > L2
    else:
        # Back-to-back steps, as a serving loop issues them: rotating instances whose
        # distinct inputs add up to more than L2 (160 MB), pools shared, the steps captured
        # once into a CUDA graph (a step is shorter than its host-side launch through the
        # binding, so eager back-to-back calls would time the host).
        n_inst = max(2, -(-(160 << 20) // nbytes))
        calls = [kv_call(binding, s, dev) for s in kv_instances(step, n_inst)]
        with torch.cuda.stream(stream):
            for c in calls:
                c[0]()                      # eager once: one-time per-device setup
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for c in calls:
                c[0]()
        replays = max(3, steps // 4)
        m = time_steps([graph.replay], replays, warmup, stream) / n_inst
        extra["timed_launches"] = replays * n_inst
        for _, w in calls:
            assert binding.inkling_attn_read_device_error(w) == 0
        del graph, calls
        # the same graph timing of as many one-element kernels: what a graph node alone costs
        tiny = torch.zeros(1, device=dev)
        with torch.cuda.stream(stream):
            tiny.add_(1)
        torch.cuda.synchronize()
        g1 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g1, stream=stream):
            for _ in range(n_inst):
                tiny.add_(1)
        extra["graph_one_element_kernel_ms"] = round(time_steps([g1.replay], replays, warmup, stream) / n_inst, 5)
        del g1, tiny
        # one call alone, L2 flushed before it, and the same timing of a one-element kernel:
        # what launch and event latency alone cost
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        extra["isolated_ms"] = round(time_flushed(fn, steps, warmup, stream, flush), 5)
        tiny = torch.zeros(1, device=dev)
        extra["one_element_kernel_ms"] = round(time_flushed(lambda: tiny.add_(1), steps, warmup, stream, flush), 5)
        extra["instances"] = n_inst
        del flush, tiny
    assert binding.inkling_attn_read_device_error(ws) == 0
    gbs = nbytes / m / 1e6
    r = {"ms": m, "value": gbs, "unit": "GB/s", "GB/s": gbs, "hbm_frac": gbs / hbm_peak,
         "tok_s": step.total_q / m * 1e3, "bytes": nbytes, "launches_per_step": 1, "bound": "hbm",
         "kv_step": step}
    r.update(extra)
    return r


def measure(binding, name, dev, steps, warmup, stream, hbm_peak, bf16_peak):
    """Time one workload; returns a dict of its numbers (value in its own unit)."""
    if name.startswith("kv_"):
        return measure_kv(binding, name, dev, steps, warmup, stream, hbm_peak)
    if name in ("mixed", "mixed_graph", "mixed_kv_graph"):
        layers = [W.mixed_layer(k, i, dev) for i, k in enumerate(W.MIXED_STACK)]
        lay, keep = [], []   # per layer: (prefill-side calls, decode-side calls)
        for li, (pre, dec) in enumerate(layers):
            sides = []
            for j, prob in enumerate((pre, dec)):
                side = []
                if name == "mixed_kv_graph":
                    # the rows' K/V write comes before the attention that reads them
                    fn, ws = kv_call(binding, W.kv_step_for(prob, W.KV_CONV_KERNEL, seed=7000 + 10 * li + j), dev)
                    keep.append((ws, None))
                    side.append(fn)
                params = binding.params_of(prob)
                ws = binding.alloc_workspace(params, True, dev)
                out = torch.empty_like(prob.q)
                keep.append((ws, out))
                side.append(make_call(binding, prob, out, ws))
                sides.append(side)
            lay.append((sides[0], sides[1]))
        calls = overlap.serial(lay)

        if name in ("mixed_graph", "mixed_kv_graph"):
            # each layer's prefill on the capturing stream, its decode on a side stream
            two = overlap.LayerStreams(dev)
            with torch.cuda.stream(stream):
                two.run(lay)               # eager once: one-time per-device setup
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                two.run(lay)
            m = time_steps([graph.replay], steps, warmup, stream)
            del graph
        else:
            def mixed_step():
                for c in calls:
                    c()
            m = time_steps([mixed_step], steps, warmup, stream)
        per_call = [round(time_steps([c], 3, 1, stream), 4) for c in calls]
        for ws, _ in keep:
            assert binding.inkling_attn_read_device_error(ws) == 0
        # every token of the step passes through all 6 layers once
        ntok = layers[0][0].total_q + layers[0][1].total_q
        return {"ms": m, "value": ntok / m * 1e3, "unit": "tok/s", "tok_s": ntok / m * 1e3,
                "tokens_per_step": ntok, "launches_per_step": len(calls), "graph": name != "mixed",
                "per_call_ms_in_step_order": per_call}
    probs = workload_instances(name, dev)
    m = bench_workload(binding, probs, steps, warmup, stream)
    p0 = probs[0]
    if p0.is_decode:
        nbytes = decode_bytes(p0)
        gbs = nbytes / m / 1e6
        return {"ms": m, "value": gbs, "unit": "GB/s", "GB/s": gbs, "hbm_frac": gbs / hbm_peak,
                "tok_s": p0.num_seqs / m * 1e3, "bytes": nbytes, "launches_per_step": 1,
                "bound": "hbm", "probs": probs}
    flops, nbytes, bias_flops = prefill_work(p0)
    tfs = flops / m / 1e9
    # the roof that binds is the one whose minimum time is longer (the bias bytes on
    # long-context configurations, the tensor cores on short ones); a low-rank bias adds
    # its own products to the tensor work
    t_hbm, t_tensor = nbytes / (hbm_peak * 1e6), (flops + bias_flops) / (bf16_peak * 1e9)
    tensor_tfs = (flops + bias_flops) / m / 1e9
    return {"ms": m, "value": tfs, "unit": "TFLOP/s", "TFLOP/s": tfs, "tensor_frac": tensor_tfs / bf16_peak,
            "GB/s": nbytes / m / 1e6, "hbm_frac": nbytes / m / 1e6 / hbm_peak,
            "tok_s": p0.total_q / m * 1e3, "flops": flops, "bias_flops": bias_flops, "bytes": nbytes,
            "launches_per_step": 1, "bound": "hbm" if t_hbm >= t_tensor else "tensor", "probs": probs}


def whole_job(ms_local, value_local, world, device):
    """(ms, value, scale) of the whole job: the step time is the slowest rank's (max over
    ranks), and the value is this rank's throughput recomputed at that time, times the
    number of replicas (every rank runs the same workload)."""
    ms = ms_local
    if world > 1:
        t = torch.tensor([ms_local], dtype=torch.float64, device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    scale = ms_local / ms
    return ms, value_local * scale * world, scale


def run_ours(args, rank, world, local_rank):
    from paged_attention_relative_gqa_gb300 import binding, build

    build.build()
    binding.load_library()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    hbm_peak, bf16_peak, peak_src = peaks()
    name = args.workload

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    clocks = Clocks(local_rank)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    r = measure(binding, name, dev, args.steps, args.warmup, stream, hbm_peak, bf16_peak)
    clk = clocks.stop()
    barrier()
    ms, value, scale = whole_job(r["ms"], r["value"], world, dev)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": r["unit"], "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": DATA,
        "config": config_of(name, world),
        "tok_s": round(r["tok_s"] * scale * world, 1),
        "gpu_launches": r.get("timed_launches", args.steps * r["launches_per_step"]),
        "clocks": clk,
    }
    if name.startswith("kv_"):
        step = r.pop("kv_step")
        line["roofline"] = {"bound": "hbm", "achieved": round(r["GB/s"], 2), "peak": hbm_peak, "unit": "GB/s",
                            "frac": round(r["GB/s"] / hbm_peak, 4), "peak_source": peak_src,
                            "traffic": profiled_traffic("kv_conv.cu", name), "algorithmic_bytes": r["bytes"],
                            "kernel": "kv_conv_staged_kernel" if name == "kv_prefill_global" else "kv_conv_write_kernel"}
        e2e_ms, h2d, d2h = e2e_kv(binding, step, max(5, args.steps // 4), args.warmup, stream)
        line["e2e"] = {"value": round(r["bytes"] / e2e_ms / 1e6 * world, 2), "unit": "GB/s",
                       "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
        del step
    elif name not in ("mixed", "mixed_graph", "mixed_kv_graph"):
        decode = "flops" not in r
        if decode:
            src, kernel = "decode.cu", "decode_persistent_kernel"
        elif "lowrank" in name:
            src, kernel = "prefill_tc.cu", "prefill_tc_kernel"
        else:   # the materialised bias runs the head-pair kernel
            src, kernel = "prefill_pair.cu", "prefill_pair_kernel"
        if r["bound"] == "hbm":
            line["roofline"] = {"bound": "hbm", "achieved": round(r["GB/s"], 2), "peak": hbm_peak,
                                "unit": "GB/s", "frac": round(r["GB/s"] / hbm_peak, 4),
                                "peak_source": peak_src, "traffic": profiled_traffic(src, name),
                                "algorithmic_bytes": r["bytes"], "kernel": kernel}
        else:
            tens = (r["flops"] + r.get("bias_flops", 0)) / r["ms"] / 1e9
            line["roofline"] = {"bound": "tensor", "achieved": round(tens, 2), "peak": bf16_peak,
                                "unit": "TFLOP/s", "frac": round(tens / bf16_peak, 4),
                                "peak_source": peak_src, "traffic": profiled_traffic(src, name),
                                "algorithmic_bytes": r["bytes"], "kernel": kernel}
        if not decode:
            line["roofline"].update({"algorithmic_flops": r["flops"] + r.get("bias_flops", 0),
                                     "attention_flops": r["flops"], "bias_flops": r.get("bias_flops", 0),
                                     "tensor_frac": round(r["tensor_frac"], 4), "hbm_frac": round(r["hbm_frac"], 4)})
        probs = r.pop("probs")
        if probs[0].is_decode:
            e2e_ms, h2d, d2h = e2e_decode(binding, probs[0], max(10, args.steps // 2), args.warmup, stream)
            pipe_ms = e2e_decode_pipelined(binding, probs[0], max(10, args.steps // 2), args.warmup, stream)
            line["e2e"] = {"value": round(r["bytes"] / pipe_ms / 1e6 * world, 2), "unit": "GB/s",
                           "ms_per_step": round(pipe_ms, 5), "h2d_bytes_per_step": h2d,
                           "d2h_bytes_per_step": d2h,
                           "issue": "inputs of step i+1 copied in and output of step i-1 copied out "
                                    "while step i computes (two buffer sets, three streams), "
                                    f"{E2E_GRAPH_STEPS} steps per CUDA graph replay",
                           "serial": {"value": round(r["bytes"] / e2e_ms / 1e6 * world, 2),
                                      "ms_per_step": round(e2e_ms, 5),
                                      "issue": "copy in, compute, copy out on one stream"}}
        elif probs[0].r is not None:
            line["e2e"] = {"value": None, "unit": "TFLOP/s",
                           "skipped": "the low-rank bias prefill is timed device-resident only"}
        elif probs[0].rel_logits.numel() * 4 > (4 << 30):
            line["e2e"] = {"value": None, "unit": "TFLOP/s",
                           "skipped": "inputs above 4 GB are not staged through pinned host memory"}
        else:
            e2e_ms, h2d, d2h = e2e_prefill(binding, probs[0], max(3, args.steps // 4), 3, stream)
            line["e2e"] = {"value": round(r["flops"] / e2e_ms / 1e9 * world, 2), "unit": "TFLOP/s",
                           "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
                           "d2h_bytes_per_step": d2h}
        del probs
    else:
        line["e2e"] = None
        line[name] = {k: v for k, v in r.items() if k not in ("value", "unit")}
    torch.cuda.empty_cache()

    # ---- the other workloads, reported beside the headline
    if not args.no_extra:
        wl = {}
        steps_x = max(5, args.steps // 4)
        for other in ("global_decode", "swa_prefill_tiny", "global_prefill", "global_prefill_bf16bias",
                      "global_prefill_lowrank", "mixed", "mixed_graph", "mixed_kv_graph", "kv_prefill_global",
                      "kv_decode_swa"):
            if other == name:
                continue
            st = steps_x if other in ("global_decode", "swa_prefill_tiny", "kv_prefill_global",
                                      "kv_decode_swa") else max(3, steps_x // 2)
            ck = Clocks(local_rank)
            ck.start()
            o = measure(binding, other, dev, st, min(args.warmup, 3), stream, hbm_peak, bf16_peak)
            o["clocks"] = ck.stop()   # sampled over the workload's setup and its timed calls
            o.pop("probs", None)
            o.pop("kv_step", None)
            wl[other] = {k: (round(v, 5) if isinstance(v, float) else v) for k, v in o.items()
                         if k not in ("value", "unit", "bound", "launches_per_step")}
            torch.cuda.empty_cache()
        line["workloads"] = wl

    # ---- CPU baseline (rank 0, N=1): the oracle, timed on the host cores
    if rank == 0 and world == 1 and not args.no_cpu_baseline and name == "swa_decode":
        prob_cpu = W.swa_decode("cpu", seed=2)
        gbs_cpu, secs, passes, cores = cpu_baseline_decode(prob_cpu)
        line["cpu_baseline"] = {"value": round(gbs_cpu, 4), "unit": "GB/s", "cores": cores,
                                "kind": "oracle",
                                "sample": f"{passes} whole passes of swa_decode (seed 2) in {secs:.1f} s"}
    return line


def e2e_prefill(binding, prob, steps, warmup, stream):
    """Prefill through the C ABI with host buffers: q, bias, table, lengths and query
    offsets copied in from pinned memory each step, output copied back."""
    dev = prob.q.device
    keys = ("q", "rel_logits", "block_table", "seq_lens", "cu_q_lens")
    host = {k: getattr(prob, k).cpu().pin_memory() for k in keys}
    dbuf = {k: torch.empty_like(getattr(prob, k)) for k in keys}
    out = torch.empty_like(prob.q)
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    params = binding.params_of(prob)
    ws = binding.alloc_workspace(params, False, dev)

    def step():
        for k in keys:
            dbuf[k].copy_(host[k], non_blocking=True)
        binding.inkling_attn_prefill(params, dbuf["q"], dbuf["cu_q_lens"], prob.max_q_len, prob.k_cache,
                                     prob.v_cache, dbuf["block_table"], dbuf["seq_lens"],
                                     dbuf["rel_logits"], out, ws)
        out_h.copy_(out, non_blocking=True)

    ms = time_steps([step], steps, warmup, stream)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * out_h.element_size()
    del host, dbuf
    return ms, h2d, d2h


def e2e_kv(binding, step, steps, warmup, stream):
    """K/V write through the C ABI with host buffers: the step's new K/V rows, state,
    lengths, offsets and table copied in from pinned memory each step, the new state
    copied back; the pools are the resident caches."""
    dev = step.k_new.device
    keys = ("k_new", "v_new", "state_k", "state_v", "block_table", "seq_lens", "cu_q_lens")
    host = {k: getattr(step, k).cpu().pin_memory() for k in keys}
    dbuf = {k: torch.empty_like(getattr(step, k)) for k in keys}
    params = binding.make_params(num_seqs=step.num_seqs, num_q_heads=step.num_kv_heads,
                                 num_kv_heads=step.num_kv_heads, head_dim=step.head_dim,
                                 page_size=step.page_size, max_pages_per_seq=step.max_pages,
                                 num_pages=step.num_pages, rel_extent=1, window=-1, sm_scale=1.0)
    ws = binding.alloc_workspace(params, False, dev)
    sk, sv = torch.empty_like(step.state_k), torch.empty_like(step.state_v)
    sk_h = torch.empty(sk.shape, dtype=sk.dtype).pin_memory()
    sv_h = torch.empty(sv.shape, dtype=sv.dtype).pin_memory()

    def one():
        for k in keys:
            dbuf[k].copy_(host[k], non_blocking=True)
        binding.inkling_attn_kv_conv_write(params, dbuf["k_new"], dbuf["v_new"], dbuf["cu_q_lens"],
                                           dbuf["seq_lens"], dbuf["block_table"], step.w_k, step.w_v,
                                           dbuf["state_k"], dbuf["state_v"], sk, sv, step.k_cache,
                                           step.v_cache, ws)
        sk_h.copy_(sk, non_blocking=True)
        sv_h.copy_(sv, non_blocking=True)

    ms = time_steps([one], steps, warmup, stream)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = 2 * sk_h.numel() * sk_h.element_size()
    return ms, h2d, d2h


def config_of(name, world):
    """The `config` object of a line; both arms print the same one for the same workload."""
    return {"workload": WORKLOAD_DESC[name],
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": "inputs larger than L2 (decode: two alternating 0.3-2.7 GB instances)"}


# ---------------------------------------------------------------- reference arm (the oracle)

def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle
    prob = W.swa_decode("cpu", seed=2)
    kw = prob.oracle_kwargs()
    B, Hq = prob.num_seqs, prob.num_q_heads
    total_rows = B * Hq
    nbytes = decode_bytes(prob)
    rows_per_step = total_rows  # a whole decode step is cheap enough for the oracle
    rng = np.random.default_rng(0)

    def step():
        idx = rng.choice(total_rows, size=rows_per_step, replace=False)
        oracle.attention_rows(**kw, rows_t=(idx // Hq).astype(np.int32), rows_h=(idx % Hq).astype(np.int32))

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    secs = time.perf_counter() - t0
    ms = secs / args.steps * 1e3
    gbs = nbytes * (rows_per_step / total_rows) / (secs / args.steps) / 1e9
    cores = oracle.num_threads()
    return {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": DATA,
        "config": config_of(HEADLINE, world),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{rows_per_step} of {total_rows} (sequence, head) rows per step "
                                   "(the whole workload)"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOAD_DESC),
                    help="workload of the timed line (default: the SWA decode headline)")
    ap.add_argument("--no-extra", action="store_true", help="timed workload only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    line = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
