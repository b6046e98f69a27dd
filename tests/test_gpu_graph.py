"""The prefill and decode calls inside one CUDA graph.

The entry points are stream-ordered, allocate nothing and never synchronise, so a serving
loop can capture a layer's calls once and replay them.  Replays must give the bits of the
eager calls (the split-K tickets are left at zero by the kernels, so every replay starts
from the same workspace state)."""
import pytest
import torch

from paged_attention_relative_gqa_gb300 import binding
from paged_attention_relative_gqa_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    yield
    torch.cuda.empty_cache()


def _calls(prob, out, ws):
    params = binding.params_of(prob)
    if prob.is_decode:
        return lambda: binding.inkling_attn_decode(params, prob.q, prob.k_cache, prob.v_cache, prob.block_table,
                                                   prob.seq_lens, prob.rel_logits, out, ws)
    return lambda: binding.inkling_attn_prefill(params, prob.q, prob.cu_q_lens, prob.max_q_len, prob.k_cache,
                                                prob.v_cache, prob.block_table, prob.seq_lens, prob.rel_logits,
                                                out, ws)


@pytest.mark.parametrize("kind,layer", [("swa", 0), ("global", 5)])
def test_layer_calls_replay_from_a_cuda_graph(kind, layer):
    pre, dec = W.mixed_layer(kind, layer, DEV)
    probs = [pre, dec]
    outs = [torch.empty_like(p.q) for p in probs]
    wss = [binding.alloc_workspace(binding.params_of(p), True, torch.device(DEV)) for p in probs]
    calls = [_calls(p, o, w) for p, o, w in zip(probs, outs, wss)]
    for c in calls:          # eager run (also the one-time per-device setup)
        c()
    torch.cuda.synchronize()
    eager = [o.clone() for o in outs]
    for o in outs:
        o.fill_(float("nan"))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for c in calls:
            c()
    for _ in range(3):
        for o in outs:
            o.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        for o, e in zip(outs, eager):
            assert torch.equal(o, e)
    for w in wss:
        assert binding.inkling_attn_read_device_error(w) == 0
    del graph, pre, dec, outs, eager
    torch.cuda.empty_cache()


def test_noalloc_decode_replays_from_a_cuda_graph():
    prob = W.swa_decode(DEV)
    params = binding.params_of(prob)
    out = torch.empty_like(prob.q)
    run = lambda: binding.inkling_attn_decode_noalloc(params, prob.q, prob.k_cache, prob.v_cache,
                                                      prob.block_table, prob.seq_lens, prob.rel_logits, out)
    run()                    # first call on the device: looks up the library's scratch
    torch.cuda.synchronize()
    eager = out.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    for _ in range(3):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
