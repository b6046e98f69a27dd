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


def test_layer_step_with_kv_write_replays_and_matches_the_oracle():
    """A layer's K/V write (conv + paged write of the prefill rows) and its prefill attention
    captured together: replays give the eager bits, and the attention output, checked on
    sampled rows against the oracle run on the pools as written, is within the prefill
    tolerances."""
    import numpy as np
    from tests.parity import sampled_check

    pre, _ = W.mixed_layer("swa", 1, DEV)
    step = W.kv_step_for(pre, W.KV_CONV_KERNEL, seed=123)
    kvp = binding.make_params(num_seqs=step.num_seqs, num_q_heads=step.num_kv_heads, num_kv_heads=step.num_kv_heads,
                              head_dim=step.head_dim, page_size=step.page_size, max_pages_per_seq=step.max_pages,
                              num_pages=step.num_pages, rel_extent=1, window=-1, sm_scale=1.0)
    ws_kv = binding.alloc_workspace(kvp, False, torch.device(DEV))
    sk, sv = torch.empty_like(step.state_k), torch.empty_like(step.state_v)
    out = torch.empty_like(pre.q)
    ws = binding.alloc_workspace(binding.params_of(pre), True, torch.device(DEV))
    attn = _calls(pre, out, ws)

    def layer():
        binding.inkling_attn_kv_conv_write(kvp, step.k_new, step.v_new, step.cu_q_lens, step.seq_lens,
                                           step.block_table, step.w_k, step.w_v, step.state_k, step.state_v,
                                           sk, sv, step.k_cache, step.v_cache, ws_kv)
        attn()

    layer()
    torch.cuda.synchronize()
    eager = out.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer()
    for _ in range(2):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    assert binding.inkling_attn_read_device_error(ws_kv) == 0
    assert binding.inkling_attn_read_device_error(ws) == 0
    sampled_check(pre, out, 9, "layer step with K/V write (sampled rows)")


def test_two_stream_layers_replay_bitwise_from_a_cuda_graph():
    """Per layer, the prefill on the capturing stream and the decode on a side stream (fork and
    join per layer): the graph's replays give the bits of the serial eager calls."""
    from paged_attention_relative_gqa_gb300 import overlap
    layers, outs, keep = [], [], []
    for i, kind in enumerate(["swa", "global"]):
        pre, dec = W.mixed_layer(kind, i, DEV, n_prefill=2, n_decode=32)
        sides = []
        for prob in (pre, dec):
            out = torch.empty_like(prob.q)
            ws = binding.alloc_workspace(binding.params_of(prob), True, torch.device(DEV))
            outs.append(out)
            keep.append((prob, ws))
            sides.append([_calls(prob, out, ws)])
        layers.append((sides[0], sides[1]))
    for c in overlap.serial(layers):
        c()
    torch.cuda.synchronize()
    eager = [o.clone() for o in outs]
    two = overlap.LayerStreams(torch.device(DEV))
    capture = torch.cuda.Stream()
    with torch.cuda.stream(capture):
        two.run(layers)                  # eager on two streams once
    torch.cuda.synchronize()
    assert all(torch.equal(o, e) for o, e in zip(outs, eager))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=capture):
        two.run(layers)
    for _ in range(3):
        for o in outs:
            o.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        for o, e in zip(outs, eager):
            assert torch.equal(o, e)
    for _, ws in keep:
        assert binding.inkling_attn_read_device_error(ws) == 0
    del graph, layers, outs, eager, keep
    torch.cuda.empty_cache()
