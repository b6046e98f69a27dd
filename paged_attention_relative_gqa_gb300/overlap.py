"""Two-stream issue of a serving step: per layer, the prefill call on the caller's stream and
the decode call on a side stream, forked and joined so that the layers stay in order.

The prefill of a layer is bound by the tensor cores and shared memory, its decode by HBM, and
the two read the same pools without writing them, so nothing orders one before the other.
On one stream the decode waits for the prefill's last wave; on two, its CTAs take the SMs
that the prefill's tail frees, and the decode's own tail overlaps the prefill.  Issued under
CUDA-graph capture the fork and join become graph edges: each layer's two kernels are sibling
nodes between the previous layer's join and the next layer's fork.  (The mixed serving batch,
prompts prefilled beside running decodes in every layer: "Support Inkling-NVFP4 model",
TensorRT-LLM PR #17062, section "Architecture".)
"""
from typing import Callable, List, Sequence, Tuple

import torch

Calls = Sequence[Callable[[], None]]


class LayerStreams:
    """Issues each layer's (prefill calls, decode calls) on two streams.

    Every call must launch on the current stream (the binding's calls do when given no
    stream).  ``decode_first`` issues the side stream's calls before the main stream's.  With
    the persistent one-CTA-per-SM prefill, prefill first is the better order: the decode's
    CTAs then take the SMs the prefill's last wave leaves (decode first delays the whole
    prefill wave behind the decode's CTAs).
    """

    def __init__(self, device=None, decode_first: bool = False):
        self.side = torch.cuda.Stream(device=device)
        self.decode_first = decode_first

    def run(self, layers: Sequence[Tuple[Calls, Calls]]) -> None:
        main = torch.cuda.current_stream()
        for main_calls, side_calls in layers:
            self.side.wait_stream(main)            # fork: the side starts after the previous layer
            if self.decode_first:
                self._issue(side_calls, self.side)
                self._issue(main_calls, main)
            else:
                self._issue(main_calls, main)
                self._issue(side_calls, self.side)
            main.wait_stream(self.side)            # join: the next layer starts after both

    @staticmethod
    def _issue(calls: Calls, stream) -> None:
        with torch.cuda.stream(stream):
            for c in calls:
                c()


def serial(layers: Sequence[Tuple[Calls, Calls]]) -> List[Callable[[], None]]:
    """The same step as one stream of calls, layer by layer, prefill before decode."""
    return [c for main_calls, side_calls in layers for c in (*main_calls, *side_calls)]
