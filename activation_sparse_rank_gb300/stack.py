"""A stack of sparse-FFN layers run in decode order, captured as a CUDA graph.

One step feeds T tokens (each a batch of B rows) through the L layers in
sequence: for token t and layer l, ``pi_layer_forward`` computes the predictor,
the active list and the sparse FFN of x[t, l] into y[t, l].  The active count
of every (token, layer) is kept on the device, so touched bytes can be
counted after the step without any host round trip inside it.  The whole
step is one graph launch; successive kernels are chained with programmatic
dependent launch inside libpi.
"""
from __future__ import annotations

from typing import List, Optional

import torch

from .binding import Layer


class SparseFFNStack:
    def __init__(self, layers: List[Layer], tokens: int, B: int = 1):
        if not layers:
            raise ValueError("empty stack")
        self.layers = layers
        self.L = len(layers)
        self.T = int(tokens)
        self.B = int(B)
        self.d = layers[0].d
        self.ffn_max = max(l.ffn for l in layers)
        dev = layers[0].device
        self.device = dev
        self.ws = torch.empty(max(l.workspace_bytes(B) for l in layers), dtype=torch.uint8,
                              device=dev)
        self.idx = torch.empty(self.L, self.ffn_max, dtype=torch.int32, device=dev)
        self.count = torch.zeros(self.T, self.L, dtype=torch.int32, device=dev)
        self.x = torch.empty(self.T, self.L, B, self.d, dtype=torch.float16, device=dev)
        self.y = torch.empty(self.T, self.L, B, self.d, dtype=torch.float32, device=dev)
        self.graph: Optional[torch.cuda.CUDAGraph] = None
        self.stream = torch.cuda.Stream(device=dev)

    def launches_per_step(self) -> int:
        return sum(l.forward_launches(self.B) for l in self.layers) * self.T

    def enqueue(self, stream=None, tokens=None):
        """Enqueue the step (all tokens, all layers) on `stream` without a graph."""
        for t in range(self.T if tokens is None else tokens):
            for li, layer in enumerate(self.layers):
                layer.forward(self.x[t, li], self.idx[li], self.count[t, li:li + 1],
                              self.y[t, li], ws=self.ws, stream=stream)

    def capture(self, timing_events=None):
        """Capture one step as a CUDA graph.  timing_events: optional dict
        {(t, l): (before, after)} of external torch events recorded around the
        main up/down kernel of those launches."""
        s = self.stream
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.enqueue(stream=s)            # warm-up outside capture (same work)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for t in range(self.T):
                for li, layer in enumerate(self.layers):
                    ev = timing_events.get((t, li)) if timing_events else None
                    if ev is not None:
                        layer.set_timing_events(*ev)
                    layer.forward(self.x[t, li], self.idx[li], self.count[t, li:li + 1],
                                  self.y[t, li], ws=self.ws, stream=s)
                    if ev is not None:
                        layer.set_timing_events(None, None)
        return g

    def build_graph(self):
        self.graph = self.capture()
        return self.graph

    def replay(self):
        if self.graph is None:
            self.build_graph()
        self.graph.replay()

    def run_host(self, x_host: torch.Tensor, y_host: torch.Tensor, stream=None):
        """One step from host memory: copy x_host [T, L, B, d] (pinned fp16) in,
        replay the step, copy y [T, L, B, d] fp32 out to pinned y_host."""
        if self.graph is None:
            self.build_graph()
        s = stream or torch.cuda.current_stream()
        with torch.cuda.stream(s):
            self.x.copy_(x_host, non_blocking=True)
            self.graph.replay()
            y_host.copy_(self.y, non_blocking=True)
