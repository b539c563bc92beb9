"""A stack of sparse-FFN layers run in decode order, captured as a CUDA graph.

One step feeds T tokens (each a batch of B rows) through the L layers in
sequence: token t is one ``pi_stack_forward`` call over all layers (for
B <= 2 a single persistent cooperative kernel), reading x[t] [L, B, d] and
writing y[t] [L, B, d].  The active count of every (token, layer) stays on
the device, so touched bytes can be counted after the step without any host
round trip inside it.  The whole step is one graph launch.
"""
from __future__ import annotations

import ctypes as C
from typing import List, Optional

import torch

from .binding import PI_STACK_LAYERS_PER_LAUNCH, Layer, stack_forward, stack_forward_host


class SparseFFNStack:
    def __init__(self, layers: List[Layer], tokens: int, B: int = 1, want_idx: bool = False,
                 chained: bool = False):
        if not layers:
            raise ValueError("empty stack")
        self.layers = layers
        self.L = len(layers)
        self.T = int(tokens)
        self.B = int(B)
        self.d = layers[0].d
        self.ffn = layers[0].ffn
        dev = layers[0].device
        self.device = dev
        self.ws = layers[0].workspace(B)
        # ascending active lists of the last token, only when asked for (B <= 2
        # computes the counts without them; B > 2 always needs them)
        self.want_idx = want_idx or B > 2
        self.idx = torch.empty(self.L, self.ffn, dtype=torch.int32, device=dev) if self.want_idx else None
        self.count = torch.zeros(self.T, self.L, dtype=torch.int32, device=dev)
        self.x = torch.empty(self.T, self.L, B, self.d, dtype=torch.float16, device=dev)
        self.y = torch.empty(self.T, self.L, B, self.d, dtype=torch.float32, device=dev)
        self.handles = (C.c_void_p * self.L)(*[l.handle.value for l in layers])
        self.graph: Optional[torch.cuda.CUDAGraph] = None
        self.stream = torch.cuda.Stream(device=dev)
        # chained: each token's layer l >= 1 takes fp16(y_{l-1} / RMS(y_{l-1}))
        # as its input (formed on the device); only x[t, 0] is read
        self.chained = bool(chained)

    def launches_per_step(self) -> int:
        """Kernels of this library launched per step (memsets not counted)."""
        if self.B <= 2:
            n_launch = -(-self.L // PI_STACK_LAYERS_PER_LAUNCH)
            return (2 if self.want_idx else 1) * n_launch * self.T
        return sum(l.forward_launches(self.B) for l in self.layers) * self.T

    def _token(self, t: int, stream):
        stack_forward(self.layers, self.x[t], self.y[t], idx=self.idx, count=self.count[t],
                      ws=self.ws, stream=stream, handles=self.handles, chained=self.chained)

    def enqueue(self, stream=None, tokens=None):
        """Enqueue the step (all tokens, all layers) on `stream` without a graph."""
        for t in range(self.T if tokens is None else tokens):
            self._token(t, stream)

    def capture(self, timing_events=None, tokens=None):
        """Capture one step as a CUDA graph.  timing_events: optional dict
        {t: (before, after)} of external torch events recorded around the main
        kernel of token t."""
        T = self.T if tokens is None else tokens
        s = self.stream
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.enqueue(stream=s, tokens=T)       # warm-up outside capture (same work)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        first = self.layers[0]
        with torch.cuda.graph(g, stream=s):
            for t in range(T):
                ev = timing_events.get(t) if timing_events else None
                if ev is not None:
                    first.set_timing_events(*ev)
                self._token(t, s)
                if ev is not None:
                    first.set_timing_events(None, None)
        return g

    def build_graph(self):
        self.graph = self.capture()
        return self.graph

    def replay(self):
        if self.graph is None:
            self.build_graph()
        self.graph.replay()

    def run_host(self, x_host: torch.Tensor, y_host: torch.Tensor, stream=None):
        """One step from host memory through one library call
        (pi_stack_forward_host): x_host [T, L, B, d] (pinned fp16) is copied
        in, every token runs through the stack, y [T, L, B, d] fp32 is copied
        out to pinned y_host; all on `stream`, not captured in a graph."""
        s = stream or torch.cuda.current_stream()
        stack_forward_host(self.layers, x_host, y_host, self.x, self.y, idx=self.idx,
                           count=self.count, ws=self.ws, stream=s, handles=self.handles,
                           chained=self.chained)
