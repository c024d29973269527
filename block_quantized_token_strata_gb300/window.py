"""A full verify window on one GPU: every projection of every layer, then the head's argmax.

One step = for each of the window's matrices (48 layers x qkv/o/up/down Q4, then the Q8 head):
quantize that projection's T fp32 input rows, run the T-column GEMV (or the head GEMV + argmax).
The layers are not chained (no model between them): each projection has its own seeded input,
so the step measures what the window costs — every dense weight byte read once for T tokens.
All work is enqueued through the C ABI on one stream and can be captured in one CUDA graph;
consecutive kernels overlap their weight prefetch with the previous kernel's tail
(programmatic dependent launch).
"""
from __future__ import annotations

import numpy as np
import torch

from . import strata, synth


class WindowWeights:
    """Device copies of every matrix of the window (generated once, seeded)."""

    def __init__(self, layers: int = synth.WINDOW_LAYERS, device="cuda", key="window", host_copy=False):
        self.shapes = synth.window_shapes(layers)
        self.dev = []
        self.host = [] if host_copy else None
        for name, rows, cols, fmt in self.shapes:
            w = synth.make_weights(rows, cols, fmt, key, name)
            self.dev.append(torch.from_numpy(w.buf).to(device))
            if host_copy:
                self.host.append(w)
        self.weight_bytes = sum(synth.weight_nbytes(r, c, f) for _, r, c, f in self.shapes)


class VerifyWindow:
    """Buffers and launch sequence of one T-token window over ``WindowWeights``."""

    def __init__(self, weights: WindowWeights, T: int, device="cuda", key="window-x", logits=False):
        assert 1 <= T <= strata.MAX_T
        self.wts, self.T = weights, T
        self.shapes = weights.shapes
        self.cols_total = sum(c for _, _, c, _ in self.shapes)
        # one flat fp32 input buffer (so a host->device copy of a step's inputs is one copy)
        self.x_flat = torch.empty(T * self.cols_total, dtype=torch.float32, device=device)
        self.x, self.xq, self.xd, self.xs, self.y = [], [], [], [], []
        off = 0
        for i, (name, rows, cols, fmt) in enumerate(self.shapes):
            xi = self.x_flat[off: off + T * cols].view(T, cols)
            off += T * cols
            self.x.append(xi)
            self.xq.append(torch.empty((T, cols), dtype=torch.int8, device=device))
            self.xd.append(torch.empty((T, cols // 32), dtype=torch.float32, device=device))
            self.xs.append(torch.empty((T, cols // 32), dtype=torch.int32, device=device))
            last = i == len(self.shapes) - 1
            self.y.append(torch.empty((T, rows), dtype=torch.float32, device=device)
                          if (not last or logits) else None)
        self.ids = torch.empty(T, dtype=torch.int32, device=device)
        vocab, hid = self.shapes[-1][1], self.shapes[-1][2]
        self.head_ws = torch.empty(strata.head_argmax_workspace(vocab, T), dtype=torch.uint8, device=device)
        self.key = key

    def host_inputs(self) -> np.ndarray:
        """The seeded fp32 inputs of every projection, flattened in launch order."""
        parts = [synth.make_activations(self.T, cols, self.key, name).reshape(-1)
                 for name, rows, cols, fmt in self.shapes]
        return np.concatenate(parts)

    def load_inputs(self, host: np.ndarray | None = None) -> None:
        host = self.host_inputs() if host is None else host
        self.x_flat.copy_(torch.from_numpy(host))

    def launches_per_step(self) -> int:
        return 2 * (len(self.shapes) - 1) + 3   # quantize + GEMV per layer matrix; quantize + head + finalize

    def enqueue(self, stream=None, first: int = 0, last: int | None = None) -> None:
        """Enqueue the window's matrices [first, last) (default: all) on ``stream`` (default: torch's
        current stream): quantize each input, then its GEMV, or the head GEMV + argmax."""
        n = len(self.shapes)
        last = n if last is None else last
        for i in range(first, last):
            name, rows, cols, fmt = self.shapes[i]
            strata.quantize_act(self.x[i], self.xq[i], self.xd[i], self.xs[i], stream=stream)
            if i < n - 1:
                strata.mmvq_multi(self.wts.dev[i], rows, cols, fmt, self.xq[i], self.xd[i], self.xs[i],
                                  self.T, self.y[i], stream=stream)
            else:
                strata.head_argmax(self.wts.dev[i], rows, cols, fmt, self.xq[i], self.xd[i], self.xs[i],
                                   self.T, self.ids, self.y[i], self.head_ws, stream=stream)

    def capture(self, first: int = 0, last: int | None = None) -> torch.cuda.CUDAGraph:
        """One CUDA graph of matrices [first, last) (default: the whole step), after one eager
        warm-up pass on a side stream."""
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.enqueue(first=first, last=last)
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.enqueue(first=first, last=last)
        return g

    def run_host(self, graph: torch.cuda.CUDAGraph, x_host: torch.Tensor, ids_host: torch.Tensor) -> None:
        """End to end from host buffers: copy the step's inputs in, run the window, copy the ids out
        (asynchronous on the current stream; pinned host tensors make the copies asynchronous)."""
        self.x_flat.copy_(x_host, non_blocking=True)
        graph.replay()
        ids_host.copy_(self.ids, non_blocking=True)
