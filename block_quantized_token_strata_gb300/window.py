"""A full verify window on one GPU: every projection of every layer, then the head's argmax.

One step reads every dense weight byte of the window once for T tokens: 48 layers x (qkv, o, up,
down) Q4 projections, then the Q8 head GEMV with its per-token argmax. The layers are not chained
(there is no model between them): each projection has its own seeded fp32 input. Two launch
structures are provided:

  * "grouped" (the step the benchmark times): every input is quantized by ONE launch (inputs, codes,
    scales and sums are each one flat buffer in the same block order), all 192 layer GEMVs run as
    ONE grouped launch (strata_mmvq_grouped: the matrices stream back to back, every SM busy), then
    the head GEMV + argmax;
  * "chained": one quantize + one GEMV launch per projection, each kernel ordered after the one
    before it — the launch structure a chained model would need — kept for comparison.

All work is enqueued through the C ABI on one stream and can be captured in one CUDA graph.
"""
from __future__ import annotations

import numpy as np
import torch

from . import strata, synth


class WindowWeights:
    """Device copies of every matrix of the window (generated once, seeded)."""

    def __init__(self, layers: int = synth.WINDOW_LAYERS, device="cuda", key="window", host_copy=False,
                 layer_fmt: int = synth.Q4):
        self.layer_fmt = layer_fmt
        self.shapes = synth.window_shapes(layers, layer_fmt)
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

    def __init__(self, weights: WindowWeights, T: int, device="cuda", key="window-x", logits=False,
                 mode: str = "grouped"):
        assert 1 <= T <= strata.MAX_T and mode in ("grouped", "chained")
        self.wts, self.T, self.mode, self.key = weights, T, mode, key
        self.shapes = weights.shapes
        n = len(self.shapes)
        # inputs grouped by width; x and its quantized codes, scales and sums are each one flat buffer
        # in the same block order, so one quantize launch covers every input of the window (the
        # quantizer works on each 32-value block alone, whatever the row length)
        self.widths = sorted({c for _, _, c, _ in self.shapes})
        members = {c: [i for i, s in enumerate(self.shapes) if s[2] == c] for c in self.widths}
        total = sum(T * c for _, _, c, _ in self.shapes)
        self.x_flat = torch.empty(total, dtype=torch.float32, device=device)
        self.q_flat = torch.empty(total, dtype=torch.int8, device=device)
        self.d_flat = torch.empty(total // 32, dtype=torch.float32, device=device)
        self.s_flat = torch.empty(total // 32, dtype=torch.int32, device=device)
        self.offset = [0] * n          # element offset of each projection's input in x_flat
        self.gx, self.gq, self.gd, self.gs = {}, {}, {}, {}
        off = 0
        for c in self.widths:
            k = len(members[c])
            self.gx[c] = self.x_flat[off: off + k * T * c].view(k * T, c)
            self.gq[c] = self.q_flat[off: off + k * T * c].view(k * T, c)
            self.gd[c] = self.d_flat[off // 32: (off + k * T * c) // 32].view(k * T, c // 32)
            self.gs[c] = self.s_flat[off // 32: (off + k * T * c) // 32].view(k * T, c // 32)
            for j, i in enumerate(members[c]):
                self.offset[i] = off + j * T * c
            off += k * T * c
        self.x, self.xq, self.xd, self.xs, self.y = [], [], [], [], []
        for i, (name, rows, cols, fmt) in enumerate(self.shapes):
            j = members[cols].index(i)
            self.x.append(self.gx[cols][j * T:(j + 1) * T])
            self.xq.append(self.gq[cols][j * T:(j + 1) * T])
            self.xd.append(self.gd[cols][j * T:(j + 1) * T])
            self.xs.append(self.gs[cols][j * T:(j + 1) * T])
            last = i == n - 1
            self.y.append(torch.empty((T, rows), dtype=torch.float32, device=device)
                          if (not last or logits) else None)
        self.ids = torch.empty(T, dtype=torch.int32, device=device)
        vocab = self.shapes[-1][1]
        self.head_ws = torch.empty(strata.head_argmax_workspace(vocab, T), dtype=torch.uint8, device=device)
        self.descs = strata.gemv_descs([(self.wts.dev[i], r, c, self.xq[i], self.xd[i], self.xs[i], self.y[i])
                                        for i, (_, r, c, _) in enumerate(self.shapes[:-1])])

    # ---- inputs ----
    def host_inputs(self) -> np.ndarray:
        """The seeded fp32 inputs of every projection, laid out as ``x_flat``."""
        out = np.empty(self.x_flat.numel(), dtype=np.float32)
        for i, (name, rows, cols, fmt) in enumerate(self.shapes):
            out[self.offset[i]: self.offset[i] + self.T * cols] = \
                synth.make_activations(self.T, cols, self.key, name).reshape(-1)
        return out

    def proj_input(self, host: np.ndarray, i: int) -> np.ndarray:
        """Projection i's [T][cols] input from a ``host_inputs`` array."""
        cols = self.shapes[i][2]
        return host[self.offset[i]: self.offset[i] + self.T * cols].reshape(self.T, cols)

    def load_inputs(self, host: np.ndarray | None = None) -> None:
        host = self.host_inputs() if host is None else host
        self.x_flat.copy_(torch.from_numpy(host))

    # ---- launches ----
    def launches_per_step(self) -> int:
        if self.mode == "grouped":
            return 1 + 1 + 2                    # one quantize, grouped GEMV, head + finalize
        return 2 * (len(self.shapes) - 1) + 3   # quantize + GEMV per layer matrix; quantize + head + finalize

    def enqueue(self, stream=None, part: str = "all", x_src: torch.Tensor | None = None) -> None:
        """Enqueue one window (``part``: "all", "layers" = everything before the head, "head"). In the
        grouped mode ``x_src`` (a buffer shaped like ``x_flat``) replaces ``x_flat`` as the input."""
        n = len(self.shapes)
        name, vocab, hcols, hfmt = self.shapes[-1]
        if self.mode == "grouped":
            if part in ("all", "layers"):
                xs = self.x_flat if x_src is None else x_src
                strata.quantize_act(xs.view(1, -1), self.q_flat.view(1, -1), self.d_flat.view(1, -1),
                                    self.s_flat.view(1, -1), stream=stream)
                strata.mmvq_grouped(self.descs, self.wts.layer_fmt, self.T, stream=stream)
        else:
            if part in ("all", "layers"):
                for i in range(n - 1):
                    _, rows, cols, fmt = self.shapes[i]
                    strata.quantize_act(self.x[i], self.xq[i], self.xd[i], self.xs[i], stream=stream)
                    strata.mmvq_multi(self.wts.dev[i], rows, cols, fmt, self.xq[i], self.xd[i], self.xs[i],
                                      self.T, self.y[i], stream=stream)
            if part in ("all", "head"):
                strata.quantize_act(self.x[n - 1], self.xq[n - 1], self.xd[n - 1], self.xs[n - 1], stream=stream)
        if part in ("all", "head"):
            strata.head_argmax(self.wts.dev[n - 1], vocab, hcols, hfmt, self.xq[n - 1], self.xd[n - 1],
                               self.xs[n - 1], self.T, self.ids, self.y[n - 1], self.head_ws, stream=stream)

    def capture(self, part: str = "all", x_src: torch.Tensor | None = None) -> torch.cuda.CUDAGraph:
        """One CUDA graph of ``part`` of the step, after one eager warm-up pass on a side stream."""
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.enqueue(part=part, x_src=x_src)
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.enqueue(part=part, x_src=x_src)
        return g

    def run_host(self, graph: torch.cuda.CUDAGraph, x_host: torch.Tensor, ids_host: torch.Tensor) -> None:
        """End to end from host buffers: copy the step's inputs in, run the window, copy the ids out
        (asynchronous on the current stream; pinned host tensors make the copies asynchronous)."""
        self.x_flat.copy_(x_host, non_blocking=True)
        graph.replay()
        ids_host.copy_(self.ids, non_blocking=True)


class HostPipeline:
    """Windows fed from host memory, each step's input copy overlapped with the previous window's
    compute: two device input buffers, a CUDA graph of the whole (grouped) window for each, and a copy
    stream. Every step still copies its own fp32 inputs host -> device and its ids device -> host; the
    copy into a buffer waits only for the window that last read that buffer."""

    def __init__(self, win: VerifyWindow):
        assert win.mode == "grouped"
        self.win = win
        self.xbuf = [win.x_flat, torch.empty_like(win.x_flat)]
        self.graphs = [win.capture(), win.capture(x_src=self.xbuf[1])]
        self.copy_stream = torch.cuda.Stream()
        self.copied = [torch.cuda.Event(), torch.cuda.Event()]
        self.consumed = [torch.cuda.Event(), torch.cuda.Event()]  # the window that read buffer j is done

    def _copy(self, j: int, x_host: torch.Tensor) -> None:
        with torch.cuda.stream(self.copy_stream):
            self.copy_stream.wait_event(self.consumed[j])
            self.xbuf[j].copy_(x_host, non_blocking=True)
            self.copied[j].record(self.copy_stream)

    def run(self, x_hosts, ids_hosts) -> None:
        """Windows k = 0 .. len(x_hosts) - 1 on the current stream (asynchronous): window k reads
        x_hosts[k] (pinned fp32, laid out as ``x_flat``) and leaves its ids in ids_hosts[k] (pinned)."""
        cur = torch.cuda.current_stream()
        self.copy_stream.wait_stream(cur)  # nothing of this run starts before the work already enqueued
        n = len(x_hosts)
        if n:
            self._copy(0, x_hosts[0])
        for k in range(n):
            j = k & 1
            if k + 1 < n:
                self._copy(j ^ 1, x_hosts[k + 1])   # streams in while window k computes
            cur.wait_event(self.copied[j])
            self.graphs[j].replay()
            self.consumed[j].record(cur)
            ids_hosts[k].copy_(self.win.ids, non_blocking=True)
