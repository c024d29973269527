#!/usr/bin/env python3
"""Benchmark of the block-quantized verify window on GB300.

One step = one full verify window (48 layers x {qkv, o, up, down} Q4 projections + the Q8 head
GEMV and per-token argmax) at T tokens: quantize each projection's T input rows, run the T-column
GEMV, finish with the head's argmax. The step is one CUDA graph replayed K times after W warm-up
replays. Weights (1.52 GB) are larger than L2, so every step streams them from HBM.

Prints ONE JSON line (rank 0). --impl reference times the CPU oracle instead (the reference arm).
Multi-GPU: one process per GPU under torchrun; every rank runs its own independent windows
(weak scaling, no collective on the data path); the timed region is bracketed by barriers and the
maximum time over ranks is reported.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verify-window tokens/s and weight GB/s (% of HBM roofline) at T=1/2/4/8"
WORKLOAD = ("full verify window: 48 layers x {qkv 2048->5120, o 4096->2048, up 2048->6144, "
            "down 6144->2048} Q4 + Q8 head 151936x2048 with per-token argmax")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="strata", choices=["strata", "reference"])
    ap.add_argument("--T", type=int, default=4)
    ap.add_argument("--layers", type=int, default=48)
    ap.add_argument("--no-moe", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the decode GEMV and verify FFN lines")
    ap.add_argument("--case", default="window",
                    choices=["window", "mmvq", "head", "moe", "layers", "mma_peaks", "gemm"],
                    help="window: the timed step; mmvq/head/moe/layers: a few launches of one kernel "
                         "(profiling); mma_peaks: cuBLAS int8 vs fp16 dense GEMM rates on this GPU")
    ap.add_argument("--rows", type=int, default=2048)
    ap.add_argument("--cols", type=int, default=6144)
    ap.add_argument("--fmt", type=int, default=0)
    ap.add_argument("--reps", type=int, default=5)
    return ap.parse_args()


def tensor_peak():
    """Dense fp16/bf16 tensor peak (the MoE MMAs are kind::f16): the measured bf16 figure (same rate)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (bf16 burst; fp16 runs at the same rate)"
    except Exception:
        return 1900.0, "fallback"


def recorded_traffic(kernel_file: str, key: str):
    """Per-launch DRAM bytes of a kernel from a committed ncu summary, or None when the kernel's
    source has changed since the counters were taken (the summary stores the source's sha256)."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[key]
        with open(os.path.join(ROOT, "block_quantized_token_strata_gb300", "csrc", kernel_file), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != rec["source_sha256"]:
                return None
        return rec["dram_bytes_per_launch"]
    except Exception:
        return None


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---- CPU oracle baseline: the whole window ----------------------------------------------------------
class OracleWindow:
    """The oracle on the full verify window as it stands: each projection's T input rows quantized,
    every row of every layer matrix and of the head at T tokens, the head's argmax. ``run()`` is one
    whole window; ``run(n_layer_mats)`` covers only the first layer matrices and the head (a bounded
    sample for long reference runs) and returns the share of the window's weight x token work it did.
    The oracle runs one OpenMP thread per core this process may use (sched_getaffinity)."""

    def __init__(self, T: int, layers: int, host_weights=None):
        import oracle
        from block_quantized_token_strata_gb300 import synth
        oracle.build()
        self.cores = len(os.sched_getaffinity(0))
        oracle.set_threads(self.cores)
        self.oracle, self.T = oracle, T
        shapes = synth.window_shapes(layers)
        self.total = sum(r * c for _, r, c, _ in shapes)
        self.mats = []
        for i, (name, rows, cols, fmt) in enumerate(shapes):
            w = host_weights[i] if host_weights is not None else synth.make_weights(rows, cols, fmt, "window", name)
            self.mats.append((name, w.buf, rows, cols, fmt, synth.make_activations(T, cols, "window-x", name)))

    def run(self, n_layer_mats: int | None = None) -> float:
        o = self.oracle
        sel = self.mats if n_layer_mats is None else self.mats[:n_layer_mats] + self.mats[-1:]
        part = 0
        for name, buf, rows, cols, fmt, x in sel:
            xq, xd, _ = o.quantize_act(x)
            y, _ = o.mmvq(buf, rows, cols, fmt, xq, xd)
            if name == "head":
                o.argmax(y)
            part += rows * cols
        return part / self.total

    def full_rate(self, reps: int = 3):
        """Median wall time of ``reps`` whole windows -> (tokens/s, seconds per window)."""
        times = []
        for _ in range(reps):
            t0 = time.perf_counter()
            self.run()
            times.append(time.perf_counter() - t0)
        per = statistics.median(times)
        return self.T / per, per


# ---- clocks ----------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if uuid:
            cmd += ["-i", uuid]
        try:
            self.p = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None

    def stop(self) -> dict:
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except Exception:
            self.p.kill()
            out = ""
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [v.strip() for v in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---- reference arm -------------------------------------------------------------------------------------
def run_reference(args, rank: int) -> None:
    """The CPU oracle timed as it stands on the same window. Each step is one whole window when the
    --steps/--warmup run fits in about four minutes that way (the normal case); for longer runs each
    step covers the first layer matrices and the head, and the line says so."""
    if rank != 0:
        return
    smp = OracleWindow(args.T, args.layers)
    t0 = time.perf_counter()
    smp.run()                                   # the first warm-up step, timed to size the rest
    t_full = time.perf_counter() - t0
    n_steps = args.steps + max(args.warmup - 1, 0)
    n_mats = None
    if n_steps * t_full > 240.0:                # bounded sample per step
        share_target = max(0.01, 240.0 / n_steps / t_full)
        n_mats = max(1, int(share_target * (len(smp.mats) - 1)))
    for _ in range(max(args.warmup - 1, 0)):
        smp.run(n_mats)
    times, share = [], 1.0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        share = smp.run(n_mats)
        times.append(time.perf_counter() - t0)
    per_window = statistics.median(times) / share
    value = args.T / per_window
    if n_mats is None:
        sample = f"per step one whole window (192 layer matrices + the head, T={args.T}); median of {args.steps} steps"
    else:
        sample = (f"per step the first {n_mats} layer matrices and the head ({share:.2%} of the window's weight x "
                  f"token work), T={args.T}; time divided by that share")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "T": args.T, "layers": args.layers},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": smp.cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---- multi-process bookkeeping (one process per GPU under torchrun; replicas, no data exchange) ----
def dist_env():
    """(world size, global rank, local rank) from the launcher's environment; (1, 0, 0) alone."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time for the timed region (all_reduce MAX); the identity for one process."""
    if world == 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, units_per_rank: float, ms: float) -> float:
    """Whole-job throughput: every rank processed ``units_per_rank`` in at most ``ms``."""
    return world * units_per_rank / (ms * 1e-3)


# ---- GPU arm -------------------------------------------------------------------------------------------
def main():
    args = parse()
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if args.case != "window":
        run_case(args)
        return

    import torch
    import torch.distributed as dist
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    from block_quantized_token_strata_gb300 import build, strata, synth
    from block_quantized_token_strata_gb300.window import VerifyWindow, WindowWeights
    build.build()
    hbm_peak, peak_kind = peaks()

    wts = WindowWeights(layers=args.layers, device="cuda", host_copy=(rank == 0 and not args.no_cpu))
    T = args.T
    wins = {t: VerifyWindow(wts, t) for t in sorted({1, 2, 4, 8, T})}
    for w in wins.values():
        w.load_inputs()
    graphs = {t: w.capture() for t, w in wins.items()}
    torch.cuda.synchronize()
    launches = wins[T].launches_per_step()

    # --- headline: K steps of the T-token window, device-resident inputs ---
    g = graphs[T]
    for _ in range(args.warmup):
        g.replay()
    try:
        uuid = str(torch.cuda.get_device_properties(local).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    barrier()
    sampler = ClockSampler(uuid) if rank == 0 else None
    time.sleep(0.3 if rank == 0 else 0.0)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        g.replay()
    e1.record()
    barrier()
    clocks = sampler.stop() if sampler else None
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, "cuda")
    value = job_rate(world, T, ms)

    # --- per-T lines (same graph structure), weight GB/s ---
    per_T = {}
    for t, gg in graphs.items():
        for _ in range(3):
            gg.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n = max(20, args.steps // 5)
        a.record()
        for _ in range(n):
            gg.replay()
        b.record()
        torch.cuda.synchronize()
        mt = a.elapsed_time(b) / n
        gbs = wts.weight_bytes / (mt * 1e-3) / 1e9
        per_T[str(t)] = {"ms_per_window": mt, "tokens_per_s": t / (mt * 1e-3), "weight_gbs": gbs,
                         "hbm_frac": gbs / hbm_peak}

    # --- roofline of the dominant kernel: the grouped layer GEMV launch. The same launches as the
    # step, captured as two graphs (layers = one quantize launch + grouped GEMV; head) so that CUDA
    # events on the launching stream bracket each part.
    win = wins[T]
    g_lay, g_head = win.capture("layers"), win.capture("head")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    lay, head = [], []
    for i in range(max(20, args.steps // 10)):
        ev[0].record()
        g_lay.replay()
        ev[1].record()
        g_head.replay()
        ev[2].record()
        torch.cuda.synchronize()
        if i >= 3:
            lay.append(ev[0].elapsed_time(ev[1]))
            head.append(ev[1].elapsed_time(ev[2]))
    layer_bytes = sum(synth.weight_nbytes(r, c, f) + T * c * 1.25 + T * r * 4 for _, r, c, f in win.shapes[:-1])
    lay_ms = statistics.median(lay)
    achieved = layer_bytes / (lay_ms * 1e-3) / 1e9
    _, vr, vc, vf = win.shapes[-1]
    head_bytes = synth.weight_nbytes(vr, vc, vf) + T * vc * 1.25
    head_ms = statistics.median(head)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak, "traffic": recorded_traffic("mmvq.cu", f"layers_T{T}"),
                "kernel": "gemv_kernel<Q4,T,grouped>: one launch streams all 192 layer matrices",
                "bytes_per_launch": layer_bytes, "us_per_launch": lay_ms * 1e3,
                "peak_kind": peak_kind,
                "note": "time of the layer section = the quantize launch + the grouped GEMV launch",
                "head": {"gbs": head_bytes / (head_ms * 1e-3) / 1e9, "us": head_ms * 1e3,
                         "frac": head_bytes / (head_ms * 1e-3) / 1e9 / hbm_peak}}

    # --- batch head: 8 independent sequences at one token each, ids + top-2 margin per sequence
    wb = wins[8]
    hb = {"T": 8}
    ids_b = torch.empty(8, dtype=torch.int32, device="cuda")
    mg_b = torch.empty(8, dtype=torch.float32, device="cuda")
    def head_margin():
        strata.head_argmax_margin(wb.wts.dev[-1], vr, vc, vf, wb.xq[-1], wb.xd[-1], wb.xs[-1], 8, ids=ids_b,
                                  margin=mg_b, workspace=wb.head_ws)
    for _ in range(3):
        head_margin()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(20):
        head_margin()
    b.record()
    torch.cuda.synchronize()
    hm_ms = a.elapsed_time(b) / 20
    hb_bytes = synth.weight_nbytes(vr, vc, vf) + 8 * vc * 1.25
    hb.update({"us": hm_ms * 1e3, "gbs": hb_bytes / (hm_ms * 1e-3) / 1e9,
               "frac": hb_bytes / (hm_ms * 1e-3) / 1e9 / hbm_peak,
               "note": "strata_head_argmax_margin on the Q8 head: ids and top-1 minus top-2 logit per sequence"})

    # --- the same window with one quantize + GEMV launch per projection (chained launch structure)
    wch = VerifyWindow(wts, T, mode="chained")
    wch.load_inputs()
    gch = wch.capture()
    for _ in range(3):
        gch.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    n_ch = max(20, args.steps // 5)
    for _ in range(n_ch):
        gch.replay()
    b.record()
    torch.cuda.synchronize()
    ch_ms = a.elapsed_time(b) / n_ch
    chained = {"ms_per_window": ch_ms, "tokens_per_s": T / (ch_ms * 1e-3),
               "weight_gbs": wts.weight_bytes / (ch_ms * 1e-3) / 1e9,
               "hbm_frac": wts.weight_bytes / (ch_ms * 1e-3) / 1e9 / hbm_peak,
               "launches": wch.launches_per_step()}
    del wch, gch

    # --- end to end through the public API: pinned host inputs in, ids out, every step. Each step's
    # input copy streams in while the previous window computes (two device input buffers, one CUDA
    # graph each, a copy stream); two input sets alternate. ---
    from block_quantized_token_strata_gb300.window import HostPipeline
    pipe = HostPipeline(win)
    host0 = win.host_inputs()
    x_hosts = [torch.from_numpy(host0).pin_memory(), torch.from_numpy(np.ascontiguousarray(host0[::-1])).pin_memory()]
    n_e2e = max(20, args.steps // 5)
    ids_hosts = [torch.empty(T, dtype=torch.int32).pin_memory() for _ in range(n_e2e)]
    pipe.run([x_hosts[k & 1] for k in range(3)], ids_hosts[:3])
    barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall = time.perf_counter()
    a.record()
    pipe.run([x_hosts[k & 1] for k in range(n_e2e)], ids_hosts)
    b.record()
    barrier()
    wall = (time.perf_counter() - t_wall) / n_e2e
    e2e_ms = a.elapsed_time(b) / n_e2e
    e2e_ms = max_over_ranks(max(e2e_ms, wall * 1e3), world, "cuda")
    e2e = {"value": job_rate(world, T, e2e_ms), "unit": "tokens/s",
           "h2d_bytes_per_step": int(x_hosts[0].numel() * 4), "d2h_bytes_per_step": int(T * 4),
           "overlap": "each step's host->device input copy runs on a copy stream during the previous window"}
    del pipe

    # --- prompt-chunk MoE (grouped experts), reported beside the window ---
    moe = gemm = q6 = None
    if not args.no_moe:
        moe = bench_moe(torch, strata, synth, args)
        gemm = bench_prompt_gemm(torch, strata, synth)
        q6 = {name: bench_superblock_layers(torch, strata, synth, hbm_peak, fmt)
              for name, fmt in (("Q6", synth.Q6), ("Q4K", synth.Q4K), ("Q5K", synth.Q5K))}

    decode = ffn = None
    if not args.no_configs:
        decode = bench_decode(torch, strata, synth, hbm_peak)
        ffn = bench_verify_ffn(torch, strata, synth, hbm_peak)

    cpu = None
    if rank == 0 and not args.no_cpu:
        ow = OracleWindow(T, args.layers, wts.host)
        rate, per = ow.full_rate(3)
        cpu = {"value": rate, "unit": "tokens/s", "cores": ow.cores, "kind": "oracle",
               "sample": f"3 whole windows (192 layer matrices + the head, T={T}), median {per:.2f} s a window"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int8 dots (dp4a, exact int32) + fp32 scale/accumulate",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "T": T, "layers": args.layers,
                       "weight_bytes_per_window": wts.weight_bytes,
                       "l2": "inputs larger than L2 (1.52 GB of weights per step)",
                       "graph": "one CUDA graph per window: one quantize launch over every input, one grouped GEMV "
                                "launch over the 192 layer matrices, head GEMV + argmax"},
            "weight_gbs": wts.weight_bytes / (ms * 1e-3) / 1e9 * world,
            "hbm_frac": wts.weight_bytes / (ms * 1e-3) / 1e9 / hbm_peak,
            "per_T": per_T, "chained_launches": chained, "batch_head_margin": hb, "roofline": roofline,
            "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches * args.steps, "clocks": clocks, "moe": moe, "prompt_gemm": gemm,
            "superblock_layers": q6, "decode_gemv": decode, "verify_ffn": ffn,
            "device_error_word": strata.device_error(),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def _graph(torch, fn):
    """One CUDA graph of fn() (after one eager pass on a side stream)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def _time_graph(torch, g, reps):
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def _rotating_copies(torch, nbytes):
    """How many weight copies make ceil(3 L2 / size): a rotation through them streams from HBM."""
    l2 = int(torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size)
    return max(2, -(-3 * l2 // nbytes)), l2


def bench_decode(torch, strata, synth, hbm_peak, reps=20):
    """Decode GEMV: one token (T = 1) through a 4096 x 4096 matrix in Q4 and in Q8, activations N(0,1)
    with 1% of elements x20, one quantize launch + one GEMV launch a step. The matrix fits in L2, so
    the steps run as one CUDA graph over ceil(3 L2 / size) weight copies in turn (each step reads
    its copy from HBM)."""
    rows = cols = 4096
    x = torch.from_numpy(synth.make_activations(1, cols, "decode", outliers=True)).cuda()
    xq = torch.empty((1, cols), dtype=torch.int8, device="cuda")
    xd = torch.empty((1, cols // 32), dtype=torch.float32, device="cuda")
    xs = torch.empty((1, cols // 32), dtype=torch.int32, device="cuda")
    y = torch.empty((1, rows), dtype=torch.float32, device="cuda")
    out = {"workload": "4096x4096, T=1, activations with 1% outliers x20; quantize + GEMV per step"}
    for name, fmt in (("Q4", synth.Q4), ("Q8", synth.Q8)):
        nbytes = synth.weight_nbytes(rows, cols, fmt)
        n, l2 = _rotating_copies(torch, nbytes)
        W0 = torch.from_numpy(synth.make_weights(rows, cols, fmt, "decode").buf).cuda()
        copies = [W0.clone() for _ in range(n)]

        def steps():
            for Wc in copies:
                strata.quantize_act(x, xq, xd, xs)
                strata.mmvq_multi(Wc, rows, cols, fmt, xq, xd, xs, 1, y)
        g = _graph(torch, steps)
        ms = _time_graph(torch, g, reps) / n
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"us": ms * 1e3, "tokens_per_s": 1.0 / (ms * 1e-3), "weight_gbs": gbs, "hbm_frac": gbs / hbm_peak,
                     "roofline_us": nbytes / (hbm_peak * 1e9) * 1e6, "weight_bytes": nbytes, "copies": n,
                     "l2_bytes": l2}
        del g, copies, W0
    torch.cuda.empty_cache()
    return out


def bench_verify_ffn(torch, strata, synth, hbm_peak, reps=20):
    """Verify-window FFN: a Q4 up projection 4096 -> 14336 and a down projection 14336 -> 4096 (66 MB)
    at T = 1/2/3/4/8 columns, each input its own seeded N(0,1) rows (no activation function between
    them). Per step either one quantize launch over both inputs + one grouped GEMV launch of the two
    matrices ("grouped"), or a quantize + GEMV launch per projection ("chained"). Timed as one CUDA
    graph over ceil(3 L2 / size) weight copies in turn."""
    H, F = 4096, 14336
    shapes = (("up", F, H), ("down", H, F))
    nbytes = sum(synth.weight_nbytes(r, c, synth.Q4) for _, r, c in shapes)
    n, l2 = _rotating_copies(torch, nbytes)
    base = [torch.from_numpy(synth.make_weights(r, c, synth.Q4, "verify-ffn", nm).buf).cuda() for nm, r, c in shapes]
    copies = [[b.clone() for b in base] for _ in range(n)]
    out = {"workload": "Q4 up 4096->14336 + down 14336->4096, independent inputs", "weight_bytes": nbytes,
           "copies": n, "roofline_us": nbytes / (hbm_peak * 1e9) * 1e6}
    for T in (1, 2, 3, 4, 8):
        tot = T * (H + F)
        xf = torch.from_numpy(np.concatenate([synth.make_activations(T, c, "verify-ffn-x", nm).reshape(-1)
                                              for nm, _, c in shapes])).cuda()
        qf = torch.empty(tot, dtype=torch.int8, device="cuda")
        df = torch.empty(tot // 32, dtype=torch.float32, device="cuda")
        sf = torch.empty(tot // 32, dtype=torch.int32, device="cuda")
        xs_ = [xf[:T * H].view(T, H), xf[T * H:].view(T, F)]
        qs = [qf[:T * H].view(T, H), qf[T * H:].view(T, F)]
        ds = [df[:T * H // 32].view(T, H // 32), df[T * H // 32:].view(T, F // 32)]
        ss = [sf[:T * H // 32].view(T, H // 32), sf[T * H // 32:].view(T, F // 32)]
        ys = [torch.empty((T, r), dtype=torch.float32, device="cuda") for _, r, _ in shapes]
        descs = [strata.gemv_descs([(cp[i], shapes[i][1], shapes[i][2], qs[i], ds[i], ss[i], ys[i]) for i in range(2)])
                 for cp in copies]

        def grouped():
            for d in descs:
                strata.quantize_act(xf.view(1, -1), qf.view(1, -1), df.view(1, -1), sf.view(1, -1))
                strata.mmvq_grouped(d, synth.Q4, T)

        def chained():
            for cp in copies:
                for i, (_, r, c) in enumerate(shapes):
                    strata.quantize_act(xs_[i], qs[i], ds[i], ss[i])
                    strata.mmvq_multi(cp[i], r, c, synth.Q4, qs[i], ds[i], ss[i], T, ys[i])
        line = {}
        for mode, fn in (("grouped", grouped), ("chained", chained)):
            g = _graph(torch, fn)
            ms = _time_graph(torch, g, reps) / n
            gbs = nbytes / (ms * 1e-3) / 1e9
            line[mode] = {"us": ms * 1e3, "tokens_per_s": T / (ms * 1e-3), "weight_gbs": gbs,
                          "hbm_frac": gbs / hbm_peak}
            del g
        out[f"T{T}"] = line
    del copies, base
    torch.cuda.empty_cache()
    return out


def bench_superblock_layers(torch, strata, synth, hbm_peak, fmt, layers=None, reps=20):
    """The window's layer projections in a 256-weight super-block format (Q6, Q4K or Q5K; one grouped
    launch per window over the full window's 48 layers, 1.22-1.73 GB of weights) at T = 2 and 4:
    weight GB/s and HBM fraction."""
    layers = synth.WINDOW_LAYERS if layers is None else layers
    from block_quantized_token_strata_gb300.window import VerifyWindow, WindowWeights
    name = {synth.Q6: "Q6", synth.Q4K: "Q4K", synth.Q5K: "Q5K"}[fmt]
    wts = WindowWeights(layers=layers, device="cuda", key=f"{name}-window", layer_fmt=fmt)
    lay_bytes = sum(synth.weight_nbytes(r, c, f) for _, r, c, f in wts.shapes[:-1])
    out = {"workload": f"{layers} layers x {{qkv 2048->5120, o 4096->2048, up 2048->6144, down 6144->2048}} {name}",
           "weight_bytes": lay_bytes}
    for T in (2, 4):
        win = VerifyWindow(wts, T)
        win.load_inputs()
        g = win.capture("layers")
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / reps
        gbs = lay_bytes / (ms * 1e-3) / 1e9
        out[f"T{T}"] = {"us": ms * 1e3, "weight_gbs": gbs, "hbm_frac": gbs / hbm_peak}
        del g, win
    del wts
    torch.cuda.empty_cache()
    return out


def bench_prompt_gemm(torch, strata, synth, reps=20):
    """The dense prompt GEMM: a 3,259-token chunk against the window's FFN up projection (Q4 6144 x 2048),
    in both arms: no dequantization (tile operands converted from the Q4 codes inside the kernel) and
    wide dequant (one conversion pass to fp16 operand tiles per call, then a bulk-copy-fed GEMM; the
    time is the whole call, conversion included). Both give bitwise equal outputs."""
    rows, cols, n_tok = 6144, 2048, 3259
    W = torch.from_numpy(synth.make_weights(rows, cols, synth.Q4, "prompt-gemm").buf).cuda()
    xq, xd, _ = strata.quantize_act(torch.from_numpy(synth.make_activations(n_tok, cols, "prompt-gemm")).cuda())
    y = torch.empty((n_tok, rows), dtype=torch.float32, device="cuda")
    ws = torch.empty(strata.gemm_q4_dequant_workspace(rows, cols, n_tok), dtype=torch.uint8, device="cuda")
    peak, kind = tensor_peak()
    out = {"workload": "3,259-token prompt chunk x Q4 6144x2048 (the window's FFN up projection)"}
    arms = (("no_dequant", lambda: strata.gemm_q4(W, rows, cols, xq, xd, y=y)),
            ("wide_dequant", lambda: strata.gemm_q4_dequant(W, rows, cols, xq, xd, y=y, workspace=ws)))
    for name, fn in arms:
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / reps
        tf = 2.0 * n_tok * rows * cols / (ms * 1e-3) / 1e12
        out[name] = {"ms": ms, "tokens_per_s": n_tok / (ms * 1e-3),
                     "tensor": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s", "frac": tf / peak,
                                "peak_kind": kind}}
    best = min(("no_dequant", "wide_dequant"), key=lambda k: out[k]["ms"])
    out["faster_arm"] = best
    out["ms"] = out[best]["ms"]
    out["tensor"] = out[best]["tensor"]
    del ws
    return out


def bench_moe(torch, strata, synth, args, reps=20):
    """One prompt chunk of the MoE experts (3,256 tokens, 128 experts, top-8), CUDA graph replays."""
    E, H, I, N, K = synth.MOE_EXPERTS, synth.MOE_HIDDEN, synth.MOE_INTER, synth.MOE_TOKENS, synth.MOE_TOPK
    dev = [tuple(torch.from_numpy(synth.make_weights(r, c, synth.Q4, "prompt-moe", w, e).buf).cuda()
                 for w, r, c in (("g", I, H), ("u", I, H), ("d", H, I))) for e in range(E)]
    tab = strata.expert_table(dev, "cuda")
    ids = torch.from_numpy(synth.make_routing(N, E, K, "prompt-moe")).cuda()
    x = torch.from_numpy(synth.make_activations(N, H, "prompt-moe")).cuda()
    y = torch.empty((N * K, H), dtype=torch.float32, device="cuda")
    ws = torch.empty(strata.moe_grouped_workspace(E, N, K, H, I), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def step():
        strata.moe_grouped(tab, E, H, I, ids, x, y=y, workspace=ws, err_word=err)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = reps
    a.record()
    for _ in range(n):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / n
    flops = 2.0 * N * K * (2 * I * H + H * I)   # the integer block dots, run as exact fp16 MMAs
    peak, kind = tensor_peak()
    tf = flops / (ms * 1e-3) / 1e12
    return {"workload": "3,256 tokens x top-8 of 128 experts, Q4 gate/up 2048->768, down 768->2048",
            "ms_per_chunk": ms, "tokens_per_s": N / (ms * 1e-3),
            "tensor": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s", "frac": tf / peak,
                       "peak_kind": kind, "mma": "tcgen05.mma kind::f16 (fp16 operands holding the exact codes)"},
            "err_word": int(err.item())}


def run_case(args):
    """A few plain launches of one kernel on one workload (for profilers); prints its mean time."""
    import torch
    from block_quantized_token_strata_gb300 import build, strata, synth
    build.build()
    torch.cuda.set_device(0)
    T = args.T
    if args.case == "mma_peaks":  # why the MoE runs its exact integer dots as fp16 MMAs
        n = 8192
        out = {"case": "mma_peaks", "shape": f"{n}x{n}x{n}", "how": "cuBLAS via torch, best of 10, CUDA events"}
        a8 = torch.randint(-127, 128, (n, n), dtype=torch.int8, device="cuda")
        b8 = torch.randint(-127, 128, (n, n), dtype=torch.int8, device="cuda")
        ah, bh = a8.to(torch.float16), b8.to(torch.float16)
        ab, bb = a8.to(torch.bfloat16), b8.to(torch.bfloat16)
        for name, fn in (("int8_tops", lambda: torch._int_mm(a8, b8.t())),
                         ("fp16_tflops", lambda: torch.matmul(ah, bh.t())),
                         ("bf16_tflops", lambda: torch.matmul(ab, bb.t()))):
            try:
                for _ in range(3):
                    fn()
                torch.cuda.synchronize()
            except Exception as exc:  # an unsupported layout or dtype on this build: say so
                out[name] = f"unavailable: {type(exc).__name__}: {exc}"[:200]
                continue
            best = 1e9
            for _ in range(10):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                fn()
                b.record()
                torch.cuda.synchronize()
                best = min(best, a.elapsed_time(b))
            out[name] = 2.0 * n ** 3 / (best * 1e-3) / 1e12
        print(json.dumps(out))
        return
    if args.case == "gemm":  # the dense prompt GEMM
        print(json.dumps({"case": "gemm", **bench_prompt_gemm(torch, strata, synth, reps=args.reps)}))
        return
    if args.case == "layers":  # the window's grouped layer launch (one quantize launch + one GEMV launch)
        from block_quantized_token_strata_gb300.window import VerifyWindow, WindowWeights
        wts = WindowWeights(layers=args.layers, device="cuda", layer_fmt=args.fmt)
        win = VerifyWindow(wts, T)
        win.load_inputs()
        g = win.capture("layers")
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.reps):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / args.reps
        nbytes = wts.weight_bytes - synth.weight_nbytes(synth.HEAD_VOCAB, synth.WINDOW_HIDDEN, synth.Q8)
        print(json.dumps({"case": "layers", "layers": args.layers, "fmt": args.fmt, "T": T, "us": ms * 1e3,
                          "weight_gbs": nbytes / (ms * 1e-3) / 1e9, "device_error": strata.device_error()}))
        return
    if args.case in ("mmvq", "head"):
        rows = synth.HEAD_VOCAB if args.case == "head" else args.rows
        cols = synth.WINDOW_HIDDEN if args.case == "head" else args.cols
        fmt = synth.Q8 if args.case == "head" else args.fmt
        W = torch.from_numpy(synth.make_weights(rows, cols, fmt, "case").buf).cuda()
        xq, xd, xs = strata.quantize_act(torch.from_numpy(synth.make_activations(T, cols, "case")).cuda())
        y = torch.empty((T, rows), dtype=torch.float32, device="cuda")
        ids = torch.empty(T, dtype=torch.int32, device="cuda")
        ws = torch.empty(strata.head_argmax_workspace(rows, T), dtype=torch.uint8, device="cuda")

        def step():
            if args.case == "head":
                strata.head_argmax(W, rows, cols, fmt, xq, xd, xs, T, ids, None, ws)
            else:
                strata.mmvq_multi(W, rows, cols, fmt, xq, xd, xs, T, y)
        nbytes = synth.weight_nbytes(rows, cols, fmt)
    else:
        out = bench_moe(torch, strata, synth, args, reps=args.reps)
        print(json.dumps({"case": "moe", **out}))
        return
    for _ in range(2):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.reps):
        step()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.reps
    print(json.dumps({"case": args.case, "rows": rows, "cols": cols, "fmt": fmt, "T": T, "us": ms * 1e3,
                      "weight_gbs": nbytes / (ms * 1e-3) / 1e9}))


if __name__ == "__main__":
    main()
