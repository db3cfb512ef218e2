"""Benchmark of the NVFP4 hot path on GB300; prints one JSON line.

Step (the headline): one decode-layer pass of the decode-shape workload. For
each token count M in {1, 2, 4, 8, 16}, bf16 activations x [M, K] go through
the three NVFP4 linears of a 31B-class layer (fused gate/up [43008, 5376],
down [5376, 21504], qkv [8192, 5376]), each with an E4M3/16 scale plane and a
per-linear float32 global scale: 15 QuantizedMatmuls, run by the public API
as one `nvfp4_qmm_sequence` call (one persistent decode launch for the whole
step). `value` is the algorithmic HBM traffic of those calls (9/16 byte per
weight element + activations + outputs + one global scale) divided by the
step time, in GB/s. Five rotating weight copies (1.1 GB per step) keep every
call's weights out of L2. The same 15 calls as single `nvfp4_qmm` calls (15
launches) are timed beside it (`step_single_calls`), and per call
(`us_per_call`).

`routes` reports the other configurations measured the same way (prefill
QuantizedMatmul TFLOP/s, MoE GatherQMM, transcode, dequantize) for context.

`--impl reference` times the CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

K_HIDDEN = 5376
LINEARS = (("gate_up", 43008, 5376), ("down", 5376, 21504), ("qkv", 8192, 5376))
DECODE_M = (1, 2, 4, 8, 16)
ROTATE = 5
WORKLOAD = ("decode-shape qmv: bf16 x [M in {1,2,4,8,16}, K] through NVFP4 gate/up [43008,5376], "
            "down [5376,21504], qkv [8192,5376]; E4M3/16 scales log-uniform in [2^-6,2^2]; "
            "per-linear f32 global scale in [0.5,2]*2688; bf16 out, f32 accumulate")
METRIC = "qmv HBM GB/s & µs/call, qmm TFLOP/s; fraction of GB300 roofline (1 GPU)"

# DRAM bytes (read + write) of the decode kernel over one step, from an ncu
# capture of `--case decode_step`; reported per launch, and only while the
# kernel sources still hash to kernel_sha.
TRAFFIC = {"kernel_sha": "ef5de1eef8d909cb", "bytes_per_step": 1128225024}
TRAFFIC_FILES = ("nvfp4_qmv_stream.cu", "nvfp4_qmv_common.cuh", "nvfp4_common.cuh", "nvfp4_pipe.cuh")


def qmv_bytes(m, n, k):
    return 0.5625 * n * k + 2 * m * k + 2 * m * n + 4


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            p = [v.strip() for v in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for name, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def source_sha(names):
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "nvfp4_quantized_matmul_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# ----------------------------------------------------------------------------- our arm

def build_decode(nv, synth, torch, dev, rank, copies=ROTATE):
    """Weights (`copies` rotating copies), activations and outputs for the decode step."""
    g = synth.rng(1000 + rank)
    ncopies = copies
    lin = []
    for name, n, k in LINEARS:
        copies = []
        for c in range(ncopies):
            w = torch.randint(-2**31, 2**31 - 1, (n, k // 8), dtype=torch.int32, device=dev,
                              generator=torch.Generator(device=dev).manual_seed(17 * c + n))
            s = torch.from_numpy(synth.log_uniform_scales(g, (n, k // 16), 2.0**-6, 4.0)).to(dev)
            gs = torch.from_numpy(synth.global_scales(g, 1)).to(dev)
            copies.append((w, s, gs))
        lin.append((name, n, k, copies))
    xs = {}
    for m in DECODE_M:
        for name, n, k, _ in lin:
            xs[(m, name)] = synth.activations(g, (m, k), "bf16").to(dev)
    ys = {(m, name): torch.empty((m, n), dtype=torch.bfloat16, device=dev) for m in DECODE_M for name, n, _, _ in lin}
    return lin, xs, ys


def decode_step_calls(nv, lin, xs, ys, copy_shift=0):
    calls = []
    for mi, m in enumerate(DECODE_M):
        for name, n, k, copies in lin:
            w, s, gs = copies[(mi + copy_shift) % len(copies)]
            calls.append((m, n, k, xs[(m, name)], w, s, gs, ys[(m, name)]))
    return calls


def reduce_step_time(torch, dist, dev, ms_total):
    """The timed region's length for the whole job: the maximum over ranks
    (replicas run independently; the job ends with its slowest rank)."""
    if dist is None:
        return ms_total
    t = torch.tensor([ms_total], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(step_bytes, world, ms_step):
    """Whole-job throughput in GB/s: every rank moves step_bytes per step."""
    return step_bytes * world / (ms_step * 1e-3) / 1e9


def run_ours(args):
    import torch

    import nvfp4_quantized_matmul_gb300 as nv
    from nvfp4_quantized_matmul_gb300 import synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    hbm_peak, bf16_peak, peak_kind = peaks()

    # Decode-step weights are constant, so consecutive calls may overlap
    # (programmatic dependent launch): each call starts streaming its weights
    # while the previous one finishes; activations and outputs stay ordered.
    nv.set_launch_overlap(args.launch_overlap == "on")
    lin, xs, ys = build_decode(nv, synth, torch, dev, rank)
    step_bytes = sum(qmv_bytes(m, n, k) for m in DECODE_M for _, n, k, _ in lin)
    launches_per_step = 1

    def step_sequence(shift):
        return [(x, w, s, gs, y, False) for (m, n, k, x, w, s, gs, y) in decode_step_calls(nv, lin, xs, ys, shift)]

    # One CUDA graph per rotation phase: the step's one sequence launch,
    # weights rotated so consecutive steps never touch the same copy; and the
    # same step as 15 single calls.
    stream = torch.cuda.Stream(device=dev)
    graphs, single_graphs = [], []
    with torch.cuda.stream(stream):
        for shift in range(ROTATE):
            nv.qmm_sequence(step_sequence(shift))  # warm the path outside capture
            for (m, n, k, x, w, s, gs, y) in decode_step_calls(nv, lin, xs, ys, shift):
                nv.qmm(x, w, s, gs=gs, out=y)
        torch.cuda.synchronize(dev)
        for shift in range(ROTATE):
            gph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gph, stream=stream):
                nv.qmm_sequence(step_sequence(shift))
            graphs.append(gph)
            gph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gph, stream=stream):
                for (m, n, k, x, w, s, gs, y) in decode_step_calls(nv, lin, xs, ys, shift):
                    nv.qmm(x, w, s, gs=gs, out=y)
            single_graphs.append(gph)
    torch.cuda.synchronize(dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            graphs[i % ROTATE].replay()
    barrier()

    def window(gs_list):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            for i in range(args.steps):
                gs_list[i % ROTATE].replay()
            b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b)

    with ClockSampler(local) as clk:
        ms_window = window(graphs)  # the timed region: exactly K steps
        barrier()
        # further windows of K steps, for the spread of the step rate
        extra = [window(graphs) for _ in range(args.windows - 1)]
    barrier()
    ms_total = reduce_step_time(torch, dist, dev, ms_window)
    ms_step = ms_total / args.steps
    value = job_value(step_bytes, world, ms_step)
    rates = sorted(step_bytes / (ms / args.steps * 1e-3) / 1e9 for ms in [ms_window] + extra)
    spread = {"windows": len(rates), "steps_per_window": args.steps, "GBps_min": round(rates[0], 1),
              "GBps_median": round(statistics.median(rates), 1), "GBps_max": round(rates[-1], 1)}
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            single_graphs[i % ROTATE].replay()
    torch.cuda.synchronize(dev)
    ms_single = window(single_graphs) / args.steps
    step_single = {"ms_per_step": round(ms_single, 5),
                   "GBps": round(step_bytes / (ms_single * 1e-3) / 1e9, 1),
                   "launches_per_step": len(DECODE_M) * len(LINEARS),
                   "path": "the same 15 calls as single nvfp4_qmm calls (one launch each, launch overlap as "
                           "configured), one CUDA graph per step"}

    # Per-call latency (µs/call) per shape: ten calls (rotating weight copies)
    # captured in one CUDA graph, replayed, device time / 10.
    per_call = {}
    with torch.cuda.stream(stream):
        for mi, m in enumerate(DECODE_M):
            for name, n, k, copies in lin:
                gph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gph, stream=stream):
                    for rep in range(2 * ROTATE):
                        w, s, gs = copies[rep % ROTATE]
                        nv.qmm(xs[(m, name)], w, s, gs=gs, out=ys[(m, name)])
                gph.replay()
                torch.cuda.synchronize(dev)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for _ in range(3):
                    gph.replay()
                b.record(stream)
                torch.cuda.synchronize(dev)
                us = a.elapsed_time(b) * 1e3 / (3 * 2 * ROTATE)
                per_call[f"{name}_M{m}"] = {"us": round(us, 2),
                                            "GBps": round(qmv_bytes(m, n, k) / (us * 1e-6) / 1e9, 1)}
                del gph

    # End to end through the public API: pinned host activations in, bf16
    # outputs back to pinned host memory, every step.
    e2e = run_e2e(nv, torch, dev, stream, lin, xs, ys, args, step_bytes)
    del single_graphs

    routes = {} if args.no_routes else run_routes(nv, synth, torch, dev, stream, args)
    kernel_sha = source_sha(TRAFFIC_FILES)
    traffic = TRAFFIC["bytes_per_step"] if TRAFFIC["kernel_sha"] == kernel_sha else None

    if rank == 0:
        cpu = run_cpu_baseline(args) if world == 1 and not args.no_cpu else None
        achieved = step_bytes / (ms_step * 1e-3) / 1e9
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": list(DECODE_M), "calls_per_step": len(DECODE_M) * len(LINEARS),
                       "launches_per_step": launches_per_step, "api": "nvfp4_qmm_sequence (15 calls, one launch)",
                       "bytes_per_step": step_bytes, "l2": "inputs larger than L2: 5 rotating weight copies "
                       "(1.1 GB per step)", "graph": "one CUDA graph per step",
                       "launch_overlap": args.launch_overlap == "on"},
            "spread": spread,
            "step_single_calls": step_single,
            "us_per_call": per_call,
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                         "frac": round(achieved / hbm_peak, 4), "peak_kind": f"{peak_kind} copy bandwidth",
                         "frac_of_8TBps": round(achieved / 8000.0, 4),
                         "kernel": "qmv_seq_kernel (one launch per step)",
                         "traffic": None if traffic is None else round(traffic / launches_per_step)},
            "gpu_launches": launches_per_step * args.steps,
            "e2e": e2e,
            "clocks": clk.summary(),
            "routes": routes,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


def run_e2e(nv, torch, dev, stream, lin, xs, ys, args, step_bytes):
    """The step through the public API, one nvfp4_qmm_sequence call per step
    (no graph), with the step's activations copied in from pinned host memory
    and its outputs copied back to pinned host memory every step. The 15 activation blocks live in one
    buffer and the 15 outputs in another (views), so a step moves its inputs
    and outputs with one host-to-device and one device-to-host copy. As in a
    serving loop, the copies run on their own streams, double-buffered: step
    i + 1's inputs go in and step i - 1's outputs come out while step i
    computes."""
    keys = list(xs.keys())
    xsz = [xs[k].numel() for k in keys]
    ysz = [ys[k].numel() for k in keys]
    host_x = torch.cat([xs[k].reshape(-1).cpu() for k in keys]).pin_memory()
    ydt = ys[keys[0]].dtype
    dev_xbuf = [torch.empty_like(host_x, device=dev) for _ in range(2)]
    dev_ybuf = [torch.empty(sum(ysz), dtype=ydt, device=dev) for _ in range(2)]
    host_y = [torch.empty(sum(ysz), dtype=ydt).pin_memory() for _ in range(2)]
    dev_x, dev_y = [{}, {}], [{}, {}]
    for b in range(2):
        ox = oy = 0
        for k, nx, ny in zip(keys, xsz, ysz):
            dev_x[b][k] = dev_xbuf[b][ox:ox + nx].view(xs[k].shape)
            dev_y[b][k] = dev_ybuf[b][oy:oy + ny].view(ys[k].shape)
            ox += nx
            oy += ny
    h2d = host_x.numel() * host_x.element_size()
    d2h = host_y[0].numel() * host_y[0].element_size()
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()
    x_in, y_done, y_out = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    started = [False, False]

    def step(i):
        b = i % 2
        with torch.cuda.stream(up):  # inputs of step i, once step i - 2 is done with the buffer
            if started[b]:
                up.wait_event(y_done[b])
            dev_xbuf[b].copy_(host_x, non_blocking=True)
            x_in[b].record(up)
        with torch.cuda.stream(stream):
            stream.wait_event(x_in[b])
            if started[b]:
                stream.wait_event(y_out[b])  # step i - 2's outputs have been copied out
            calls = []
            for mi, m in enumerate(DECODE_M):
                for name, n, k, copies in lin:
                    w, s, gs = copies[(mi + i) % ROTATE]
                    calls.append((dev_x[b][(m, name)], w, s, gs, dev_y[b][(m, name)], False))
            nv.qmm_sequence(calls)
            y_done[b].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(y_done[b])
            host_y[b].copy_(dev_ybuf[b], non_blocking=True)
            y_out[b].record(down)
        started[b] = True

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(up)
    for i in range(args.steps):
        step(args.warmup + i)
    z.record(down)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(z) / args.steps
    return {"value": round(step_bytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 4),
            "path": "one nvfp4_qmm_sequence call per step (no graph); per step one pinned-host copy in and one copy "
                    "out, on their own streams, double-buffered so the copies of neighbouring steps overlap this "
                    "step's launch"}


def time_calls(torch, dev, stream, fn, reps):
    """Device time per call (ms): `reps` calls captured in one CUDA graph (after
    a warm-up call outside capture) and replayed, so that host launch overhead
    does not count."""
    with torch.cuda.stream(stream):
        fn(0)
        torch.cuda.synchronize(dev)
        gph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gph, stream=stream):
            for i in range(reps):
                fn(i)
        gph.replay()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        gph.replay()
        b.record(stream)
    torch.cuda.synchronize(dev)
    del gph
    return a.elapsed_time(b) / reps


def run_routes(nv, synth, torch, dev, stream, args):
    hbm_peak, bf16_peak, _ = peaks()
    out = {}
    g = synth.rng(3000)

    def rand_w(n, k, copies=1, seed=0):
        ws = []
        for c in range(copies):
            w = torch.randint(-2**31, 2**31 - 1, (n, k // 8), dtype=torch.int32, device=dev,
                              generator=torch.Generator(device=dev).manual_seed(seed + c))
            s = torch.from_numpy(synth.log_uniform_scales(g, (n, k // 16), 2.0**-6, 4.0)).to(dev)
            ws.append((w, s))
        return ws

    # Prefill QuantizedMatmul (tensor-core route where the library picks it).
    pre = {}
    for (m, n, k) in ((512, 21504, 5376), (2048, 21504, 5376), (8192, 21504, 5376), (2048, 5376, 21504)):
        ws = rand_w(n, k, 2, seed=n + k)
        gs = torch.from_numpy(synth.global_scales(g, 1)).to(dev)
        x = synth.activations(g, (m, k), "bf16").to(dev)
        y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        reps = 3 if m >= 8192 else 5
        ms = time_calls(torch, dev, stream, lambda i: nv.qmm(x, ws[i % 2][0], ws[i % 2][1], gs=gs, out=y), reps)
        tf = 2.0 * m * n * k / (ms * 1e-3) / 1e12
        pre[f"M{m}_N{n}_K{k}"] = {"us": round(ms * 1e3, 1), "TFLOPs": round(tf, 1),
                                  "frac_bf16": round(tf / bf16_peak, 4),
                                  "route": "tc" if m >= nv.qmm_crossover(torch.bfloat16, n, k) else "qmv"}
        del ws, x, y
    out["qmm_prefill"] = pre

    # Route crossover: the decode-shape route against the tensor-core route
    # for M = 16 .. 8192 on each decode linear (two weight copies alternate,
    # so the weights come from HBM); M* is the first M where the tensor cores
    # win.
    cross = {}
    for name, n, k in LINEARS:
        ws = rand_w(n, k, 2, seed=7 * n + k)
        row = {"M": [], "qmv_us": [], "tc_us": []}
        first = None
        for m in (16, 24, 32, 48, 64, 96, 128, 192, 256, 512, 1024, 2048, 4096, 8192):
            x = synth.activations(g, (m, k), "bf16").to(dev)
            y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
            t = {}
            for route in ("qmv", "tc"):
                t[route] = time_calls(torch, dev, stream,
                                      lambda i: nv.qmm(x, ws[i % 2][0], ws[i % 2][1], route=route, out=y),
                                      6 if m <= 256 else 2)
            row["M"].append(m)
            row["qmv_us"].append(round(t["qmv"] * 1e3, 1))
            row["tc_us"].append(round(t["tc"] * 1e3, 1))
            if first is None and t["tc"] < t["qmv"]:
                first = m
            del x, y
        row["first_M_tc_faster"] = first
        row["library_crossover"] = nv.qmm_crossover(torch.bfloat16, n, k)
        cross[name] = row
        del ws
    out["route_crossover"] = cross

    # Transcode: one layer's three ModelOpt triplets -> native planes, timed
    # as whole layers (the three calls back to back, 440 MB per layer, more
    # than L2) so that no call finds its inputs in L2 from the previous
    # replay; gate/up alone (260 MB) is timed per call as well.
    trip = []
    for name, n, k in LINEARS:
        mo_w = torch.randint(0, 256, (n, k // 2), dtype=torch.uint8, device=dev)
        mo_s = torch.randint(0, 127, (n, k // 16), dtype=torch.uint8, device=dev)
        ws2 = torch.tensor([0.005], dtype=torch.float32, device=dev)
        outp = (torch.empty((n, k // 8), dtype=torch.int32, device=dev),
                torch.empty((n, k // 16), dtype=torch.uint8, device=dev),
                torch.empty((1,), dtype=torch.float32, device=dev))
        trip.append((name, n, k, mo_w, mo_s, ws2, outp))

    def layer(i):
        for (_, _, _, mo_w, mo_s, ws2, outp) in trip:
            nv.transcode(mo_w, mo_s, ws2, out=outp)

    ms_layer = time_calls(torch, dev, stream, layer, 5)
    layer_b = sum(2 * 0.5625 * n * k + 8 for (_, n, k, *_rest) in trip)
    _, n0, k0, w0, s0, g0, o0 = trip[0]
    ms_gu = time_calls(torch, dev, stream, lambda i: nv.transcode(w0, s0, g0, out=o0), 5)
    b_gu = 2 * 0.5625 * n0 * k0 + 8
    del trip
    # The whole 60-layer workload: every layer's three triplets resident on
    # the device (13.2 GB in, 13.2 GB out), the 180 transcodes in one pass.
    layers = []
    for layer in range(60):
        for j, (_, n, k) in enumerate(LINEARS):
            mo_w, mo_s, ws2 = synth.device_modelopt_triplet(9000 + 3 * layer + j, n, k, dev)
            outp = (torch.empty((n, k // 8), dtype=torch.int32, device=dev),
                    torch.empty((n, k // 16), dtype=torch.uint8, device=dev),
                    torch.empty((1,), dtype=torch.float32, device=dev))
            layers.append((mo_w, mo_s, torch.tensor([float(ws2)], dtype=torch.float32, device=dev), outp))

    def all_layers(i):
        for (mo_w, mo_s, ws2, outp) in layers:
            nv.transcode(mo_w, mo_s, ws2, out=outp)

    ms_60 = time_calls(torch, dev, stream, all_layers, 1)
    b_60 = 60 * layer_b
    out["transcode"] = {"layer_us": round(ms_layer * 1e3, 1), "layer_GBps": round(layer_b / (ms_layer * 1e-3) / 1e9, 1),
                        "layer_frac_hbm": round(layer_b / (ms_layer * 1e-3) / 1e9 / hbm_peak, 4),
                        "gate_up": {"us": round(ms_gu * 1e3, 1), "GBps": round(b_gu / (ms_gu * 1e-3) / 1e9, 1)},
                        "60_layers_ms": round(ms_60, 3), "60_layers_GBps": round(b_60 / (ms_60 * 1e-3) / 1e9, 1),
                        "60_layers_frac_hbm": round(b_60 / (ms_60 * 1e-3) / 1e9 / hbm_peak, 4),
                        "60_layers_bytes": b_60}
    del layers
    torch.cuda.empty_cache()

    # Fused gate/up with GeGLU on the gate/up plane [43008, 5376] (I = 21504):
    # decode at M = 1 and 16 (bytes as for the plain call, output I wide) and
    # prefill at M = 2048 (flops of the whole projection), beside the plain
    # projection of the same plane.
    n, k = 43008, 5376
    (w, s), = rand_w(n, k, 1, seed=7)
    gs = torch.from_numpy(synth.global_scales(g, 1)).to(dev)
    glu = {}
    for m in (1, 16, 2048):
        x = synth.activations(g, (m, k), "bf16").to(dev)
        yg = torch.empty((m, n // 2), dtype=torch.bfloat16, device=dev)
        yp = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        ms_g = time_calls(torch, dev, stream, lambda i: nv.qmm_glu(x, w, s, gs=gs, act="gelu_tanh", out=yg), 5)
        ms_p = time_calls(torch, dev, stream, lambda i: nv.qmm(x, w, s, gs=gs, out=yp), 5)
        entry = {"us": round(ms_g * 1e3, 1), "plain_qmm_us": round(ms_p * 1e3, 1)}
        if m >= 128:
            tf = 2.0 * m * n * k / (ms_g * 1e-3) / 1e12
            entry.update(TFLOPs=round(tf, 1), frac_bf16=round(tf / bf16_peak, 4))
        else:
            b = 0.5625 * n * k + 2 * m * k + 2 * m * (n // 2)
            entry.update(GBps=round(b / (ms_g * 1e-3) / 1e9, 1), frac_hbm=round(b / (ms_g * 1e-3) / 1e9 / hbm_peak, 4))
        glu[f"M{m}"] = entry
        del x, yg, yp
    out["gate_up_geglu_43008x5376"] = glu
    del w, s

    # Batched weights: 8 MoE-expert gate/up planes [1536, 2048], 4 token rows
    # each, as one expert-group launch and as one call per batch.
    bt, m, n, k = 8, 4, 1536, 2048
    wb = torch.randint(-2**31, 2**31 - 1, (bt, n, k // 8), dtype=torch.int32, device=dev)
    sb = torch.from_numpy(synth.log_uniform_scales(g, (bt, n, k // 16), 2.0**-6, 4.0)).to(dev)
    gsb = torch.from_numpy(synth.global_scales(g, bt)).to(dev)
    xb = synth.activations(g, (bt * m, k), "bf16").reshape(bt, m, k).to(dev)
    yb = torch.empty((bt, m, n), dtype=torch.bfloat16, device=dev)
    ms_one = time_calls(torch, dev, stream, lambda i: nv.qmm_batched(xb, wb, sb, gs=gsb, out=yb), 10)
    nv.set_option("gather_group", 0)  # one call per batch instead of one launch
    ms_loop = time_calls(torch, dev, stream, lambda i: nv.qmm_batched(xb, wb, sb, gs=gsb, out=yb), 10)
    nv.set_option("gather_group", 1)
    bb = bt * (0.5625 * n * k + 2 * m * k + 2 * m * n)
    out["qmm_batched_8x1536x2048_M4"] = {"us": round(ms_one * 1e3, 1), "GBps": round(bb / (ms_one * 1e-3) / 1e9, 1),
                                          "per_batch_calls_us": round(ms_loop * 1e3, 1)}
    del wb, sb, xb, yb

    # Non-transposed weights: the MLP up projection's sizes (K = 5376 inputs,
    # N = 21504 outputs) stored [K, N/8] and quantized along N, beside the
    # transposed plane of the same sizes through nv.qmm. Four copies of each
    # plane (260 MB, twice what L2 holds) take turns, so that no call finds
    # its weights left in L2 by an earlier one.
    k, n = 5376, 21504
    wts = [torch.randint(-2**31, 2**31 - 1, (k, n // 8), dtype=torch.int32, device=dev) for _ in range(4)]
    stts = [torch.from_numpy(synth.log_uniform_scales(g, (k, n // 16), 2.0**-6, 4.0)).to(dev) for _ in range(4)]
    wst = rand_w(n, k, 4, seed=9)
    ntr = {}
    for m in (1, 8, 16, 2048):
        x = synth.activations(g, (m, k), "bf16").to(dev)
        y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        reps = 24 if m < 128 else 4
        ms_nt = time_calls(torch, dev, stream, lambda i: nv.qmm_nontransposed(x, wts[i % 4], stts[i % 4], out=y), reps)
        ms_t = time_calls(torch, dev, stream, lambda i: nv.qmm(x, wst[i % 4][0], wst[i % 4][1], out=y), reps)
        entry = {"us": round(ms_nt * 1e3, 1), "transposed_qmm_us": round(ms_t * 1e3, 1)}
        if m >= 128:
            tf = 2.0 * m * n * k / (ms_nt * 1e-3) / 1e12
            entry.update(TFLOPs=round(tf, 1), frac_bf16=round(tf / bf16_peak, 4))
        else:
            b = 0.5625 * n * k + 2 * m * k + 2 * m * n
            entry.update(GBps=round(b / (ms_nt * 1e-3) / 1e9, 1), frac_hbm=round(b / (ms_nt * 1e-3) / 1e9 / hbm_peak, 4))
        ntr[f"M{m}"] = entry
        del x, y
    out["qmm_nontransposed_5376x21504"] = ntr
    del wts, stts, wst

    # Quantize a dense bf16 gate/up plane [43008, 5376] with gs = its amax.
    n, k = 43008, 5376
    xq = (torch.randn((n, k), device=dev, generator=torch.Generator(device=dev).manual_seed(11)) * 0.02).to(torch.bfloat16)
    gq = xq.abs().max().float().reshape(1)
    oq = (torch.empty((n, k // 8), dtype=torch.int32, device=dev), torch.empty((n, k // 16), dtype=torch.uint8, device=dev))
    ms = time_calls(torch, dev, stream, lambda i: nv.quantize(xq, gs=gq, out=oq), 5)
    b = 2 * n * k + 0.5625 * n * k
    out["quantize_bf16_43008x5376"] = {"us": round(ms * 1e3, 1), "GBps": round(b / (ms * 1e-3) / 1e9, 1),
                                       "frac_hbm": round(b / (ms * 1e-3) / 1e9 / hbm_peak, 4)}
    del xq, gq, oq

    # Folded-scale transcode (the variant the sidecar replaces): a ModelOpt-
    # convention triplet of the same plane (made by the quantizer, gs = amax,
    # ws2 = amax / 2688), folded, then both dequantized and compared: blocks
    # whose folded scale flushed to 0, and the error against the sidecar
    # values (the sidecar dequantization is exact).
    xq = (torch.randn((n, k), device=dev, generator=torch.Generator(device=dev).manual_seed(11)) * 0.02).to(torch.bfloat16)
    gq = xq.abs().max().float().reshape(1)
    wq, sq = nv.quantize(xq, gs=gq)
    del xq
    ws2 = gq / 2688.0
    mo_w = wq.view(torch.uint8).reshape(n, k // 2)
    of = (torch.empty_like(wq), torch.empty_like(sq))
    ms = time_calls(torch, dev, stream, lambda i: nv.transcode_folded(mo_w, sq, ws2, out=of), 5)
    b = 2 * (0.5625 * n * k)
    ref = nv.dequantize(wq, sq, gq, torch.float32)
    fold = nv.dequantize(of[0], of[1], None, torch.float32)
    nzr = ref != 0
    rel = ((fold - ref).abs()[nzr] / ref.abs()[nzr])
    flushed = int(((sq != 0) & (of[1] == 0)).sum())
    out["transcode_folded_43008x5376"] = {
        "us": round(ms * 1e3, 1), "GBps": round(b / (ms * 1e-3) / 1e9, 1),
        "blocks": int(sq.numel()), "blocks_flushed_to_zero": flushed,
        "blocks_saturated": int((of[1] == 0x7E).sum()),
        "max_abs_err_rel_to_max": round(float((fold - ref).abs().max() / ref.abs().max()), 6),
        "median_rel_err_nonzero": round(float(rel.median()), 6), "max_rel_err_nonzero": round(float(rel.max()), 6),
        "elements_zeroed": int(((fold == 0) & nzr).sum()), "elements_nonzero": int(nzr.sum())}
    del wq, sq, of, ref, fold, nzr, rel, mo_w

    # Dequantize the gate/up weight to bf16. The folded-scale entry above
    # held several GB; its blocks go back to the device first, so that the
    # output plane here is allocated afresh (left in the allocator's cache,
    # the reused blocks made this kernel about 15% slower).
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    n, k = 43008, 5376
    (w, s), = rand_w(n, k, 1, seed=5)
    d = torch.empty((n, k), dtype=torch.bfloat16, device=dev)
    ms = time_calls(torch, dev, stream, lambda i: nv.dequantize(w, s, None, torch.bfloat16, out=d), 5)
    b = 0.5625 * n * k + 2 * n * k
    out["dequantize_bf16_43008x5376"] = {"us": round(ms * 1e3, 1), "GBps": round(b / (ms * 1e-3) / 1e9, 1),
                                         "frac_hbm": round(b / (ms * 1e-3) / 1e9 / hbm_peak, 4)}
    del d, w, s

    # MoE GatherQMM: 128 experts, gate/up [1536, 2048], down [2048, 768]. The
    # routing comes from its own generator, so the drawn experts do not depend
    # on what the entries above drew.
    g = synth.rng(3100)
    E = 128
    moe = {}
    for name, n, k in (("gate_up", 1536, 2048), ("down", 2048, 768)):
        w = torch.randint(-2**31, 2**31 - 1, (E, n, k // 8), dtype=torch.int32, device=dev)
        s = torch.from_numpy(synth.log_uniform_scales(g, (E, n, k // 16), 2.0**-6, 4.0)).to(dev)
        gs = torch.from_numpy(synth.global_scales(g, E)).to(dev)
        # decode: 64 unsorted rows + experts E and E+1 (zero rows)
        rhs = np.concatenate([synth.zipf_experts(g, 64, E), np.array([E, E + 1], dtype=np.uint32)])
        rhs_d = torch.from_numpy(rhs.view(np.int32)).to(dev)
        x = synth.activations(g, (66, k), "bf16").to(dev)
        y = torch.empty((66, n), dtype=torch.bfloat16, device=dev)
        ms = time_calls(torch, dev, stream, lambda i: nv.gather_qmm(x, w, s, rhs_d, None, gs=gs, out=y), 10)
        uniq = len(set(int(v) for v in rhs if v < E))
        b = uniq * 0.5625 * n * k + 66 * 2 * (k + n)
        moe[f"decode_{name}"] = {"us": round(ms * 1e3, 1), "unique_experts": uniq,
                                 "GBps_unique": round(b / (ms * 1e-3) / 1e9, 1)}
        # prefill: 4096 tokens, top-8 Zipf(1.1) routing, rows sorted by expert;
        # the down projection takes the 32768 gate/up output rows in order.
        if name == "gate_up":
            lhs_p, rhs_p = synth.zipf_routing(g, 4096, E, 8)
            lhs, rhs = lhs_p, rhs_p
            xp = synth.activations(g, (4096, k), "bf16").to(dev)
        else:
            lhs, rhs = np.arange(rhs_p.size, dtype=np.uint32), rhs_p
            xp = synth.activations(g, (rhs_p.size, k), "bf16").to(dev)
        lhs_d = torch.from_numpy(lhs.view(np.int32)).to(dev)
        rhs_d = torch.from_numpy(rhs.view(np.int32)).to(dev)
        yp = torch.empty((rhs.size, n), dtype=torch.bfloat16, device=dev)
        ms = time_calls(torch, dev, stream,
                        lambda i: nv.gather_qmm(xp, w, s, rhs_d, lhs_d, gs=gs, sorted_indices=True, out=yp), 3)
        tf = 2.0 * rhs.size * n * k / (ms * 1e-3) / 1e12
        moe[f"prefill_{name}"] = {"rows": int(rhs.size), "us": round(ms * 1e3, 1), "TFLOPs": round(tf, 1),
                                  "frac_bf16": round(tf / bf16_peak, 4)}
        del w, s, x, y, xp, yp
    out["gather_moe"] = moe
    torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------------------- CPU oracle

def oracle_sample(rows_per_linear=192, seed=4000):
    """A bounded sample of the decode step for the CPU oracle: the first
    `rows_per_linear` output columns of every (M, linear) call."""
    from nvfp4_quantized_matmul_gb300 import synth

    g = synth.rng(seed)
    items = []
    for m in DECODE_M:
        for name, n, k in LINEARS:
            w = synth.packed_weight(g, rows_per_linear, k)
            s = synth.log_uniform_scales(g, (rows_per_linear, k // 16), 2.0**-6, 4.0)
            gs = synth.global_scales(g, 1)[0]
            x = synth.activations(g, (m, k), "bf16").double().numpy()
            items.append((m, rows_per_linear, k, x, w, s, gs))
    return items


def time_oracle(items):
    from oracle import nvfp4_oracle as O

    t0 = time.perf_counter()
    nbytes = 0.0
    for (m, n, k, x, w, s, gs) in items:
        O.qmm(x, w, s, gs)
        nbytes += qmv_bytes(m, n, k)
    return nbytes, time.perf_counter() - t0


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def run_cpu_baseline(args):
    items = oracle_sample(args.cpu_rows)
    nbytes, secs = time_oracle(items)
    return {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s", "cores": cores(), "kind": "oracle",
            "seconds": round(secs, 2),
            "sample": f"first {args.cpu_rows} weight rows of each of the 15 decode calls "
                      f"({nbytes / 1e6:.1f} MB algorithmic), numpy float64 oracle"}


def run_case(args):
    """Small profiling cases.

    qmv_small: gate/up [43008, 5376] (two copies, 260 MB, larger than L2),
    three warm-up calls then one call each at M = 1, 8 and 16.
    qmv_shapes: each decode linear (gate/up, down, qkv; 220 MB) once at M = 1
    and once at M = 16, after one warm-up call each.
    decode_step: the 15 calls of one decode step (one weight copy per linear)
    as one nvfp4_qmm_sequence launch, once as warm-up and once more.
    decode_step_single: the same 15 calls as single nvfp4_qmm calls.
    gather_prefill: the sorted MoE gate/up GatherQMM (4096 tokens, top-8 of
    128 experts), one warm-up call then one call.
    prefill: the tensor-core route at M = 2048 on the [21504, 5376] plane, one
    warm-up call then one call.
    nontransposed_prefill: nvfp4_qmm_nontransposed at M = 2048 on a [5376,
    21504 / 8] plane (whole tiles), one warm-up call then one call.
    nontransposed_decode: the same plane at M = 1 (the streaming kernel), one
    warm-up call then one call.
    quantize: nvfp4_quantize of a dense bf16 [43008, 5376] plane with gs =
    max |x|, one warm-up call then one call.
    """
    import torch

    import nvfp4_quantized_matmul_gb300 as nv
    from nvfp4_quantized_matmul_gb300 import synth

    dev = torch.device("cuda", 0)
    if args.case == "prefill":
        g = synth.rng(5200)
        n, k, m = 21504, 5376, 2048
        w = torch.randint(-2**31, 2**31 - 1, (n, k // 8), dtype=torch.int32, device=dev,
                          generator=torch.Generator(device=dev).manual_seed(7))
        s = torch.from_numpy(synth.log_uniform_scales(g, (n, k // 16), 2.0**-6, 4.0)).to(dev)
        gs = torch.from_numpy(synth.global_scales(g, 1)).to(dev)
        x = synth.activations(g, (m, k), "bf16").to(dev)
        for _ in range(2):
            nv.qmm(x, w, s, gs=gs, route="tc")
        torch.cuda.synchronize(dev)
        print("case prefill ok")
        return
    if args.case == "nontransposed_prefill":
        g = synth.rng(5400)
        k, n, m = 5376, 21504, 2048
        w = torch.randint(-2**31, 2**31 - 1, (k, n // 8), dtype=torch.int32, device=dev,
                          generator=torch.Generator(device=dev).manual_seed(9))
        s = torch.from_numpy(synth.log_uniform_scales(g, (k, n // 16), 2.0**-6, 4.0)).to(dev)
        x = synth.activations(g, (m, k), "bf16").to(dev)
        for _ in range(2):
            nv.qmm_nontransposed(x, w, s)
        torch.cuda.synchronize(dev)
        print("case nontransposed_prefill ok")
        return
    if args.case == "nontransposed_decode":
        g = synth.rng(5500)
        k, n = 5376, 21504
        w = torch.randint(-2**31, 2**31 - 1, (k, n // 8), dtype=torch.int32, device=dev,
                          generator=torch.Generator(device=dev).manual_seed(9))
        s = torch.from_numpy(synth.log_uniform_scales(g, (k, n // 16), 2.0**-6, 4.0)).to(dev)
        x = synth.activations(g, (1, k), "bf16").to(dev)
        for _ in range(2):
            nv.qmm_nontransposed(x, w, s)
        torch.cuda.synchronize(dev)
        print("case nontransposed_decode ok")
        return
    if args.case == "quantize":
        n, k = 43008, 5376
        x = (torch.randn((n, k), device=dev, generator=torch.Generator(device=dev).manual_seed(11)) * 0.02).to(
            torch.bfloat16)
        gs = x.abs().max().float().reshape(1)
        for _ in range(2):
            nv.quantize(x, gs=gs)
        torch.cuda.synchronize(dev)
        print("case quantize ok")
        return
    if args.case == "gather_prefill":
        g = synth.rng(5300)
        E, n, k, T = 128, 1536, 2048, 4096
        w = torch.randint(-2**31, 2**31 - 1, (E, n, k // 8), dtype=torch.int32, device=dev,
                          generator=torch.Generator(device=dev).manual_seed(11))
        s = torch.from_numpy(synth.log_uniform_scales(g, (E, n, k // 16), 2.0**-6, 4.0)).to(dev)
        gs = torch.from_numpy(synth.global_scales(g, E)).to(dev)
        lhs, rhs = synth.zipf_routing(g, T, E, 8)
        x = synth.activations(g, (T, k), "bf16").to(dev)
        lhs_d = torch.from_numpy(lhs.view(np.int32)).to(dev)
        rhs_d = torch.from_numpy(rhs.view(np.int32)).to(dev)
        for _ in range(2):
            nv.gather_qmm(x, w, s, rhs_d, lhs_d, gs=gs, sorted_indices=True)
        torch.cuda.synchronize(dev)
        print("case gather_prefill ok")
        return
    if args.case == "decode_step":
        lin, xs, ys = build_decode(nv, synth, torch, dev, 0, copies=1)
        calls = [(x, w, s, gs, y, False) for (m, n, k, x, w, s, gs, y) in decode_step_calls(nv, lin, xs, ys, 0)]
        for _ in range(2):
            nv.qmm_sequence(calls)
        torch.cuda.synchronize(dev)
        print("case decode_step ok")
        return
    if args.case == "decode_step_single":
        lin, xs, ys = build_decode(nv, synth, torch, dev, 0, copies=1)
        for _ in range(2):
            for (m, n, k, x, w, s, gs, y) in decode_step_calls(nv, lin, xs, ys, 0):
                nv.qmm(x, w, s, gs=gs, out=y)
        torch.cuda.synchronize(dev)
        print("case decode_step_single ok")
        return
    if args.case == "qmv_shapes":
        g = synth.rng(5100)
        lin = []
        for name, n, k in LINEARS:
            w = torch.randint(-2**31, 2**31 - 1, (n, k // 8), dtype=torch.int32, device=dev,
                              generator=torch.Generator(device=dev).manual_seed(n))
            s = torch.from_numpy(synth.log_uniform_scales(g, (n, k // 16), 2.0**-6, 4.0)).to(dev)
            gs = torch.from_numpy(synth.global_scales(g, 1)).to(dev)
            lin.append((w, s, gs, k))
        for w, s, gs, k in lin:
            nv.qmm(synth.activations(g, (1, k), "bf16").to(dev), w, s, gs=gs)
        for m in (1, 16):
            for w, s, gs, k in lin:
                nv.qmm(synth.activations(g, (m, k), "bf16").to(dev), w, s, gs=gs)
        torch.cuda.synchronize(dev)
        print("case qmv_shapes ok")
        return
    g = synth.rng(5000)
    n, k = 43008, 5376
    ws = []
    for c in range(2):
        w = torch.randint(-2**31, 2**31 - 1, (n, k // 8), dtype=torch.int32, device=dev,
                          generator=torch.Generator(device=dev).manual_seed(c))
        s = torch.from_numpy(synth.log_uniform_scales(g, (n, k // 16), 2.0**-6, 4.0)).to(dev)
        ws.append((w, s))
    gs = torch.from_numpy(synth.global_scales(g, 1)).to(dev)
    for i, m in enumerate((1, 1, 1, 1, 8, 16)):
        x = synth.activations(g, (m, k), "bf16").to(dev)
        nv.qmm(x, ws[i % 2][0], ws[i % 2][1], gs=gs)
    torch.cuda.synchronize(dev)
    print("case qmv_small ok")


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    items = oracle_sample(args.ref_rows)
    for _ in range(args.warmup):
        time_oracle(items[:3])
    tot_b, tot_s = 0.0, 0.0
    for _ in range(args.steps):
        b, s = time_oracle(items)
        tot_b += b
        tot_s += s
    value = tot_b / tot_s / 1e9
    ms_step = tot_s / args.steps * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 2), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": list(DECODE_M), "sample_rows_per_linear": args.ref_rows},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores(), "kind": "oracle",
                         "sample": f"first {args.ref_rows} weight rows of each of the 15 decode calls per step"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-routes", action="store_true")
    ap.add_argument("--launch-overlap", choices=["on", "off"], default="on",
                    help="let each decode call start while the previous one finishes (weights are constant)")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--windows", type=int, default=5,
                    help="timed windows of --steps steps; the first is the reported value, all give the spread")
    ap.add_argument("--cpu-rows", type=int, default=6144)
    ap.add_argument("--ref-rows", type=int, default=32)
    ap.add_argument("--case", choices=["qmv_small", "qmv_shapes", "decode_step", "decode_step_single", "prefill",
                                       "gather_prefill",
                                       "nontransposed_prefill", "nontransposed_decode", "quantize"],
                    default=None,
                    help="run one small profiling case instead of the benchmark")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.case:
        run_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
