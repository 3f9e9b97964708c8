"""Benchmark of the fused INT4/INT8-weight linear layer on GB300.

Default run (N=1): the decode step of a Llama-7B-like layer — the four W4A16
g128 projections (12288x4096 fused QKV, 4096x4096 O, 22016x4096 fused
gate/up, 4096x11008 down) at M=1 through tf_gemv — reported as HBM GB/s of
algorithmic bytes; in the same run the prefill GEMMs (11008x4096, 4096x11008,
12288x4096 at M=2048 with 1% outlier activation columns) through tf_gemm,
reported as TFLOP/s.  Inputs are seeded synthetic weights quantised with the
AWQ-style min/max recipe and BF16 activations.

Timing: W untimed warm-up steps, then K steps replayed from CUDA graphs on
one stream, bracketed by CUDA events with a device synchronisation on both
sides; the GEMV step rotates through weight copies totalling more than 3x
the L2 size so that every launch streams its weights from HBM.  Next to the
headline the same run reports the square 8192 x 8192 layers (W8 per channel
and W4 g64 at M = 1, 8, 64), the large W4 g128 layers at M = 1 and 4096, and
layers with fewer 16-row slabs than SMs, each as us per launch, GB/s,
TFLOP/s and the fraction of the measured peak that bounds it (HBM copy
bandwidth, or BF16 tensor throughput at M = 4096), and the float64 oracle on
all host cores (a process pool over output rows).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "W4A16 GEMV HBM GB/s (% of ~8 TB/s); prefill GEMM TFLOP/s (% BF16 peak)"
DECODE = [(12288, 4096, 1), (4096, 4096, 2), (22016, 4096, 3), (4096, 11008, 4)]  # (N, K, seed)
PREFILL = [(11008, 4096, 7), (4096, 11008, 8), (12288, 4096, 9)]
PREFILL_M = 2048
BITS, GROUP = 4, 128
# (name, N, K, bits, group, seed, M list): square layers and the large-dimension layers
SQUARE = [("w8_per_channel", 8192, 8192, 8, 0, 5, (1, 8, 64)), ("w4_g64", 8192, 8192, 4, 64, 6, (1, 8, 64))]
LARGE = [("32768x8192", 32768, 8192, 4, 128, 10, (1, 4096)), ("8192x32768", 8192, 32768, 4, 128, 11, (1, 4096)),
         ("32768x32768", 32768, 32768, 4, 128, 12, (1, 4096))]
# layers with fewer 16-row slabs than SMs (GQA-style K/V projections and the like)
SMALL = [("1024x11008_w4g128", 1024, 11008, 4, 128, 13, (1, 4)), ("2048x4096_w8", 2048, 4096, 8, 0, 14, (1, 8)),
         ("1024x11008_w4g32", 1024, 11008, 4, 32, 15, (1,))]
L2_BYTES = 129 * 1024 * 1024


def algo_bytes(M, N, K, bits=BITS, group=GROUP):
    """Weights + one BF16 scale and one b-bit zero per group + x + y."""
    g = K if group == 0 else group
    return N * K * bits / 8 + (N * K / g) * (2 + bits / 8) + 2 * M * K + 2 * M * N


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p.get("bf16_tflops_sustained", p["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, 1700.0, "fallback"


def source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


GEMV_SOURCES = ["gemv_tf_prepack_gb300/csrc/gemv_stream.cu", "gemv_tf_prepack_gb300/csrc/tf_device.cuh",
                "gemv_tf_prepack_gb300/csrc/tf_sm100.cuh", "gemv_tf_prepack_gb300/csrc/tf_format.h",
                "gemv_tf_prepack_gb300/csrc/tf_abi.h"]
GEMM_SOURCES = ["gemv_tf_prepack_gb300/csrc/gemm.cu", "gemv_tf_prepack_gb300/csrc/tf_device.cuh",
                "gemv_tf_prepack_gb300/csrc/tf_sm100.cuh", "gemv_tf_prepack_gb300/csrc/tf_format.h",
                "gemv_tf_prepack_gb300/csrc/tf_abi.h"]


def recorded_traffic(kernel: str, sources):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    want = source_hash(sources)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == kernel:
                return float(parts[1]) if parts[2] == want else None
    return None


class ClockSampler:
    """nvidia-smi clocks/throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.tmp, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.tmp.flush()

    def summary(self):
        self.tmp.seek(0)
        rows = [r.split(", ") for r in self.tmp.read().strip().splitlines() if r.strip()]
        os.unlink(self.tmp.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if len(r) > 5 + i and r[5 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# our arm


def build_layers(torch, tf, synth, shapes, M, outliers, copies):
    layers = []
    for (N, K, seed) in shapes:
        qw = synth.make_weights(N, K, BITS, GROUP, seed)
        blob = tf.prepack(qw.qweight, qw.scales, qw.zeros, N, K, BITS, GROUP)
        Ws = [tf.Weights.upload(blob) for _ in range(copies)]
        xb = synth.make_activations(M, K, seed, outliers=outliers)
        xh = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16)
        layers.append(dict(N=N, K=K, Ws=Ws, x_host=xh,
                           xs=[xh.cuda() for _ in range(copies)],
                           ys=[torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(copies)]))
    return layers


def timing_event(torch):
    """An event that becomes a real record node when captured in a CUDA graph."""
    try:
        return torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:  # older torch: no external events
        return None


def capture_step(torch, fn, layers, r, stream, events):
    """CUDA graph of one step on copy r, with an event between consecutive launches."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        if events[0] is not None:
            events[0].record(stream)
        for i, L in enumerate(layers):
            fn(L["Ws"][r], L["xs"][r], L["ys"][r])
            if events[i + 1] is not None:
                events[i + 1].record(stream)
    return g


def capture_steps(torch, fn, layers, copies, stream):
    """One CUDA graph holding one step on every copy, back to back, no events."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for r in range(copies):
            for L in layers:
                fn(L["Ws"][r], L["xs"][r], L["ys"][r])
    return g


def replay_steps(big, singles, copies, n, stream):
    """Replay exactly n steps: whole rotations from the big graph, then single steps."""
    for _ in range(n // copies):
        big.replay()
    for s in range(n % copies):
        singles[s].replay()


def launch_times(torch, ev, ncopies, layers, fn, stream):
    """Per-launch durations (ms) from the events captured in the step graphs.

    Without external graph events (older torch) the launches are timed with
    eager events on the same stream instead.
    """
    if ev[0][0] is not None:
        return [ev[r][i].elapsed_time(ev[r][i + 1]) for r in range(ncopies) for i in range(len(layers))]
    out = []
    for r in range(ncopies):
        es = [torch.cuda.Event(enable_timing=True) for _ in range(len(layers) + 1)]
        with torch.cuda.stream(stream):
            es[0].record(stream)
            for i, L in enumerate(layers):
                fn(L["Ws"][r], L["xs"][r], L["ys"][r])
                es[i + 1].record(stream)
        torch.cuda.synchronize()
        out += [es[i].elapsed_time(es[i + 1]) for i in range(len(layers))]
    return out


def rank_barrier(world: int):
    """Barrier over all ranks (a no-op on one)."""
    if world > 1:
        import torch
        torch.distributed.barrier()


def rank_max(v: float, world: int, device: str = "cuda") -> float:
    """The maximum of v over all ranks (timings: the slowest rank sets the job's time)."""
    if world == 1:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput of N independent replicas (weak scaling): every
    rank's units over the slowest rank's time, per second."""
    return world * units_per_rank / (ms * 1e-3)


def time_launches(torch, fn, Ws, x, y, stream):
    """us per launch of fn over the weight copies Ws, back to back in one CUDA
    graph (the copies together exceed the L2 size), timed with CUDA events
    after warm-up replays."""
    with torch.cuda.stream(stream):
        for W in Ws:
            fn(W, x, y)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for W in Ws:
            fn(W, x, y)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    reps = max(5, min(500, int(0.2e3 / max(e0.elapsed_time(e1), 1e-3))))  # about 0.2 s
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (reps * len(Ws))


def extra_layers(torch, tf, synth, stream, hbm_peak, tc_peak, peak_src):
    """The square 8192^2 layers (W8 per channel, W4 g64) at M = 1, 8, 64, the
    large W4 g128 layers at M = 1 and 4096, and layers with fewer 16-row slabs
    than SMs: us per launch, GB/s of algorithmic bytes, TFLOP/s, and the
    fraction of the measured peak that bounds the launch (HBM copy bandwidth
    up to M = 64, where flop/byte <= 224; the burst BF16 tensor peak at
    M = 4096)."""
    out = {}
    for group_name, cases in (("square_8192", SQUARE), ("large", LARGE), ("small_n", SMALL)):
        res = {}
        for name, N, K, bits, group, seed, Ms in cases:
            qw = synth.make_weights(N, K, bits, group, seed)
            blob = tf.prepack(qw.qweight, qw.scales, qw.zeros, N, K, bits, group)
            copies = max(2, int(np.ceil(3 * L2_BYTES / blob.size)) + 1)
            Ws = [tf.Weights.upload(blob) for _ in range(copies)]
            for M in Ms:
                xb = synth.make_activations(M, K, seed)
                x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
                y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
                call = tf.gemv if M <= 8 else tf.gemm

                def fn(W, x, y, call=call):
                    call(W, x, y, stream=stream)

                us = time_launches(torch, fn, Ws, x, y, stream)
                gbs = algo_bytes(M, N, K, bits, group) / (us * 1e-6) / 1e9
                tfs = 2.0 * M * N * K / us / 1e6
                tensor = M > 64
                res[f"{name}_M{M}"] = {"call": call.__name__, "us": round(us, 2), "GB/s": round(gbs, 1),
                                       "TFLOP/s": round(tfs, 2), "bound": "tensor" if tensor else "hbm",
                                       "frac": round(tfs / tc_peak if tensor else gbs / hbm_peak, 4)}
                del x, y
            del Ws
            torch.cuda.empty_cache()
        out[group_name] = res
    out["peak"] = {"hbm_gbs": hbm_peak, "bf16_tflops": tc_peak, "source": peak_src}
    out["l2"] = "each layer rotates through weight copies totalling more than 3x L2; one CUDA graph per layer"
    return out


def run_ours(args, rank, world):
    import torch

    import gemv_tf_prepack_gb300 as tf
    from gemv_tf_prepack_gb300 import synth

    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    hbm_peak, tc_peak, tc_peak_sus, peak_src = peaks()
    stream = torch.cuda.Stream()

    def barrier():
        rank_barrier(world)

    def max_over_ranks(v):
        return rank_max(v, world)

    # ---------------- decode GEMV step (headline value) ----------------
    step_bytes = sum(algo_bytes(1, N, K) for N, K, _ in DECODE)
    blob_bytes = sum(tf.prepack_size(N, K, BITS, GROUP) for N, K, _ in DECODE)
    copies = max(4, int(np.ceil(3 * L2_BYTES / blob_bytes)) + 1)
    dec = build_layers(torch, tf, synth, DECODE, 1, False, copies)
    for L in dec:
        for W in L["Ws"]:
            W.workspace(1)  # allocate (zero-filled) outside the graphs

    def gemv_call(W, x, y):
        tf.gemv(W, x, y, stream=stream)

    ev = [[timing_event(torch) for _ in range(len(DECODE) + 1)] for _ in range(copies)]
    with torch.cuda.stream(stream):
        for r in range(copies):  # warm the lazy paths before capture
            for L in dec:
                gemv_call(L["Ws"][r], L["xs"][r], L["ys"][r])
    torch.cuda.synchronize()
    singles = [capture_step(torch, gemv_call, dec, r, stream, [None] * (len(DECODE) + 1)) for r in range(copies)]
    big = capture_steps(torch, gemv_call, dec, copies, stream)
    with torch.cuda.stream(stream):  # replay() launches on the current stream
        replay_steps(big, singles, copies, args.warmup, stream)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev) as clk, torch.cuda.stream(stream):
        t0.record(stream)
        replay_steps(big, singles, copies, args.steps, stream)
        t1.record(stream)
        torch.cuda.synchronize()
    barrier()
    ms_step = max_over_ranks(t0.elapsed_time(t1) / args.steps)
    clocks = clk.summary()
    # Launches overlap (programmatic dependent launch), so the launch time of
    # the dominant kernel is the timed region divided by its launches.
    kernel_ms = ms_step / len(DECODE)
    per_launch_bytes = step_bytes / len(DECODE)
    achieved = per_launch_bytes / (kernel_ms * 1e-3) / 1e9
    value = job_rate(step_bytes, world, ms_step) / 1e9
    # For reference: each launch alone, bracketed by events captured in a graph
    # (no overlap with its neighbours), after the timed region.
    iso_graphs = [capture_step(torch, gemv_call, dec, r, stream, ev[r]) for r in range(copies)]
    with torch.cuda.stream(stream):
        for g in iso_graphs:
            g.replay()
    torch.cuda.synchronize()
    k_ms = launch_times(torch, ev, copies, dec, gemv_call, stream)
    iso_us = {f"{N}x{K}": round(1e3 * sum(k_ms[r * len(DECODE) + i] for r in range(copies)) / copies, 2)
              for i, (N, K, _) in enumerate(DECODE)}

    # ---------------- end to end through the public API (host buffers) ----------------
    # Each step's inputs (the four layers' x) come from pinned host memory in
    # one copy and its results (the four y) go back in one copy; the layers'
    # x and y are views into those buffers (every offset is a multiple of 8
    # elements, so every view stays 16-byte aligned).
    offx = np.cumsum([0] + [L["K"] for L in dec]).tolist()
    offy = np.cumsum([0] + [L["N"] for L in dec]).tolist()
    assert all(o % 8 == 0 for o in offx + offy)
    x_pin = torch.cat([L["x_host"].reshape(-1) for L in dec]).pin_memory()
    y_pin = torch.empty(offy[-1], dtype=torch.bfloat16).pin_memory()
    x_dev = [torch.empty(offx[-1], dtype=torch.bfloat16, device="cuda") for _ in range(copies)]
    y_dev = [torch.empty(offy[-1], dtype=torch.bfloat16, device="cuda") for _ in range(copies)]
    xv = [[x_dev[r][offx[i]:offx[i + 1]].view(1, -1) for i in range(len(dec))] for r in range(copies)]
    yv = [[y_dev[r][offy[i]:offy[i + 1]].view(1, -1) for i in range(len(dec))] for r in range(copies)]
    h2d = x_pin.numel() * 2
    d2h = y_pin.numel() * 2
    e2e_steps = max(3, min(args.steps, 200))

    def e2e_step(r):
        x_dev[r].copy_(x_pin, non_blocking=True)
        for i, L in enumerate(dec):
            tf.gemv(L["Ws"][r], xv[r][i], yv[r][i], stream=stream)
        y_pin.copy_(y_dev[r], non_blocking=True)

    # (a) eager: every step issues its copies and launches from Python
    with torch.cuda.stream(stream):
        for s in range(args.warmup + e2e_steps):
            if s == args.warmup:
                torch.cuda.synchronize()
                barrier()
                te = time.perf_counter()
            e2e_step(s % copies)
            stream.synchronize()
    eager_ms = max_over_ranks((time.perf_counter() - te) * 1e3 / e2e_steps)
    # (b) the way a serving loop runs a decode step: the step (host-to-device
    # copy, the four tf_gemv calls, device-to-host copy) captured once into a
    # CUDA graph per weight copy, replayed and waited for every step
    step_graphs = []
    with torch.cuda.stream(stream):
        for r in range(copies):
            e2e_step(r)
    torch.cuda.synchronize()
    for r in range(copies):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            e2e_step(r)
        step_graphs.append(gr)
    with torch.cuda.stream(stream):
        for s in range(args.warmup + e2e_steps):
            if s == args.warmup:
                torch.cuda.synchronize()
                barrier()
                te = time.perf_counter()
            step_graphs[s % copies].replay()
            while not stream.query():  # the step's result is on the host (poll rather than sleep)
                pass
    e2e_ms = max_over_ranks((time.perf_counter() - te) * 1e3 / e2e_steps)
    e2e_value = job_rate(step_bytes, world, e2e_ms) / 1e9
    eager_value = job_rate(step_bytes, world, eager_ms) / 1e9

    # ---------------- prefill GEMM (M=2048) ----------------
    for L in dec:
        L["Ws"].clear(); L["xs"].clear(); L["ys"].clear()
    del singles, big, iso_graphs
    torch.cuda.empty_cache()
    pcopies = 2
    pre = build_layers(torch, tf, synth, PREFILL, PREFILL_M, True, pcopies)

    def gemm_call(W, x, y):
        tf.gemm(W, x, y, stream=stream)

    pev = [[timing_event(torch) for _ in range(len(PREFILL) + 1)] for _ in range(pcopies)]
    with torch.cuda.stream(stream):
        for r in range(pcopies):
            for L in pre:
                gemm_call(L["Ws"][r], L["xs"][r], L["ys"][r])
    torch.cuda.synchronize()
    psingles = [capture_step(torch, gemm_call, pre, r, stream, [None] * (len(PREFILL) + 1)) for r in range(pcopies)]
    pbig = capture_steps(torch, gemm_call, pre, pcopies, stream)
    psteps = args.steps  # the same step count as the decode step
    with torch.cuda.stream(stream):
        replay_steps(pbig, psingles, pcopies, args.warmup, stream)
    torch.cuda.synchronize()
    barrier()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev) as pclk, torch.cuda.stream(stream):
        p0.record(stream)
        replay_steps(pbig, psingles, pcopies, psteps, stream)
        p1.record(stream)
        torch.cuda.synchronize()
    barrier()
    pms = max_over_ranks(p0.elapsed_time(p1) / psteps)
    flops = sum(2.0 * PREFILL_M * N * K for N, K, _ in PREFILL)
    p_kernel_ms = pms / len(PREFILL)
    piso = [capture_step(torch, gemm_call, pre, r, stream, pev[r]) for r in range(pcopies)]
    with torch.cuda.stream(stream):
        for g in piso:
            g.replay()
    torch.cuda.synchronize()
    pk = launch_times(torch, pev, pcopies, pre, gemm_call, stream)
    p_iso_us = {f"{N}x{K}": round(1e3 * sum(pk[r * len(PREFILL) + i] for r in range(pcopies)) / pcopies, 1)
                for i, (N, K, _) in enumerate(PREFILL)}
    p_achieved = flops / len(PREFILL) / (p_kernel_ms * 1e-3) / 1e12
    prefill_tflops = job_rate(flops, world, pms) / 1e12
    long_region = pms * psteps > 1000.0
    tc_ref = tc_peak_sus if long_region else tc_peak
    pclocks = pclk.summary()

    for L in pre:
        L["Ws"].clear(); L["xs"].clear(); L["ys"].clear()
    del psingles, pbig, piso
    torch.cuda.empty_cache()
    extras = None if args.no_extras else extra_layers(torch, tf, synth, stream, hbm_peak, tc_peak, peak_src)

    err = tf.device_error()
    if rank != 0:
        return None
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.02) weights, AWQ-style min/max W4 g128 quantisation; BF16 N(0,1) activations)",
        "config": {
            "workload": "decode step: 4 Llama-7B-like W4A16 g128 projections (12288x4096, 4096x4096, "
                        "22016x4096, 4096x11008) at M=1 through tf_gemv",
            "l2": f"rotates {copies} weight copies ({copies * blob_bytes / 1e6:.0f} MB > 3x L2) via CUDA graphs",
            "parallelism": f"replicas x{world}",
            "hbm_pct_of_8tbs": round(100 * value / world / 8000.0, 1),
        },
        "roofline": {
            "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(achieved / hbm_peak, 4), "peak_source": peak_src,
            "traffic": recorded_traffic("gemv_stream_kernel", GEMV_SOURCES),
            "kernel": "gemv_stream_kernel<4, 1, 1>", "algorithmic_bytes_per_launch": round(per_launch_bytes),
            "kernel_us_per_launch": round(kernel_ms * 1e3, 3),
            "isolated_launch_us": iso_us,
        },
        "prefill": {
            "workload": "W4A16 g128 GEMM at M=2048 (11008x4096, 4096x11008, 12288x4096), 1% outlier columns",
            "value": round(prefill_tflops, 1), "unit": "TFLOP/s", "ms_per_step": round(pms, 4),
            "roofline": {"bound": "tensor", "achieved": round(p_achieved, 1), "peak": tc_ref, "unit": "TFLOP/s",
                         "frac": round(p_achieved / tc_ref, 4), "peak_source": peak_src + (
                             " sustained" if long_region else " burst"),
                         "traffic": recorded_traffic("gemm_kernel", GEMM_SOURCES),
                         "kernel": "gemm_kernel<4,1>", "isolated_launch_us": p_iso_us},
            "clocks": pclocks,
            "gpu_launches": psteps * len(PREFILL),
        },
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                "path": "pinned host x of the four layers -> device (one copy), tf_gemv x4 through the "
                        "Python binding, the four y -> pinned host (one copy); the step captured once into a "
                        "CUDA graph and replayed every step, the host polling the stream until it is done",
                "eager": {"value": round(eager_value, 1), "ms_per_step": round(eager_ms, 4),
                          "path": "the same step issued from Python every step"}},
        "gpu_launches": args.steps * len(DECODE),
        "clocks": clocks,
        "device_error": err,
    }
    if extras is not None:
        line["layers"] = extras
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    return line


# ---------------------------------------------------------------------------
# CPU oracle (the reference arm and the cpu_baseline leg)

CPU_SAMPLE_ROWS = 2048  # output rows of each decode projection in the CPU baseline's sample


def _host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def _oracle_worker(job):
    """One worker's share: the oracle on a block of output rows (float64)."""
    from oracle import tf_oracle

    qw, sc, z, x, K = job
    t = time.perf_counter()
    tf_oracle.reference(qw, sc, z, BITS, GROUP, K, x)
    return time.perf_counter() - t


def _oracle_sample(rows):
    """The first `rows` output rows of each decode projection (the same
    generator stream as the full layers) and its activations."""
    from gemv_tf_prepack_gb300 import synth

    data = []
    for N, K, seed in DECODE:
        rng = np.random.default_rng(seed)
        w = rng.standard_normal((rows, K), dtype=np.float32) * np.float32(0.02)
        data.append((synth.quantise(w, BITS, GROUP), synth.make_activations(1, K, seed)))
    return data


def _oracle_jobs(data, r0, r1, cores):
    jobs = []
    for qw, x in data:
        for c in range(cores):
            a, b = r0 + (r1 - r0) * c // cores, r0 + (r1 - r0) * (c + 1) // cores
            if b > a:
                jobs.append((qw.qweight[a:b], qw.scales[a:b], qw.zeros[a:b], x, qw.K))
    return jobs


class OraclePool:
    """The float64 oracle on every host core: a spawn-started process pool
    (one single-threaded BLAS per worker) over blocks of output rows."""

    def __init__(self):
        import multiprocessing as mp

        self.cores = _host_cores()
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[k] = "1"  # inherited by the workers
        self.pool = mp.get_context("spawn").Pool(self.cores)

    def run(self, data, r0, r1):
        """Wall-clock seconds and algorithmic bytes of rows [r0, r1) of every projection."""
        jobs = _oracle_jobs(data, r0, r1, self.cores)
        t = time.perf_counter()
        self.pool.map(_oracle_worker, jobs, chunksize=1)
        dt = time.perf_counter() - t
        return dt, sum(algo_bytes(1, r1 - r0, qw.K) for qw, _ in data)

    def close(self):
        self.pool.close()
        self.pool.join()


def cpu_baseline() -> dict:
    data = _oracle_sample(CPU_SAMPLE_ROWS)
    op = OraclePool()
    try:
        op.run(data, 0, CPU_SAMPLE_ROWS)  # workers started and their memory touched before timing
        runs = [op.run(data, 0, CPU_SAMPLE_ROWS) for _ in range(3)]
    finally:
        op.close()
    secs = statistics.median(r[0] for r in runs)
    nbytes = runs[0][1]
    return {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s", "cores": op.cores, "kind": "oracle",
            "blas_threads_per_worker": 1,
            "sample": f"unpack + dequant + float64 product of the first {CPU_SAMPLE_ROWS} output rows of each of "
                      f"the 4 decode projections (M=1), split over {op.cores} spawn-started worker processes "
                      "(all host cores, one BLAS thread each); median of 3 after a warm-up pass"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    data = _oracle_sample(CPU_SAMPLE_ROWS)
    op = OraclePool()
    steps = args.warmup + args.steps
    # each step a slice of the sample, sized so that the whole run stays
    # within a few minutes whatever the step count
    per = max(op.cores, min(CPU_SAMPLE_ROWS, (16 * CPU_SAMPLE_ROWS) // steps))
    times, nbytes = [], 0.0
    try:
        op.run(data, 0, CPU_SAMPLE_ROWS)  # workers started and their memory touched before timing
        for s in range(steps):
            r0 = (s * per) % CPU_SAMPLE_ROWS
            r1 = min(CPU_SAMPLE_ROWS, r0 + per)
            dt, nb = op.run(data, r0, r1)
            if s >= args.warmup:
                times.append(dt)
                nbytes += nb
    finally:
        op.close()
    sec = sum(times)
    value = nbytes / sec / 1e9
    sample = (f"oracle (float64 CPU reference) on {op.cores} worker processes (all host cores, one BLAS thread each): "
              f"{per} output rows of each of the 4 decode projections per step")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec / len(times) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "decode step: 4 Llama-7B-like W4A16 g128 projections at M=1 (row sample)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": op.cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


PROFILE_CASES = {
    # name: (launch kind, M, [(N, K, seed)], outliers)
    "decode": ("gemv", 1, DECODE, False),
    "prefill": ("gemm", PREFILL_M, PREFILL, True),
    "large": ("gemv", 1, [(32768, 32768, 12)], False),
    "large_gemm": ("gemm", 4096, [(32768, 8192, 10)], False),
}


def run_profile(case: str, reps: int):
    """A short, untimed run of one workload's launches, for profiler captures.

    Every launch runs `reps` times, in the order of the benchmark's step, on
    one weight copy; nothing is timed or printed but a one-line summary.
    """
    import torch

    import gemv_tf_prepack_gb300 as tf
    from gemv_tf_prepack_gb300 import synth

    kind, M, shapes, outliers = PROFILE_CASES[case]
    torch.cuda.set_device(0)
    layers = build_layers(torch, tf, synth, shapes, M, outliers, 1)
    fn = tf.gemv if kind == "gemv" else tf.gemm
    for _ in range(reps):
        for L in layers:
            fn(L["Ws"][0], L["xs"][0], L["ys"][0])
    torch.cuda.synchronize()
    err = tf.device_error()
    print(f"profile {case}: {reps} x {len(layers)} {kind} launches, device error {err}")
    if err:
        sys.exit(1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the square, large and small-layer measurements")
    ap.add_argument("--profile", choices=sorted(PROFILE_CASES),
                    help="run one workload's launches a few times, untimed (for ncu captures)")
    ap.add_argument("--profile-reps", type=int, default=2)
    args = ap.parse_args()
    if args.profile:
        run_profile(args.profile, args.profile_reps)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and args.impl == "ours":
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        torch.distributed.init_process_group("nccl")
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, world)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and args.impl == "ours":
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
