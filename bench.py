#!/usr/bin/env python3
"""Benchmark of the B300 selective-scan (S6) hot path.

One step = one ss_scan_fwd pass over the Mamba-2.8B-shaped layer workload
(batch 4, L 2048, d_inner 5120, d_state 16, bf16 inputs and output, fp32
state), inputs resident in HBM. Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU (launched by torch.distributed.run): every rank processes its own
copy of the workload (independent batches, no data-path collective; weak
scaling); the timed region is bracketed by barriers and the slowest rank's
time is taken.
"""

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from workloads import configs, gen  # noqa: E402

METRIC = "selective-scan HBM GB/s (% of B300 peak) & channel-tokens/s; decode steps/s"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "sm_max_mhz": 2032.0}
KERNEL_SOURCES = ["selective_state_space_130_b300/csrc/ss_scan_fwd_kernel.cuh",
                  "selective_state_space_130_b300/csrc/ss_device.cuh",
                  "selective_state_space_130_b300/csrc/ss_internal.h"]
SCAN_PROFILE = "profiles/ss_scan_fwd_mamba2p8b_layer.md"
# Compute roof of the state update: each (t, d, n) needs at least 4 fp32 pipe
# operations (delta*A, (delta*u)*B, the h FMA, the C.h FMA) and one MUFU ex2.
# A B300 SM has 128 fp32 lanes and retires 32 ex2 per clock, so at most 32 state
# updates per clock per SM (both pipes saturated, no other work).
STATE_UPDATES_PER_CLK_SM = 32.0
SMS = 148


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ------------------------------------------------------------------ setup
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, local):
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(world, v):
    """Slowest rank's value (timing is max over ranks); works on nccl and gloo."""
    if world == 1:
        return v
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(w, rank):
    """Each rank scans its own batch: independent inputs, no exchange."""
    return w.seed + 1000 * rank


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region (read-only)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"ss_bench_clocks_{os.getpid()}_rank{index}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def sources_sha():
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """dram bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source; else None."""
    p = os.path.join(ROOT, SCAN_PROFILE)
    if not os.path.exists(p):
        return None
    vals = {}
    for line in open(p):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha") != sources_sha():
        return None
    try:
        return float(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------ our arm
def to_dev(x, dev):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def scan_call(ss, d, y, h, ws):
    ss.ss_scan_fwd(d["u"], d["delta_raw"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"], None,
                   y=y, h_last=h, workspace=ws)


def bench_scan(ss, w, x, steps, warmup, out_dtype, dev, nsets=None):
    """Device-resident timing. Input sets rotate so consecutive steps never
    find their inputs in L2 (each set is larger than L2 or sets are cycled
    until the cycle is). Returns per-launch and total times in ms."""
    set_bytes = w.algorithmic_bytes("bf16")
    if nsets is None:
        nsets = max(2, math.ceil(3 * 126e6 / set_bytes) + 1)
    base = to_dev(x, dev)
    sets = [base] + [{k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in base.items()}
                     for _ in range(nsets - 1)]
    Bt, L, Dm = w.batch, w.seqlen, w.dim
    ys = [torch.empty((Bt, L, Dm), dtype=out_dtype, device=dev) for _ in range(nsets)]
    hs = [torch.empty((Bt, Dm, 16), dtype=torch.float32, device=dev) for _ in range(nsets)]
    ws_bytes = ss.ss_scan_fwd_workspace_size(Bt, L, Dm)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev) if ws_bytes else None
    stream = torch.cuda.current_stream()
    for i in range(warmup):
        k = i % nsets
        scan_call(ss, sets[k], ys[k], hs[k], ws)
    torch.cuda.synchronize()
    ss.ss_scan_status(ws)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # one scan kernel per step (the workspace clear before it is a memset)
    return dict(sets=sets, ys=ys, hs=hs, ws=ws, ev=ev, t0=t0, t1=t1, nsets=nsets, stream=stream,
                launches_per_step=1)


def prime_queue(cycles=2_000_000):
    """Open a timed region behind a device-side spin (by default 2 M cycles,
    about 1 ms). While it runs the host queues the timed launches, so their
    launch latency is not counted as GPU time; every timed step's work still
    runs inside the region. (With the GPU idle at the start event, the first
    call of a batch measured 420-510 us against 224 us for the rest.)"""
    torch.cuda._sleep(int(cycles))


def spin_for(call, reps, probe=5):
    """Spin cycles that cover the host's submission of `reps` timed calls: the
    host time of one call with its two event records, measured on `probe`
    calls queued behind a spin, times reps, with margin. A kernel shorter than
    its host call (the convolution front-end: about 35 us on the device
    against 50-90 us on the host) would otherwise drain the queue after the
    default spin, and the later intervals would hold host time."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(probe)]
    torch.cuda._sleep(4_000_000)  # about 2 ms: the probe calls queue behind it
    t = time.perf_counter()
    for i in range(probe):
        ev[i][0].record()
        call(i)
        ev[i][1].record()
    host_s = (time.perf_counter() - t) / probe
    torch.cuda.synchronize()
    return max(2_000_000, min(int(1.5 * reps * host_s * 2.1e9), 40_000_000))


def run_timed(ss, st, steps):
    prime_queue()
    st["t0"].record()
    for i in range(steps):
        k = i % st["nsets"]
        st["ev"][i][0].record()
        scan_call(ss, st["sets"][k], st["ys"][k], st["hs"][k], st["ws"])
        st["ev"][i][1].record()
    st["t1"].record()


def timed_results(st, steps):
    total = st["t0"].elapsed_time(st["t1"])
    per = [a.elapsed_time(b) for a, b in st["ev"]]
    return total, per


def bench_e2e(ss, w, x, steps, warmup, out_dtype, dev, nstreams=3):
    """Through the public call with HOST buffers: every step copies its inputs
    from pinned host memory, runs the scan and copies y and h_last back. The
    batch elements are independent scans, so each one is copied in, scanned and
    copied out on one of `nstreams` streams in turn: the copies of one element
    overlap the scan of another and the two copy directions overlap each other."""
    keys = ("u", "delta_raw", "z", "B", "C")
    host = {k: x[k].pin_memory() for k in keys}
    params = to_dev({k: x[k] for k in ("A", "D", "delta_bias")}, dev)
    Bt, L, Dm = w.batch, w.seqlen, w.dim
    y_host = torch.empty((Bt, L, Dm), dtype=out_dtype).pin_memory()
    h_host = torch.empty((Bt, Dm, 16), dtype=torch.float32).pin_memory()
    S = max(1, min(nstreams, Bt))
    streams = [torch.cuda.Stream(device=dev) for _ in range(S)]
    # per-stream device buffers for one batch element
    dbuf = [{k: torch.empty_like(host[k][:1], device=dev) for k in keys} for _ in range(S)]
    ys = [torch.empty((1, L, Dm), dtype=out_dtype, device=dev) for _ in range(S)]
    hs = [torch.empty((1, Dm, 16), dtype=torch.float32, device=dev) for _ in range(S)]
    ws_bytes = ss.ss_scan_fwd_workspace_size(1, L, Dm)
    wss = [torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev) if ws_bytes else None for _ in range(S)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = y_host.numel() * y_host.element_size() + h_host.numel() * 4
    main = torch.cuda.current_stream(dev)

    def one():
        start = torch.cuda.Event()
        start.record(main)
        for st in streams:
            st.wait_event(start)
        for b in range(Bt):
            k = b % S
            with torch.cuda.stream(streams[k]):
                for key in keys:
                    dbuf[k][key].copy_(host[key][b:b + 1], non_blocking=True)
                scan_call(ss, dict(dbuf[k], **params), ys[k], hs[k], wss[k])
                y_host[b:b + 1].copy_(ys[k], non_blocking=True)
                h_host[b:b + 1].copy_(hs[k], non_blocking=True)
        for st in streams:
            done = torch.cuda.Event()
            done.record(st)
            main.wait_event(done)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(main)
    for _ in range(steps):
        one()
    b.record(main)
    torch.cuda.synchronize()
    for k in range(S):
        ss.ss_scan_status(wss[k], stream=streams[k])
    return a.elapsed_time(b) / steps, h2d, d2h, S


def bench_decode(ss, w, dev, timed_steps=64, warmup=8):
    """Decode steps of the 256-stream workload. Cold: an L2 flush (write of a
    buffer larger than L2) before every timed step, each step timed alone.
    Warm: back-to-back steps (the 84 MB state may stay in the 126 MB L2)."""
    S, Dm = w.streams, w.dim
    A, Dk, bias = gen.make_params(w.prefix)
    nin = 16
    steps = gen.make_decode_steps(w, 0, nin)
    su = {k: v.to(dev) for k, v in steps.items()}
    A, Dk, bias = A.to(dev), Dk.to(dev), bias.to(dev)
    g = torch.Generator(device=dev).manual_seed(4)
    h = 0.1 * torch.randn((S, Dm, 16), generator=g, device=dev, dtype=torch.float32)
    y = torch.empty((S, Dm), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(64 << 20, dtype=torch.float32, device=dev)  # 256 MB, read after the fill

    def step(k):
        ss.ss_state_update(h, su["u"][k], su["delta_raw"][k], A, su["B"][k], su["C"][k], Dk, su["z"][k], bias, y=y)

    for k in range(warmup):
        step(k % nin)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(timed_steps)]
    for i in range(timed_steps):
        # evict the state from L2: write a buffer larger than L2, then read
        # another one, so the step does not also pay for writing back the
        # flush's dirty lines
        flush.fill_(i & 0xFF)
        flush_rd.sum()
        ev[i][0].record()
        step(i % nin)
        ev[i][1].record()
    torch.cuda.synchronize()
    cold = [a.elapsed_time(b) for a, b in ev]
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    nwarm = 1000
    a.record()
    for i in range(nwarm):
        step(i % nin)
    b.record()
    torch.cuda.synchronize()
    warm_ms = a.elapsed_time(b) / nwarm
    # the same back-to-back steps captured in one CUDA graph: the device rate
    # without a Python call and a launch per step
    ngraph = 200
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(ngraph):
            step(i % nin)
    graph.replay()
    torch.cuda.synchronize()
    a.record()
    for _ in range(5):
        graph.replay()
    b.record()
    torch.cuda.synchronize()
    graph_ms = a.elapsed_time(b) / (5 * ngraph)
    del graph
    cold_ms = statistics.mean(cold)
    bytes_step = w.algorithmic_bytes_per_step("bf16")
    return {"workload": f"{w.name}: {S} streams x d_inner {Dm} x d_state 16, bf16 inputs/y, fp32 state",
            "steps_per_s": 1e3 / cold_ms, "ms_per_step": cold_ms, "hbm_gbs": bytes_step / (cold_ms * 1e-3) / 1e9,
            "tokens_per_s": S * 1e3 / cold_ms, "l2": "flushed before every timed step (256 MB write, 256 MB read)",
            "warm_steps_per_s": 1e3 / warm_ms,
            "warm_note": "1000 back-to-back steps, one Python call and launch each (bound by the host dispatch); "
                         "state may stay in L2",
            "graph_steps_per_s": 1e3 / graph_ms,
            "graph_note": f"{ngraph} back-to-back steps captured in one CUDA graph, replayed 5 times; state may stay in L2"}


def bench_conv1d(ss, dev, hbm_peak, Bt=4, L=2048, Dm=5120, K=4, reps=20):
    """The block's causal depthwise convolution front-end (width 4, SiLU) on the
    Mamba-2.8B layer shape, bf16 in and out: HBM-bound, 4 bytes per channel-token.
    Two rotating input/output sets (each larger than L2). Plus the decode step
    of its state for 256 streams x 5120 channels."""
    sets = []
    for i in range(2):
        x = gen.random_conv_inputs(Bt, L, Dm, K, "bf16", seed=20 + i)
        sets.append({k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()})
    ys = [torch.empty((Bt, L, Dm), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    sts = [torch.empty((Bt, Dm, K - 1), dtype=torch.bfloat16, device=dev) for _ in range(2)]

    def call(i):
        d = sets[i % 2]
        ss.ss_conv1d_fwd(d["x"], d["weight"], d["bias"], None, y=ys[i % 2], state_out=sts[i % 2])

    for i in range(3):
        call(i)
    torch.cuda.synchronize()
    spin = spin_for(call, reps)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    prime_queue(spin)
    for i in range(reps):
        ev[i][0].record()
        call(i)
        ev[i][1].record()
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    nbytes = Bt * L * Dm * 4 + Bt * Dm * (K - 1) * 2
    # decode step of the conv state: 256 streams x 5120 channels
    S = 256
    st = torch.randn(S, Dm, K - 1, device=dev).to(torch.bfloat16)
    xs = torch.randn(S, Dm, device=dev).to(torch.bfloat16)
    d = sets[0]
    yd = torch.empty((S, Dm), dtype=torch.bfloat16, device=dev)
    for _ in range(5):
        ss.ss_conv1d_update(st, xs, d["weight"], d["bias"], y=yd)
    torch.cuda.synchronize()
    # 200 steps captured in one CUDA graph: the step is a few microseconds of
    # GPU work, below the host cost of a Python call
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(200):
            ss.ss_conv1d_update(st, xs, d["weight"], d["bias"], y=yd)
    graph.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    graph.replay()
    b.record()
    torch.cuda.synchronize()
    dec_ms = a.elapsed_time(b) / 200
    return {"workload": f"causal depthwise conv1d + SiLU, width {K}, batch {Bt} x L {L} x d_inner {Dm}, bf16 in/out",
            "ms_per_launch": round(ms, 4), "hbm_gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
            "frac_of_hbm_peak": round(nbytes / (ms * 1e-3) / 1e9 / hbm_peak, 4), "algorithmic_bytes": nbytes,
            "l2": "2 rotating sets of 168 MB",
            "decode_update_us": round(dec_ms * 1e3, 2),
            "decode_update_workload": f"{S} streams x {Dm} channels, width {K}, 200 steps in one CUDA graph"}


# Compute roof of the backward pass per (t, d, n): recomputing the state and
# the readout C.h (4 fp32 lane-ops and one ex2), the adjoint update and its
# products (lambda += C dyv; lambda *= Abar; the dB and dC terms; the du, d delta
# and dA sums: 9 lane-ops), and the channel sums of the dB and dC terms (2 adds):
# 15 fp32 lane-ops, so at most 128 / 15 state updates per clock per SM.
BWD_UPDATES_PER_CLK_SM = 128.0 / 15.0


def bench_scan_bwd(ss, w, dev, hbm_peak, clock_mhz, reps=10):
    """Gradients of the scan (ss_scan_bwd) on the Mamba-2.8B layer shape: bf16
    inputs and output gradient, fp32 dh_last. One input set of 420 MB (larger
    than L2)."""
    x = to_dev(gen.make_scan_inputs(w), dev)
    Bt, L, Dm, N = w.batch, w.seqlen, w.dim, w.dstate
    dy, dh = gen.random_output_grads(Bt, L, Dm, N, "bf16", seed=5)
    dy, dh = dy.to(dev), dh.to(dev)
    ws = torch.empty(ss.ss_scan_bwd_workspace_size(Bt, L, Dm, N), dtype=torch.uint8, device=dev)

    def call(out=None):
        return ss.ss_scan_bwd(x["u"], x["delta_raw"], x["A"], x["B"], x["C"], dy, x["D"], x["z"], x["delta_bias"],
                              None, dh, out=out, workspace=ws)

    out = call()  # allocates the gradients once
    for _ in range(3):
        call(out)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    prime_queue()
    for i in range(reps):
        ev[i][0].record()
        call(out)
        ev[i][1].record()
    torch.cuda.synchronize()
    per = [a.elapsed_time(b) for a, b in ev]
    ms = statistics.mean(per)
    # algorithmic bytes: read u, delta_raw, z, dy and write du, ddelta_raw, dz
    # (bf16, 14 B per channel-token); read B, C (bf16) and write dB, dC (fp32)
    # per token; dh_last in, dh0 out (fp32); A, D, bias in and their gradients out
    nbytes = (Bt * L * Dm * 14 + Bt * L * N * (2 * 2 + 2 * 4) + 2 * Bt * Dm * N * 4 + 2 * Dm * (N + 2) * 4)
    updates = Bt * L * Dm * N
    alu_peak = BWD_UPDATES_PER_CLK_SM * SMS * clock_mhz * 1e6
    achieved = updates / (ms * 1e-3)
    del x, dy, dh, ws, out
    torch.cuda.empty_cache()
    return {"workload": f"gradients of the scan, {w.name}: batch {Bt}, L {L}, d_inner {Dm}, d_state {N}, "
                        "bf16 inputs / dy / du, ddelta_raw, dz; fp32 dA, dB, dC, dD, dbias, dh0",
            "ms_per_launch": round(ms, 4), "ms_per_launch_median": round(statistics.median(per), 4),
            "ms_per_launch_min": round(min(per), 4), "launches_per_call": 1,
            "channel_tokens_per_s": Bt * L * Dm / (ms * 1e-3),
            "roofline": {"bound": "alu", "unit": "state updates/s", "achieved": achieved, "peak": alu_peak,
                         "frac": round(achieved / alu_peak, 4),
                         "basis": "15 fp32 lane-ops per (t,d,n) (state and readout recompute 4, adjoint 9, "
                                  "channel sums of the dB/dC terms 2): 128 lanes / 15 per clk per SM x 148 SMs "
                                  "x median SM clock of the main run"},
            "hbm": {"algorithmic_bytes": nbytes, "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
                    "frac_of_hbm_peak": round(nbytes / (ms * 1e-3) / 1e9 / hbm_peak, 4)},
            "l2": "one input set of 420 MB (larger than L2)"}


# Compute roof of the generalised scan per (t, d, n): first order as the scan
# (4 fp32 lane-ops and one ex2: 32 per clock per SM); the zero-order hold adds
# Abar - 1 and the products with u / A (7 lane-ops: 128 / 7 per clock per SM).
GEN_UPDATES_PER_CLK_SM = {"first_order": 32.0, "zoh": 128.0 / 7.0}


def bench_general(ss, w, dev, hbm_peak, clock_mhz, N, G, disc, reps=10):
    """ss_scan_fwd_general on the Mamba-2.8B layer shape with a larger state:
    bf16 inputs and y; one input set (larger than L2)."""
    x = to_dev(gen.random_general_inputs(w.batch, w.seqlen, w.dim, N, G, in_dtype="bf16", seed=N + G), dev)
    Bt, L, Dm = w.batch, w.seqlen, w.dim
    y = torch.empty((Bt, L, Dm), dtype=torch.bfloat16, device=dev)
    h = torch.empty((Bt, Dm, N), dtype=torch.float32, device=dev)
    # the split's workspace, allocated once outside the timed region
    ws_bytes = ss.ss_scan_fwd_general_workspace_size(Bt, L, Dm, N, G, disc, torch.bfloat16)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else False

    def call():
        ss.ss_scan_fwd_general(x["u"], x["delta_raw"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"], None,
                               disc=disc, y=y, h_last=h, workspace=ws)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    prime_queue()
    for i in range(reps):
        ev[i][0].record()
        call()
        ev[i][1].record()
    torch.cuda.synchronize()
    per = [a.elapsed_time(b) for a, b in ev]
    ms = statistics.mean(per)
    nbytes = Bt * L * Dm * 8 + Bt * L * G * N * 2 * 2 + Bt * Dm * N * 4 + Dm * (N + 2) * 4
    updates = Bt * L * Dm * N
    alu_peak = GEN_UPDATES_PER_CLK_SM[disc] * SMS * clock_mhz * 1e6
    achieved = updates / (ms * 1e-3)
    del x, y, h, ws
    torch.cuda.empty_cache()
    return {"workload": f"generalised scan, {w.name} shape: batch {Bt}, L {L}, d_inner {Dm}, d_state {N}, "
                        f"{G} group(s) of B/C, {disc} Bbar, bf16 inputs and y",
            "ms_per_launch": round(ms, 4), "ms_per_launch_median": round(statistics.median(per), 4),
            "ms_per_launch_min": round(min(per), 4),
            "roofline": {"bound": "alu", "unit": "state updates/s", "achieved": achieved, "peak": alu_peak,
                         "frac": round(achieved / alu_peak, 4),
                         "basis": ("4 fp32 lane-ops + 1 ex2 per (t,d,n): 32 per clk per SM" if disc == "first_order"
                                   else "7 fp32 lane-ops per (t,d,n) (first order's 4, Abar - 1, u / A and its "
                                        "product): 128 / 7 per clk per SM") + " x 148 SMs x median SM clock"},
            "hbm": {"algorithmic_bytes": nbytes, "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
                    "frac_of_hbm_peak": round(nbytes / (ms * 1e-3) / 1e9 / hbm_peak, 4)},
            "l2": "one input set larger than L2"}


def bench_ssd(ss, dev, hbm_peak, tensor_peak, Bt=4, L=2048, H=80, N=128, G=1, reps=10):
    """ss_ssd_fwd (state-space-dual layer, tensor-core chunked form) on a Mamba-2
    2.7B-shaped layer: batch 4, L 2048, 80 heads x 64 channels (d_inner 5120),
    d_state 128, one group, bf16 in and out. One input set (larger than L2)."""
    P = 64
    Q = 128 if N == 128 else 64  # the kernel's chunk length
    x = to_dev(gen.random_ssd_inputs(Bt, L, H, P, N, G, in_dtype="bf16", seed=11), dev)
    y = torch.empty((Bt, L, H, P), dtype=torch.bfloat16, device=dev)
    hl = torch.empty((Bt, H, P, N), dtype=torch.float32, device=dev)
    nws = ss.ss_ssd_fwd_workspace_size(Bt, L, H, N)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev) if nws else False

    def call():
        ss.ss_ssd_fwd(x["x"], x["dt"], x["A"], x["B"], x["C"], x["D"], x["dt_bias"], None, y=y, h_last=hl,
                      workspace=ws)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    spin = spin_for(lambda i: call(), reps)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    prime_queue(spin)
    for i in range(reps):
        ev[i][0].record()
        call()
        ev[i][1].record()
    torch.cuda.synchronize()
    per = [a.elapsed_time(b) for a, b in ev]
    ms = statistics.mean(per)
    # bytes: x in and y out (bf16), dt, B, C in, the final state out
    nbytes = Bt * L * H * P * 2 * 2 + Bt * L * H * 2 + Bt * L * G * N * 2 * 2 + Bt * H * P * N * 4
    # flops of the chunked form per (batch, head, chunk): the causal half of C B^T
    # (Q(Q+1)/2 x N) and of M X (Q(Q+1)/2 x P), C H_in (Q x N x P) and B^T X (N x Q x P), 2 per multiply-add
    tri = Q * (Q + 1) // 2
    flops = Bt * H * ((L + Q - 1) // Q) * 2 * (tri * N + tri * P + Q * N * P + N * Q * P)
    t = ms * 1e-3
    del x, y, hl
    torch.cuda.empty_cache()
    return {"workload": f"state-space-dual (Mamba-2) layer: batch {Bt}, L {L}, {H} heads x {P} channels, d_state {N}, "
                        f"{G} group, chunks of {Q}, bf16 in/out",
            "ms_per_launch": round(ms, 4), "ms_per_launch_median": round(statistics.median(per), 4),
            "ms_per_launch_min": round(min(per), 4), "channel_tokens_per_s": Bt * L * H * P / t,
            "roofline": {"bound": "hbm", "achieved": round(nbytes / t / 1e9, 1), "peak": hbm_peak, "unit": "GB/s",
                         "frac": round(nbytes / t / 1e9 / hbm_peak, 4), "algorithmic_bytes": nbytes,
                         "note": "at the measured peaks the bytes take longer than the algorithmic flops"},
            "tensor": {"algorithmic_flops": flops, "achieved_tflops": round(flops / t / 1e12, 2),
                       "peak_tflops": tensor_peak, "frac": round(flops / t / 1e12 / tensor_peak, 4),
                       "note": "tcgen05.mma kind::f16 (bf16 operands, fp32 accumulators in tensor memory); "
                               "operands computed on chip (M, X', the state) run as two bf16 parts, so the tensor "
                               "pipe executes about 1.8x the algorithmic flops"},
            "l2": "one input set of 176 MB (larger than L2)"}


def cpu_baseline_scan(w, x, target_s=12.0):
    """The float64 oracle as it stands, on the host cores, over channels of the
    same workload; scaled to algorithmic GB/s of the sample."""
    import oracle

    nthreads = oracle.default_threads()
    per_ch_bytes = w.algorithmic_bytes("bf16") / (w.batch * w.dim)
    rng = np.random.default_rng(0)
    n = min(w.batch * w.dim, 256)
    total_ch, total_t = 0, 0.0
    while True:
        ch = np.stack([rng.integers(0, w.batch, n), rng.integers(0, w.dim, n)], axis=1)
        t = time.perf_counter()
        oracle.scan(x, channels=ch, nthreads=nthreads)
        dt = time.perf_counter() - t
        total_ch += n
        total_t += dt
        if total_t >= target_s or total_ch >= w.batch * w.dim:
            break
        n = int(min(w.batch * w.dim - total_ch, max(n, n * (target_s - total_t) / max(dt, 1e-3))))
        n = max(n, 1)
    gbs = per_ch_bytes * total_ch / total_t / 1e9
    return {"value": gbs, "unit": "GB/s", "cores": nthreads, "kind": "oracle",
            "sample": f"{total_ch} of {w.batch * w.dim} channels x {w.seqlen} tokens of {w.name}, "
                      f"{total_t:.1f} s wall", "channel_tokens_per_s": total_ch * w.seqlen / total_t}


def cpu_oracle_sample(w, x, target_s=3.0):
    """The float64 oracle on a bounded sample of channels of workload w: all
    host cores, and (on the short-sequence layers) one thread, as
    channel-tokens/s and algorithmic GB/s of the sample."""
    import oracle

    nthreads = oracle.default_threads()
    per_ch_bytes = w.algorithmic_bytes("bf16") / (w.batch * w.dim)
    rng = np.random.default_rng(2)
    out = {"cores": nthreads}
    for label, nt in (("all_cores", nthreads), ("one_thread", 1)):
        if label == "one_thread" and w.seqlen > 65536:
            continue
        n, total_ch, total_t = nt, 0, 0.0
        while total_t < target_s and total_ch < w.batch * w.dim:
            ch = np.stack([rng.integers(0, w.batch, n), rng.integers(0, w.dim, n)], axis=1)
            t = time.perf_counter()
            oracle.scan(x, channels=ch, nthreads=nt)
            dt = time.perf_counter() - t
            total_ch += n
            total_t += dt
            n = max(nt, int(min(w.batch * w.dim - total_ch, n * max(1.0, (target_s - total_t) / max(dt, 1e-3)))))
        out[label] = {"channel_tokens_per_s": total_ch * w.seqlen / total_t,
                      "gbs": per_ch_bytes * total_ch / total_t / 1e9, "threads": nt,
                      "sample": f"{total_ch} channels x {w.seqlen} tokens, {total_t:.1f} s wall"}
    return out


def run_ours(args, world, rank, local):
    import selective_state_space_130_b300 as ss

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = configs.get_config(args.workload)
    out_dtype = torch.bfloat16
    peaks, peak_kind = load_peaks()
    x = gen.make_scan_inputs(w, seed=rank_seed(w, rank))

    st = bench_scan(ss, w, x, args.steps, args.warmup, out_dtype, dev)
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    run_timed(ss, st, args.steps)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ss.ss_scan_status(st["ws"])
    total_ms, per = timed_results(st, args.steps)
    ms_step = max_over_ranks(world, total_ms / args.steps)
    per_launch_ms = statistics.mean(per)

    bytes_step = w.algorithmic_bytes("bf16")
    value = world * bytes_step / (ms_step * 1e-3) / 1e9
    achieved = bytes_step / (per_launch_ms * 1e-3) / 1e9
    hbm_peak = float(peaks["hbm_gbs"])
    clock_mhz = clk.get("sm_mhz") or float(peaks.get("sm_max_mhz", 2032.0))
    states = w.channel_tokens * w.dstate
    alu_peak = STATE_UPDATES_PER_CLK_SM * SMS * clock_mhz * 1e6
    alu_achieved = states / (per_launch_ms * 1e-3)

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{w.name}: batch {w.batch}, L {w.seqlen}, d_inner {w.dim}, d_state {w.dstate}, "
                               "bf16 u/delta_raw/z/B/C and y, fp32 A/D/bias/state",
                   "batch": w.batch, "seq_len": w.seqlen, "d_inner": w.dim, "d_state": w.dstate,
                   "global_batch": w.batch * world, "parallelism": f"replicas x{world} (independent batches)",
                   "l2": f"inputs larger than L2; {st['nsets']} rotating input/output sets"},
        "channel_tokens_per_s": world * w.channel_tokens / (ms_step * 1e-3),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "traffic": profiled_traffic(),
                     "peak_kind": peak_kind, "kernel": "ss_scan_fwd (scan_fwd_kernel)",
                     "per_launch_ms": round(per_launch_ms, 5),
                     "per_launch_ms_median": round(statistics.median(per), 5),
                     "per_launch_ms_min": round(min(per), 5), "algorithmic_bytes_per_launch": bytes_step},
        "compute_roofline": {"bound": "alu", "unit": "state updates/s", "achieved": alu_achieved,
                             "peak": alu_peak, "frac": round(alu_achieved / alu_peak, 4),
                             "basis": "4 fp32 lane-ops + 1 MUFU ex2 per (t,d,n): 128 fp32 lanes and 32 ex2 "
                                      "per clk per SM give 32 updates per clk per SM x 148 SMs x median SM "
                                      "clock under load"},
        "gpu_launches": args.steps * st["launches_per_step"],
        "clocks": clk,
    }
    del st
    torch.cuda.empty_cache()

    if rank == 0 and not args.no_e2e:
        e2e_ms, h2d, d2h, nstr = bench_e2e(ss, w, x, max(3, min(args.steps, 10)), 2, out_dtype, dev)
        result["e2e"] = {"value": round(bytes_step / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                         "path": "pinned host -> device copies, ss_scan_fwd, device -> pinned host copies, "
                                 f"one batch element per call on {nstr} streams in turn (copies overlap scans)"}
        torch.cuda.empty_cache()
    if rank == 0 and not args.no_decode:
        result["decode"] = bench_decode(ss, configs.DECODE256, dev)
        torch.cuda.empty_cache()
    if rank == 0 and not args.no_extra:
        extra = {}
        for name in ("mamba130m_layer", "dna_1m"):
            wc = configs.get_config(name)
            xc = gen.make_scan_inputs(wc)
            reps = 10 if name == "mamba130m_layer" else 3
            stc = bench_scan(ss, wc, xc, reps, 2, out_dtype, dev)
            torch.cuda.synchronize()
            run_timed(ss, stc, reps)
            torch.cuda.synchronize()
            tot, per = timed_results(stc, reps)
            ms = statistics.mean(per)
            bts = wc.algorithmic_bytes("bf16")
            extra[wc.name] = {"ms_per_launch": round(ms, 4), "hbm_gbs": round(bts / (ms * 1e-3) / 1e9, 1),
                              "frac_of_hbm_peak": round(bts / (ms * 1e-3) / 1e9 / hbm_peak, 4),
                              "channel_tokens_per_s": wc.channel_tokens / (ms * 1e-3),
                              "launches_per_step": stc["launches_per_step"], "l2": f"{stc['nsets']} rotating sets"}
            if not args.no_cpu_baseline:
                extra[wc.name]["cpu_oracle"] = cpu_oracle_sample(wc, xc)
            del stc, xc
            torch.cuda.empty_cache()
        extra["conv1d_front_end"] = bench_conv1d(ss, dev, hbm_peak)
        extra["scan_backward"] = bench_scan_bwd(ss, w, dev, hbm_peak, clock_mhz)
        extra["general_dstate64_zoh"] = bench_general(ss, w, dev, hbm_peak, clock_mhz, 64, 1, "zoh")
        extra["general_dstate128_8groups"] = bench_general(ss, w, dev, hbm_peak, clock_mhz, 128, 8, "first_order")
        extra["ssd_mamba2_2p7b_layer"] = bench_ssd(ss, dev, hbm_peak, float(peaks.get("bf16_tflops", 1786.4)))
        result["per_config"] = extra
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline_scan(w, x)
    return result


# ------------------------------------------------------------------ reference arm
def run_reference(args, world, rank):
    """The reference arm is the float64 CPU oracle as it stands, timed on the
    host cores over a bounded sample of the same workload per step."""
    if rank != 0:
        return None
    import oracle

    w = configs.get_config(args.workload)
    x = gen.make_scan_inputs(w)
    nthreads = oracle.default_threads()
    rng = np.random.default_rng(1)
    n = max(64, min(w.batch * w.dim, 256 * nthreads))
    per_ch_bytes = w.algorithmic_bytes("bf16") / (w.batch * w.dim)
    ch = np.stack([rng.integers(0, w.batch, n), rng.integers(0, w.dim, n)], axis=1)
    for _ in range(args.warmup):
        oracle.scan(x, channels=ch[: max(1, n // 8)], nthreads=nthreads)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle.scan(x, channels=ch, nthreads=nthreads)
    dt = (time.perf_counter() - t) / args.steps
    value = per_ch_bytes * n / dt / 1e9
    sample = f"{n} of {w.batch * w.dim} channels x {w.seqlen} tokens of {w.name} per step"
    return {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": f"{w.name}: batch {w.batch}, L {w.seqlen}, d_inner {w.dim}, d_state {w.dstate}, "
                               "bf16 inputs (oracle in float64)", "batch": w.batch, "seq_len": w.seqlen,
                   "d_inner": w.dim, "d_state": w.dstate},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": nthreads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def profile_launches(args):
    """Two launches of the scan (decode, backward) kernel on the chosen workload, no
    timing: the target of `ncu -k regex:... -s 1 -c 1`."""
    import selective_state_space_130_b300 as ss

    dev = torch.device("cuda", 0)
    if args.profile == "scan":
        w = configs.get_config(args.workload)
        x = to_dev(gen.make_scan_inputs(w), dev)
        Bt, L, Dm = w.batch, w.seqlen, w.dim
        y = torch.empty((Bt, L, Dm), dtype=torch.bfloat16, device=dev)
        h = torch.empty((Bt, Dm, 16), dtype=torch.float32, device=dev)
        nb = ss.ss_scan_fwd_workspace_size(Bt, L, Dm)
        ws = torch.empty(nb, dtype=torch.uint8, device=dev) if nb else None
        for _ in range(2):
            scan_call(ss, x, y, h, ws)
        ss.ss_scan_status(ws)
    elif args.profile == "conv1d":
        x = to_dev(gen.random_conv_inputs(4, 2048, 5120, 4, "bf16", seed=20), dev)
        for _ in range(2):
            ss.ss_conv1d_fwd(x["x"], x["weight"], x["bias"], None)
    elif args.profile == "ssd":
        x = to_dev(gen.random_ssd_inputs(4, 2048, 80, 64, 128, 1, in_dtype="bf16", seed=11), dev)
        for _ in range(2):
            ss.ss_ssd_fwd(x["x"], x["dt"], x["A"], x["B"], x["C"], x["D"], x["dt_bias"], None)
    elif args.profile in ("general", "general128"):
        # d_state 64, one group, zero-order hold; or d_state 128, 8 groups, first order
        N, G, disc = (64, 1, "zoh") if args.profile == "general" else (128, 8, "first_order")
        w = configs.get_config(args.workload)
        x = to_dev(gen.random_general_inputs(w.batch, w.seqlen, w.dim, N, G, in_dtype="bf16", seed=N + 1), dev)
        for _ in range(2):
            ss.ss_scan_fwd_general(x["u"], x["delta_raw"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"],
                                   None, disc=disc)
    elif args.profile == "bwd":
        w = configs.get_config(args.workload)
        x = to_dev(gen.make_scan_inputs(w), dev)
        Bt, L, Dm = w.batch, w.seqlen, w.dim
        dy, dh = gen.random_output_grads(Bt, L, Dm, 16, "bf16", seed=5)
        dy, dh = dy.to(dev), dh.to(dev)
        ws = torch.empty(ss.ss_scan_bwd_workspace_size(Bt, L, Dm), dtype=torch.uint8, device=dev)
        out = None
        for _ in range(2):
            out = ss.ss_scan_bwd(x["u"], x["delta_raw"], x["A"], x["B"], x["C"], dy, x["D"], x["z"],
                                 x["delta_bias"], None, dh, out=out, workspace=ws)
    else:
        w = configs.DECODE256
        A, Dk, bias = (t.to(dev) for t in gen.make_params(w.prefix))
        st = {k: v.to(dev) for k, v in gen.make_decode_steps(w, 0, 2).items()}
        h = torch.zeros((w.streams, w.dim, 16), dtype=torch.float32, device=dev)
        for k in range(2):
            ss.ss_state_update(h, st["u"][k], st["delta_raw"][k], A, st["B"][k], st["C"][k], Dk, st["z"][k], bias)
    torch.cuda.synchronize()


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mamba2p8b_layer",
                    help="tiny_fp32, mamba130m_layer, mamba2p8b_layer (default), dna_1m")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the per-config timings")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", choices=["scan", "decode", "bwd", "general", "general128", "ssd", "conv1d"],
                    default=None,
                    help="run 2 launches of one kernel (for an ncu capture of the 2nd) and exit")
    args = ap.parse_args()
    if args.profile:
        profile_launches(args)
        return
    if args.warmup < 3:
        log("warmup raised to 3 (timing rule)")
        args.warmup = 3
    world, rank, local = dist_env()
    if args.impl == "reference":
        res = run_reference(args, world, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    dist_init(world, local)
    res = run_ours(args, world, rank, local)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
