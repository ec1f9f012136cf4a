#!/usr/bin/env python3
"""Benchmark: bitmap SpMM GB/s (% of HBM peak) and effective TOPS at N = 1/8/16.

Workload (headline): W4A4 SpMM, W = 4096 x 4096 int4, 50 % magnitude-pruned
(per-row), 64 x 64 bitmap tiles, N in {1, 8, 16} int4 tokens, int32 accumulators
plus the fp16 dequantised output.  One step = one pass of the hot path
(staging, popcount/prefix decode, multiply, split-K reduction, epilogue) at
N = 1, 8 and 16 over every resident weight copy.  The encoded matrix is
replicated into enough distinct device buffers that one pass streams more than
twice the L2 size, so each launch reads its weights from HBM.  Launches are
captured in CUDA graphs (one per N) and timed with CUDA events on the launching
stream.

Bytes per call (algorithmic): bitmap M*K/8 + tile_off 4*(nT+1) + values (used
bytes, padding included) + X K*N/2 + scales 2M + 2N + outputs M*N*(4 + 2).
Effective TOPS = 2*M*K*N / t (dense-equivalent).

``--impl reference`` times the CPU oracle (test infrastructure, the reference
arm of this benchmark) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

M_, K_, SPARSITY, TM_, TK_ = 4096, 4096, 0.5, 64, 64
NS = (1, 8, 16)
HBM_MEASURED_FALLBACK = 6800.0


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1900.0)), "measured"
    except Exception:
        return HBM_MEASURED_FALLBACK, 1900.0, "fallback"


def call_bytes(values_bytes: int, M: int, K: int, N: int, TM: int, TK: int) -> int:
    nT = (M // TM) * (K // TK)
    return M * K // 8 + 4 * (nT + 1) + values_bytes + K * N // 2 + 2 * M + 2 * N + M * N * 6


# ----------------------------------------------------------------- clocks --
class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# -------------------------------------------------------------- reference --
class CpuSample:
    """The oracle on one 4096 x 4096 W4A4 matrix: decode the encoded form, then
    multiply, once for each of N = 1, 8 and 16 (one call each)."""

    def __init__(self):
        from bitmap_encoded_unstructured_ie_gb300 import workloads as wl
        from oracle import oracle as orc
        self.orc = orc
        self.d = wl.w4a4(M_, K_, max(NS), SPARSITY, seed=0)
        self.enc = orc.encode(self.d["Wq"], TM_, TK_, orc.I4, orc.ROW)
        self.pass_bytes = sum(call_bytes(self.enc[2].size, M_, K_, N, TM_, TK_) for N in NS)

    def one_pass(self, nthreads: int) -> float:
        orc, d = self.orc, self.d
        t0 = time.perf_counter()
        for N in NS:
            Wd = orc.decode(*self.enc, M_, K_, TM_, TK_, orc.I4, orc.ROW)
            orc.spmm_w4a4(Wd, d["Xq"][:N], d["s_w"], d["s_x"][:N], nthreads=nthreads)
        return time.perf_counter() - t0

    def timed(self, nthreads: int, min_seconds: float):
        passes, el = 0, 0.0
        while passes == 0 or el < min_seconds:
            el += self.one_pass(nthreads)
            passes += 1
        return self.pass_bytes * passes / el / 1e9, el / passes, passes


def run_reference(args):
    from bitmap_encoded_unstructured_ie_gb300 import replicas
    if replicas.rank_env()[1] != 0:
        return 0
    from oracle import oracle as orc
    orc.build()
    threads = orc.max_threads()
    smp = CpuSample()
    for _ in range(args.warmup):
        smp.one_pass(threads)
    times = [smp.one_pass(threads) for _ in range(args.steps)]
    step_s = sum(times) / len(times)
    value = smp.pass_bytes / step_s / 1e9
    line = {
        "impl": "reference", "metric": "bitmap SpMM GB/s (% of GB300 HBM peak) & effective TOPS at N=1/8/16",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_s * 1e3, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int4xint4->int32", "data": "synthetic",
        "config": {"workload": "W4A4 bitmap SpMM 4096x4096, 50% magnitude-pruned per row, 64x64 tiles, N=1/8/16",
                   "sample": "one weight matrix per step (of the GPU arm's rotating copies): oracle decode + "
                             "multiply at N=1, 8, 16"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": "one 4096x4096 W4A4 matrix per step (decode + N=1,8,16)"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm --
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--copies", type=int, default=0, help="resident weight copies (0 = enough for 2x L2)")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-baseline leg")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import torch
    from bitmap_encoded_unstructured_ie_gb300 import build as us_build
    from bitmap_encoded_unstructured_ie_gb300 import binding as us
    from bitmap_encoded_unstructured_ie_gb300 import workloads as wl

    from bitmap_encoded_unstructured_ie_gb300 import replicas
    world, rank, local = replicas.rank_env()
    dist = replicas.init(world, "nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    us_build.build()
    us.load()
    hbm_peak, bf16_peak, peak_src = peaks()
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20)

    # ---- workload and resident copies
    d = wl.w4a4(M_, K_, max(NS), SPARSITY, seed=0)
    E0 = us.us_encode(torch.from_numpy(d["Wq"]).to(dev), TM_, TK_, us.US_I4, us.US_ORDER_ROW)
    assert us.us_get_last_device_status() == us.US_OK
    E0.flags = us.US_BITMAP_STATIC          # inference weights: nothing earlier on the stream writes them
    per_copy = E0.nbytes()
    L = args.copies or max(4, math.ceil(2.2 * l2 / per_copy))
    copies = [E0] + [us.Encoded(E0.M, E0.K, E0.TM, E0.TK, E0.elem, E0.order, E0.bitmap.clone(),
                                E0.tile_off.clone(), E0.values.clone(), E0.values_bytes, E0.flags)
                     for _ in range(L - 1)]
    sw = torch.from_numpy(d["s_w"].view(np.int16)).to(dev)
    X, SX, Yacc, Y, WS = {}, {}, {}, {}, {}
    for N in NS:
        X[N] = torch.from_numpy(wl.pack_int4(d["Xq"][:N])).to(dev)
        SX[N] = torch.from_numpy(d["s_x"][:N].view(np.int16)).to(dev)
        Yacc[N] = torch.empty(N, M_, dtype=torch.int32, device=dev)
        Y[N] = torch.empty(N, M_, dtype=torch.int16, device=dev)
        WS[N] = us.workspace(us.US_OP_SPMM_W4A4, E0, N)

    stream = torch.cuda.Stream(dev)

    def launch_all(N):
        for E in copies:
            us.us_spmm_w4a4(E, X[N], sw, SX[N], N, Yacc[N], Y[N], WS[N], 0, stream)

    with torch.cuda.stream(stream):
        for N in NS:                       # eager warm-up (module load, attributes)
            launch_all(N)
    stream.synchronize()
    assert us.us_get_last_device_status(stream) == us.US_OK
    graphs = {}
    for N in NS:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            launch_all(N)
        graphs[N] = g
    with torch.cuda.stream(stream):        # replays run on the current stream
        for _ in range(args.warmup):
            for N in NS:
                graphs[N].replay()
    stream.synchronize()
    assert us.us_get_last_device_status(stream) == us.US_OK

    # ---- timed region
    ev = {N: ([], []) for N in NS}
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    replicas.barrier(dist)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for _ in range(args.steps):
            for N in NS:
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                graphs[N].replay()
                b.record(stream)
                ev[N][0].append(a)
                ev[N][1].append(b)
        t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    replicas.barrier(dist)
    total_ms = replicas.max_over_ranks(dist, t_start.elapsed_time(t_end), dev)
    assert us.us_get_last_device_status(stream) == us.US_OK

    per_n = {}
    step_bytes = 0
    for N in NS:
        ms = sum(a.elapsed_time(b) for a, b in zip(*ev[N]))
        us_per_launch = ms * 1e3 / (args.steps * L)
        b_call = call_bytes(E0.values_bytes, M_, K_, N, TM_, TK_)
        step_bytes += b_call * L
        gbs = b_call / (us_per_launch * 1e-6) / 1e9
        per_n[str(N)] = {
            "us_per_launch": round(us_per_launch, 3), "bytes_per_call": b_call, "GB/s": round(gbs, 1),
            "pct_hbm_measured": round(100 * gbs / hbm_peak, 1), "pct_hbm_8TBs": round(100 * gbs / 8000, 1),
            "eff_TOPS": round(2 * M_ * K_ * N / (us_per_launch * 1e-6) / 1e12, 2),
            "split_k": us.us_pick_split_k(us.US_OP_SPMM_W4A4, E0, N),
            "kernel": kernel_name(N), "share": None,
        }
    tot = sum(v["us_per_launch"] for v in per_n.values())
    for v in per_n.values():
        v["share"] = round(v["us_per_launch"] / tot, 3)
    step_ms = total_ms / args.steps
    value = replicas.aggregate_rate(step_bytes, world, step_ms * 1e-3) / 1e9
    # dominant kernel: largest time share
    dom_n = max(per_n, key=lambda k: per_n[k]["us_per_launch"])
    dom = per_n[dom_n]
    traffic = load_traffic(dom["kernel"])
    roofline = {"bound": "hbm", "achieved": dom["GB/s"], "peak": hbm_peak, "unit": "GB/s",
                "frac": round(dom["GB/s"] / hbm_peak, 4), "traffic": traffic,
                "kernel": dom["kernel"], "at_N": int(dom_n), "peak_source": peak_src}

    e2e = measure_e2e(us, torch, wl, d, copies, sw, dev, stream, args, L)
    # whole job: every replica's bytes over the slowest replica's time
    e2e_ms = replicas.max_over_ranks(dist, e2e["ms_per_step"], dev)
    e2e["value"] = round(replicas.aggregate_rate(e2e.pop("_bytes_per_step"), world, e2e_ms * 1e-3) / 1e9, 1)
    e2e["ms_per_step"] = round(e2e_ms, 4)

    extras = {}
    if not args.no_extras and rank == 0:
        # secondary rows: a failure there is reported in the line, and does not
        # take the headline measurement down with it
        try:
            extras = measure_extras(us, torch, wl, dev, stream, hbm_peak, bf16_peak,
                                    cpu=(world == 1 and not args.no_cpu))
        except Exception as e:                       # noqa: BLE001
            extras = {"error": f"{type(e).__name__}: {e}"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        from oracle import oracle as orc
        threads = orc.max_threads()
        gbs, t_pass, passes = CpuSample().timed(threads, args.cpu_seconds)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": f"one 4096x4096 W4A4 matrix: oracle decode + multiply at N=1,8,16, {passes} passes "
                         f"({t_pass:.2f} s each) on {threads} threads"}

    line = {
        "metric": "bitmap SpMM GB/s (% of GB300 HBM peak) & effective TOPS at N=1/8/16",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int4xint4->int32", "data": "synthetic",
        "config": {"workload": "W4A4 bitmap SpMM 4096x4096, 50% magnitude-pruned per row, 64x64 tiles, N=1/8/16",
                   "weight_copies": L, "bytes_per_copy": per_copy,
                   "l2": f"inputs larger than L2: {L} resident weight copies = {L * per_copy / 2**20:.0f} MiB "
                         f"> 2 x L2 ({l2 / 2**20:.0f} MiB)", "graphs": "one CUDA graph per N, L launches each",
                   "parallelism": f"replicas x{world} (independent weight sets, no collective)",
                   "weights": "flagged US_BITMAP_STATIC: a launch may fetch its weights while the previous "
                              "launch drains (programmatic dependent launch)"},
        "per_n": per_n,
        "roofline": roofline,
        "gpu_launches": args.steps * L * len(NS),
        "clocks": clk,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "extras": extras,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    replicas.finish(dist)
    return 0


def kernel_name(N: int) -> str:
    """The kernel the library dispatches for W4A4 64x64 tiles at N tokens."""
    if N <= 7:
        return f"w4a4_sk_kernel<{N},0>"             # dp4a consumer
    if N <= 32:
        nt = 1 if N <= 8 else (2 if N <= 16 else 4)
        return f"w4a4_sk_kernel<{8 * nt},{nt}>"      # mma.sync consumer, 8-token blocks
    return "spmm_generic_kernel<I4,64>"


KERNEL_SOURCES = {"w4a4_sk_kernel": ("us_w4a4_sk.cuh", "us_w4a4_sk.cu"),
                  "w4a4_small_n_kernel": ("us_w4a4.cu",), "spmm_generic_kernel": ("us_spmm.cu",)}


def kernel_source_sha(kernel: str):
    """sha256 over the kernel's source files and the shared device header."""
    import hashlib
    srcs = KERNEL_SOURCES.get(kernel.split("<")[0])
    if not srcs:
        return None
    h = hashlib.sha256()
    for f in (*srcs, "us_common.cuh"):
        with open(os.path.join(ROOT, "bitmap_encoded_unstructured_ie_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def load_traffic(kernel: str):
    """Per-launch DRAM bytes of this kernel from the committed ncu summary, if
    it was taken on the current kernel source (else null)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        ent = d.get(kernel)
        if not ent or ent.get("source_sha256") != kernel_source_sha(kernel):
            return None
        return ent.get("dram_bytes_per_launch")
    except Exception:
        return None


def measure_e2e(us, torch, wl, d, copies, sw, dev, stream, args, L):
    """Same metric through the C ABI with host buffers: every step copies each
    N's activations from pinned host memory and every output back to pinned
    host memory, inside the timed region (captured with the launches).  Each
    launch writes its own slice of one device output buffer per N, read back in
    one copy after that N's launches (per-launch copies of ~100 KB cost more in
    copy set-up than in bytes, and would break the launches' overlap)."""
    steps = max(3, min(args.steps, 20))
    hX, hY, dX, dSX, dYacc, dY, ws = {}, {}, {}, {}, {}, {}, {}
    h2d = d2h = 0
    for N in NS:
        px = torch.from_numpy(wl.pack_int4(d["Xq"][:N])).pin_memory()
        hX[N] = px
        dX[N] = torch.empty_like(px, device=dev)
        dSX[N] = torch.from_numpy(d["s_x"][:N].view(np.int16)).to(dev)
        dYacc[N] = torch.empty(N, M_, dtype=torch.int32, device=dev)
        dY[N] = torch.empty(L, N, M_, dtype=torch.int16, device=dev)
        hY[N] = torch.empty(L, N, M_, dtype=torch.int16).pin_memory()
        ws[N] = us.workspace(us.US_OP_SPMM_W4A4, copies[0], N)
        h2d += px.numel()
        d2h += L * N * M_ * 2

    def step():
        for N in NS:
            dX[N].copy_(hX[N], non_blocking=True)
            for i, E in enumerate(copies):
                us.us_spmm_w4a4(E, dX[N], sw, dSX[N], N, dYacc[N], dY[N][i], ws[N], 0, stream)
            hY[N].copy_(dY[N], non_blocking=True)

    with torch.cuda.stream(stream):
        step()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    with torch.cuda.stream(stream):        # replays run on the current stream
        for _ in range(3):
            g.replay()
    stream.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(steps):
            g.replay()
        b.record(stream)
    stream.synchronize()
    assert us.us_get_last_device_status(stream) == us.US_OK
    ms = a.elapsed_time(b) / steps
    bytes_step = sum(call_bytes(copies[0].values_bytes, M_, K_, N, TM_, TK_) for N in NS) * L
    return {"value": round(bytes_step / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 4), "_bytes_per_step": bytes_step,
            "how": "CUDA graph of the C-ABI calls with pinned-host H2D of X and D2H of every fp16 output "
                   "(one copy per N per step)"}


def time_graph(torch, stream, us, fn, reps=5):
    """Mean device time (ms) of one replay of a CUDA graph of fn(), captured and
    replayed on `stream`; the library's device status must stay clean."""
    with torch.cuda.stream(stream):
        fn()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    with torch.cuda.stream(stream):        # replays run on the current stream
        g.replay()
    stream.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
    stream.synchronize()
    assert us.us_get_last_device_status(stream) == us.US_OK
    return a.elapsed_time(b) / reps


def oracle_ms(fn, min_s: float = 0.25, max_reps: int = 20) -> float:
    """Mean wall time (ms) of one oracle call, repeated for at least min_s."""
    reps, el = 0, 0.0
    while reps == 0 or (el < min_s and reps < max_reps):
        t0 = time.perf_counter()
        fn()
        el += time.perf_counter() - t0
        reps += 1
    return el / reps * 1e3


class OracleRows:
    """The CPU oracle's time for one call of a configuration, measured on the
    first `bands` tile-row bands of the encoded matrix (decode + multiply of
    that shard) and scaled to the whole matrix by the band count."""

    def __init__(self):
        from oracle import oracle as orc
        from bitmap_encoded_unstructured_ie_gb300 import sharding
        self.orc, self.sharding = orc, sharding
        self.threads = orc.max_threads()

    def w4a4(self, Wq, Xq, s_w, s_x, bands: int):
        orc = self.orc
        M, K = Wq.shape
        enc = orc.encode(Wq, 64, 64, orc.I4, orc.ROW)
        bands = min(bands, M // 64)
        bm, off, vals, Ms = self.sharding.shard_arrays(*enc, M, K, 64, 64, orc.I4, 0, bands)

        def call():
            Wd = orc.decode(bm, off, vals, Ms, K, 64, 64, orc.I4, orc.ROW)
            orc.spmm_w4a4(Wd, Xq, s_w[:Ms], s_x, nthreads=self.threads)
        return self._row(oracle_ms(call) * (M // 64) / bands, bands, M // 64)

    def f16(self, W, X, order: int, bands: int):
        orc = self.orc
        M, K = W.shape
        enc = orc.encode(W, 64, 64, orc.F16, order)
        bands = min(bands, M // 64)
        bm, off, vals, Ms = self.sharding.shard_arrays(*enc, M, K, 64, 64, orc.F16, 0, bands)

        def call():
            Wd = orc.decode(bm, off, vals, Ms, K, 64, 64, orc.F16, order)
            orc.spmm_f16(Wd, X, nthreads=self.threads)
        return self._row(oracle_ms(call) * (M // 64) / bands, bands, M // 64)

    def spmspv(self, W, x, bands: int):
        orc = self.orc
        M, K = W.shape
        enc = orc.encode(W, 64, 64, orc.F16, orc.COL)
        bands = min(bands, M // 64)
        bm, off, vals, Ms = self.sharding.shard_arrays(*enc, M, K, 64, 64, orc.F16, 0, bands)

        def call():
            Wd = orc.decode(bm, off, vals, Ms, K, 64, 64, orc.F16, orc.COL)
            orc.spmspv_f16(Wd, x, 0.0, nthreads=self.threads)
        return self._row(oracle_ms(call) * (M // 64) / bands, bands, M // 64)

    def _row(self, ms, bands, total):
        return {"us_per_call": round(ms * 1e3, 1), "cores": self.threads, "kind": "oracle",
                "sample": f"decode + multiply of {bands} of {total} tile-row bands, scaled"}


def pct(gbs: float, peak: float) -> float:
    return round(100.0 * gbs / peak, 2)


def tensor_peaks(torch, dev):
    """Dense int8 tensor throughput of this GPU (cuBLAS through torch._int_mm,
    8192^3, best of 5), the denominator for an int8 tensor path."""
    try:
        a = torch.randint(-8, 8, (8192, 8192), dtype=torch.int8, device=dev)
        b = torch.randint(-8, 8, (8192, 8192), dtype=torch.int8, device=dev)
        torch._int_mm(a, b)
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(5):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            torch._int_mm(a, b)
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        return {"int8_dense_TOPS": round(2 * 8192 ** 3 / (best * 1e-3) / 1e12, 1),
                "how": "torch._int_mm (cuBLAS) int8 x int8 -> int32, 8192^3, best of 5, CUDA events"}
    except Exception as e:                            # noqa: BLE001
        return {"int8_dense_TOPS": None, "error": f"{type(e).__name__}: {e}"}


def measure_extras(us, torch, wl, dev, stream, hbm_peak, bf16_peak, cpu=True):
    """Secondary rows, each timed on its own: every configuration besides the
    headline (fp16 256 x 512, W4A4 4096^2 at 30 and 70 % sparsity, the FFN
    shapes, fp16 prefill and decode, spMspV), the encoder, W2A4, IE-BME areas,
    the activation quantiser.  Copies rotate so every launch reads from HBM.
    Each row gives its % of the measured HBM (or fp16 tensor) peak and, where
    `cpu`, the oracle's time for the same call."""
    out = {}
    l2 = 126 * 2 ** 20
    ocpu = OracleRows() if cpu else None
    out["tensor_peaks"] = tensor_peaks(torch, dev)
    # fp16 bitmap SpMM 256 x 512, 50 % uniform sparsity, N = 1 (latency row):
    # enough rotating copies that the chain streams more than twice L2
    c1 = wl.f16_spmm(256, 512, 1, 0.5, seed=0)
    E1 = us.us_encode(torch.from_numpy(c1["W"].view(np.int16)).to(dev), 64, 64, us.US_F16, us.US_ORDER_ROW)
    E1.flags = us.US_BITMAP_STATIC
    n1 = max(4, math.ceil(2.2 * l2 / E1.nbytes()))
    cp1 = [E1] + [us.Encoded(E1.M, E1.K, E1.TM, E1.TK, E1.elem, E1.order, E1.bitmap.clone(), E1.tile_off.clone(),
                             E1.values.clone(), E1.values_bytes, E1.flags) for _ in range(n1 - 1)]
    X1 = torch.from_numpy(c1["X"].view(np.int16)).to(dev)
    Y1 = torch.empty(1, 256, dtype=torch.int16, device=dev)
    ws1 = us.workspace(us.US_OP_SPMM_F16, E1, 1)
    ms = time_graph(torch, stream, us, lambda: [us.us_spmm_f16(E, X1, 1, Y1, ws1, 0, stream) for E in cp1], 3)
    t = ms * 1e3 / n1
    b1 = E1.nbytes() + 512 * 2 + 256 * 2
    out["f16_256x512_s50_n1"] = {"us_per_call": round(t, 3), "bytes": b1, "GB/s": round(b1 / (t * 1e-6) / 1e9, 1),
                                 "pct_hbm_measured": pct(b1 / (t * 1e-6) / 1e9, hbm_peak), "copies": n1,
                                 "cpu_oracle": ocpu.f16(c1["W"], c1["X"], 0, 4) if ocpu else None}
    # W4A4 4096^2 at 30 % and 70 % sparsity (the headline is 50 %), N = 1 / 8 / 16
    spars = {}
    for sp_ in (0.3, 0.7):
        ds = wl.w4a4(4096, 4096, 16, sp_, seed=0)
        Es = us.us_encode(torch.from_numpy(ds["Wq"]).to(dev), 64, 64, us.US_I4, us.US_ORDER_ROW)
        Es.flags = us.US_BITMAP_STATIC
        ns_ = max(4, math.ceil(2.2 * l2 / Es.nbytes()))
        cps_ = [Es] + [us.Encoded(Es.M, Es.K, Es.TM, Es.TK, Es.elem, Es.order, Es.bitmap.clone(), Es.tile_off.clone(),
                                  Es.values.clone(), Es.values_bytes, Es.flags) for _ in range(ns_ - 1)]
        sws = torch.from_numpy(ds["s_w"].view(np.int16)).to(dev)
        row = {"copies": ns_, "value_bytes": Es.values_bytes}
        for N in NS:
            Xs = torch.from_numpy(wl.pack_int4(ds["Xq"][:N])).to(dev)
            sxs = torch.from_numpy(ds["s_x"][:N].view(np.int16)).to(dev)
            Yas = torch.empty(N, 4096, dtype=torch.int32, device=dev)
            Yhs = torch.empty(N, 4096, dtype=torch.int16, device=dev)
            wss = us.workspace(us.US_OP_SPMM_W4A4, Es, N)
            ms = time_graph(torch, stream, us, lambda: [us.us_spmm_w4a4(E, Xs, sws, sxs, N, Yas, Yhs, wss, 0, stream)
                                                    for E in cps_], 20)
            t = ms * 1e3 / ns_
            bs = call_bytes(Es.values_bytes, 4096, 4096, N, 64, 64)
            gbs = bs / (t * 1e-6) / 1e9
            row[f"N{N}"] = {"us_per_launch": round(t, 3), "bytes_per_call": bs, "GB/s": round(gbs, 1),
                            "pct_hbm_measured": pct(gbs, hbm_peak),
                            "eff_TOPS": round(2 * 4096 * 4096 * N / (t * 1e-6) / 1e12, 2),
                            "cpu_oracle": ocpu.w4a4(ds["Wq"], ds["Xq"][:N], ds["s_w"], ds["s_x"][:N], 8)
                            if ocpu else None}
        spars[f"s{int(sp_ * 100)}"] = row
    out["w4a4_4096_sparsity"] = spars
    # spMspV 14336 x 4096, 50 % static sparsity, activations with 50/70/90 % zeros
    s = wl.spmspv(14336, 4096, 0.5, 0.5, seed=0)
    Es = us.us_encode(torch.from_numpy(s["W"].view(np.int16)).to(dev), 64, 64, us.US_F16, us.US_ORDER_COL)
    n_cp = max(2, math.ceil(2.2 * l2 / Es.nbytes()))
    cps = [Es] + [us.Encoded(Es.M, Es.K, Es.TM, Es.TK, Es.elem, Es.order, Es.bitmap.clone(), Es.tile_off.clone(),
                             Es.values.clone(), Es.values_bytes) for _ in range(n_cp - 1)]
    wsb = us.workspace(us.US_OP_SPMSPV_F16, Es, 1)
    ys = torch.empty(14336, dtype=torch.int16, device=dev)
    rng = np.random.default_rng(2)
    sp = {}
    Wnz = (s["W"].view(np.uint16) & 0x7FFF) != 0
    for zf in (0.5, 0.7, 0.9):
        x = wl.relu_threshold(rng.standard_normal(4096).astype(np.float32), zf).astype(np.float16)
        xt = torch.from_numpy(x.view(np.int16)).to(dev)
        active = np.abs(x.astype(np.float32)) > 0
        act_vals = int(Wnz[:, active].sum()) * 2
        nT = (14336 // 64) * (4096 // 64)
        alg = 14336 * 4096 // 8 + 4 * (nT + 1) + act_vals + 4096 * 2 + 14336 * 2
        ms = time_graph(torch, stream, us, lambda: [us.us_spmspv_f16(E, xt, 0.0, ys, wsb, stream) for E in cps])
        t = ms * 1e3 / n_cp
        sp[f"zeros_{int(zf * 100)}"] = {"us_per_launch": round(t, 3), "alg_bytes": alg,
                                        "GB/s": round(alg / (t * 1e-6) / 1e9, 1),
                                        "pct_hbm_measured": pct(alg / (t * 1e-6) / 1e9, hbm_peak),
                                        "cpu_oracle": ocpu.spmspv(s["W"], x, 8) if ocpu else None}
    out["spmspv_f16_14336x4096"] = sp
    # the same with ColInfo (per tile column: offset and count), N = 1 and a batch of 8
    cis = [us.us_colinfo(E, None, stream) for E in cps]
    stream.synchronize()
    nTM_s = 14336 // 64
    sci = {}
    for zf, N in ((0.5, 1), (0.7, 1), (0.9, 1), (0.9, 8), (0.7, 8)):
        X = np.stack([wl.relu_threshold(rng.standard_normal(4096).astype(np.float32), zf) for _ in range(N)])
        X = X.astype(np.float16)
        Xt = torch.from_numpy(X.view(np.int16)).to(dev)
        Yt = torch.empty(N, 14336, dtype=torch.int16, device=dev)
        active = (np.abs(X.astype(np.float32)) > 0).any(axis=0)
        alg = (4 * nTM_s * 4096 + 4 * (nTM_s * 64 + 1) + nTM_s * int(active.sum()) * 8 +
               int(Wnz[:, active].sum()) * 2 + N * 4096 * 2 + N * 14336 * 2)
        ms = time_graph(torch, stream, us,
                        lambda: [us.us_spmspv_f16_ci(E, c, Xt, N, 0.0, Yt, None, stream) for E, c in zip(cps, cis)])
        t = ms * 1e3 / n_cp
        sci[f"zeros_{int(zf * 100)}_N{N}"] = {"us_per_launch": round(t, 3), "alg_bytes": alg,
                                              "active_columns": round(float(active.mean()), 3),
                                              "GB/s": round(alg / (t * 1e-6) / 1e9, 1),
                                              "pct_hbm_measured": pct(alg / (t * 1e-6) / 1e9, hbm_peak)}
    out["spmspv_colinfo_f16_14336x4096"] = sci
    # encoder, W4A4 4096^2 (dense int8 codes in): count + scan + pack
    d = wl.w4a4(4096, 4096, 1, 0.5, seed=0)
    Wd = torch.from_numpy(d["Wq"]).to(dev)
    Ee = us.us_encode(Wd, 64, 64, us.US_I4, us.US_ORDER_ROW, None, False)
    wse = torch.zeros(us.encode_sizes(4096, 4096, 64, 64, us.US_I4)[3], dtype=torch.uint8, device=dev)
    ms = time_graph(torch, stream, us, lambda: us.us_encode_into(Wd, Ee, wse, stream), 5)
    out["encode_w4a4_4096"] = {"ms_per_encode": round(ms, 4),
                               "dense_GB/s": round(4096 * 4096 / (ms * 1e-3) / 1e9, 1),
                               "pct_hbm_measured": pct(4096 * 4096 / (ms * 1e-3) / 1e9, hbm_peak)}
    # fp16 prefill 4096^2, 60 % sparsity, N = 256 / 1024 / 2048
    f = wl.f16_spmm(4096, 4096, 2048, 0.6, seed=0)
    Ef = us.us_encode(torch.from_numpy(f["W"].view(np.int16)).to(dev), 64, 64, us.US_F16, us.US_ORDER_ROW)
    Xf = torch.from_numpy(f["X"].view(np.int16)).to(dev)
    pf = {}
    for N in (256, 1024, 2048):
        Yf = torch.empty(N, 4096, dtype=torch.int16, device=dev)
        wsf = us.workspace(us.US_OP_SPMM_F16, Ef, N)
        ms = time_graph(torch, stream, us, lambda: us.us_spmm_f16(Ef, Xf[:N], N, Yf, wsf, 0, stream), 3)
        fl = 2 * 4096 * 4096 * N
        tf = fl / (ms * 1e-3) / 1e12
        pf[str(N)] = {"ms": round(ms, 4), "eff_TFLOPs": round(tf, 2), "pct_f16_tensor_measured": pct(tf, bf16_peak),
                      "cpu_oracle": ocpu.f16(f["W"], f["X"][:N], 0, 1) if ocpu else None}
    out["prefill_f16_4096_s60"] = pf
    # fp16 decode 4096^2, 50 % sparsity, N = 1 / 8 / 16 / 32 (mma.sync decode
    # kernel); rotating weight copies so every launch reads from HBM
    fd = wl.f16_spmm(4096, 4096, 32, 0.5, seed=1)
    Eg = us.us_encode(torch.from_numpy(fd["W"].view(np.int16)).to(dev), 64, 64, us.US_F16, us.US_ORDER_ROW)
    ng = max(2, math.ceil(2.2 * l2 / Eg.nbytes()))
    cpg = [Eg] + [us.Encoded(Eg.M, Eg.K, Eg.TM, Eg.TK, Eg.elem, Eg.order, Eg.bitmap.clone(), Eg.tile_off.clone(),
                             Eg.values.clone(), Eg.values_bytes) for _ in range(ng - 1)]
    Xg = torch.from_numpy(fd["X"].view(np.int16)).to(dev)
    dec = {"copies": ng}
    for N in (1, 8, 16, 32):
        Yg = torch.empty(N, 4096, dtype=torch.int16, device=dev)
        wsg = us.workspace(us.US_OP_SPMM_F16, Eg, N)
        ms = time_graph(torch, stream, us, lambda: [us.us_spmm_f16(E, Xg[:N], N, Yg, wsg, 0, stream) for E in cpg])
        t = ms * 1e3 / ng
        byt = Eg.nbytes() + 2 * N * 4096 * 2
        dec[str(N)] = {"us_per_call": round(t, 3), "bytes": byt, "GB/s": round(byt / (t * 1e-6) / 1e9, 1),
                       "pct_hbm_measured": pct(byt / (t * 1e-6) / 1e9, hbm_peak),
                       "cpu_oracle": ocpu.f16(fd["W"], fd["X"][:N], 0, 8) if ocpu else None}
    out["decode_f16_4096_s50"] = dec
    # the same on COL tiles: the format spMspV reads serves prefill too
    Efc = us.us_encode(torch.from_numpy(f["W"].view(np.int16)).to(dev), 64, 64, us.US_F16, us.US_ORDER_COL)
    pfc = {}
    for N in (256, 1024, 2048):
        Yf = torch.empty(N, 4096, dtype=torch.int16, device=dev)
        wsf = us.workspace(us.US_OP_SPMM_F16, Efc, N)
        ms = time_graph(torch, stream, us, lambda: us.us_spmm_f16(Efc, Xf[:N], N, Yf, wsf, 0, stream), 3)
        fl = 2 * 4096 * 4096 * N
        tf = fl / (ms * 1e-3) / 1e12
        pfc[str(N)] = {"ms": round(ms, 4), "eff_TFLOPs": round(tf, 2), "pct_f16_tensor_measured": pct(tf, bf16_peak)}
    out["prefill_f16_col_tiles_4096_s60"] = pfc
    # the FFN shapes: W4A4 11008 x 4096 and 4096 x 11008, 50 % sparsity with a
    # per-row Beta(2,2) keep rate, N = 1 / 4 / 16 / 32, static weights
    ffn = {}
    for (Mf, Kf) in ((11008, 4096), (4096, 11008)):
        df = wl.w4a4(Mf, Kf, 32, 0.5, seed=0, rows="beta")
        Ef = us.us_encode(torch.from_numpy(df["Wq"]).to(dev), 64, 64, us.US_I4, us.US_ORDER_ROW)
        Ef.flags = us.US_BITMAP_STATIC
        nf = max(4, math.ceil(2.2 * l2 / Ef.nbytes()))
        cpf = [Ef] + [us.Encoded(Ef.M, Ef.K, Ef.TM, Ef.TK, Ef.elem, Ef.order, Ef.bitmap.clone(), Ef.tile_off.clone(),
                                 Ef.values.clone(), Ef.values_bytes, Ef.flags) for _ in range(nf - 1)]
        swf = torch.from_numpy(df["s_w"].view(np.int16)).to(dev)
        row = {"copies": nf}
        for N in (1, 4, 16, 32):
            Xf_ = torch.from_numpy(wl.pack_int4(df["Xq"][:N])).to(dev)
            sxf = torch.from_numpy(df["s_x"][:N].view(np.int16)).to(dev)
            Yaf = torch.empty(N, Mf, dtype=torch.int32, device=dev)
            Yhf = torch.empty(N, Mf, dtype=torch.int16, device=dev)
            wsf_ = us.workspace(us.US_OP_SPMM_W4A4, Ef, N)
            ms = time_graph(torch, stream, us, lambda: [us.us_spmm_w4a4(E, Xf_, swf, sxf, N, Yaf, Yhf, wsf_, 0, stream)
                                                    for E in cpf], 10)
            t = ms * 1e3 / nf
            bf = call_bytes(Ef.values_bytes, Mf, Kf, N, 64, 64)
            row[f"N{N}"] = {"us_per_launch": round(t, 3), "bytes_per_call": bf, "GB/s": round(bf / (t * 1e-6) / 1e9, 1),
                            "pct_hbm_measured": pct(bf / (t * 1e-6) / 1e9, hbm_peak),
                            "eff_TOPS": round(2 * Mf * Kf * N / (t * 1e-6) / 1e12, 2),
                            "cpu_oracle": ocpu.w4a4(df["Wq"], df["Xq"][:N], df["s_w"], df["s_x"][:N], 4)
                            if ocpu else None}
        ffn[f"{Mf}x{Kf}"] = row
    out["w4a4_ffn_beta_s50"] = ffn
    # W2A4 4096^2 at 50 %: int2 weights decoded into the same dense tiles
    d2 = wl.w2a4(4096, 4096, 16, 0.5, seed=0)
    E2 = us.us_encode(torch.from_numpy(d2["Wq"]).to(dev), 64, 64, us.US_I2, us.US_ORDER_ROW)
    E2.flags = us.US_BITMAP_STATIC
    n2 = max(4, math.ceil(2.2 * l2 / E2.nbytes()))
    cps2 = [E2] + [us.Encoded(E2.M, E2.K, E2.TM, E2.TK, E2.elem, E2.order, E2.bitmap.clone(), E2.tile_off.clone(),
                              E2.values.clone(), E2.values_bytes, E2.flags) for _ in range(n2 - 1)]
    sw2 = torch.from_numpy(d2["s_w"].view(np.int16)).to(dev)
    w2 = {"copies": n2, "value_bytes": E2.values_bytes}
    for N in (1, 8, 16):
        X2 = torch.from_numpy(wl.pack_int4(d2["Xq"][:N])).to(dev)
        sx2 = torch.from_numpy(d2["s_x"][:N].view(np.int16)).to(dev)
        Ya2 = torch.empty(N, 4096, dtype=torch.int32, device=dev)
        Yh2 = torch.empty(N, 4096, dtype=torch.int16, device=dev)
        ws2 = us.workspace(us.US_OP_SPMM_W4A4, E2, N)
        ms = time_graph(torch, stream, us, lambda: [us.us_spmm_w4a4(E, X2, sw2, sx2, N, Ya2, Yh2, ws2, 0, stream)
                                                for E in cps2], 20)
        t = ms * 1e3 / n2
        b2 = call_bytes(E2.values_bytes, 4096, 4096, N, 64, 64)
        w2[f"N{N}"] = {"us_per_launch": round(t, 3), "bytes_per_call": b2, "GB/s": round(b2 / (t * 1e-6) / 1e9, 1),
                       "pct_hbm_measured": pct(b2 / (t * 1e-6) / 1e9, hbm_peak)}
    out["w2a4_4096_s50"] = w2
    # IE-BME with areas: W4A4 4096^2 at 50 %, 16 x 64 local tiles, 2 x 2 areas, with
    # and without the offline row reordering; encoded bytes and the SpMM time
    d = wl.w4a4(4096, 4096, 16, 0.5, seed=0)
    Wq = torch.from_numpy(d["Wq"]).to(dev)
    ie = {}
    E1 = us.us_encode(Wq, 64, 64, us.US_I4, us.US_ORDER_ROW)
    ie["plain_64x64"] = {"bitmap_bytes": E1.bitmap.numel() * 8, "value_bytes": E1.values_bytes,
                         "total_bytes": E1.nbytes()}
    import time as _t
    t_re = _t.time()
    perm = us.us_reorder_rows(d["Wq"], 16, 64, 2, 2, us.US_I4)
    reorder_s = _t.time() - t_re
    permt = torch.from_numpy(perm).to(dev)
    swi = torch.from_numpy(d["s_w"].view(np.int16)).to(dev)
    for name, pm in (("areas_2x2_16x64", None), ("areas_2x2_16x64_reordered", permt)):
        Ei = us.us_encode_ie(Wq, 16, 64, 2, 2, us.US_I4, pm)
        Ei.E.flags = us.US_BITMAP_STATIC
        pbytes = 0 if pm is None else pm.numel()
        wbytes = Ei.E.nbytes() + pbytes
        ni = max(2, math.ceil(2.2 * l2 / wbytes))      # rotating copies: every launch reads from HBM
        cpi = [Ei] + [us.EncodedIE(us.Encoded(Ei.E.M, Ei.E.K, 16, 64, Ei.E.elem, Ei.E.order, Ei.E.bitmap.clone(),
                                              Ei.E.tile_off.clone(), Ei.E.values.clone(), Ei.E.values_bytes,
                                              us.US_BITMAP_STATIC), 2, 2, None if pm is None else pm.clone())
                      for _ in range(ni - 1)]
        row = {"bitmap_bytes": Ei.E.bitmap.numel() * 8, "value_bytes": Ei.E.values_bytes, "perm_bytes": pbytes,
               "total_bytes": wbytes, "copies": ni,
               "kernel": "balanced" if us.us_pick_split_k_ie(Ei, 1) == 0 else "generic"}
        for N in (1, 8, 16):
            X = torch.from_numpy(wl.pack_int4(d["Xq"][:N])).to(dev)
            sxi = torch.from_numpy(d["s_x"][:N].view(np.int16)).to(dev)
            Ya = torch.empty(N, 4096, dtype=torch.int32, device=dev)
            Yh = torch.empty(N, 4096, dtype=torch.int16, device=dev)
            wsi = us.workspace_ie(Ei, N)
            ms = time_graph(torch, stream, us, lambda: [us.us_spmm_w4a4_ie(E, X, swi, sxi, N, Ya, Yh, wsi, 0, stream)
                                                    for E in cpi], 10)
            t = ms * 1e3 / ni
            b = wbytes + N * 4096 // 2 + 2 * (4096 + N) + N * 4096 * 6       # weights, X, scales, Yacc + Y
            row[f"N{N}"] = {"us_per_launch": round(t, 3), "bytes_per_call": b, "GB/s": round(b / (t * 1e-6) / 1e9, 1),
                            "pct_hbm_measured": pct(b / (t * 1e-6) / 1e9, hbm_peak)}
        # the generic CUDA-core kernel on the same matrix (split_k = 1), N = 1
        X = torch.from_numpy(wl.pack_int4(d["Xq"][:1])).to(dev)
        Ya = torch.empty(1, 4096, dtype=torch.int32, device=dev)
        wsg = us.workspace_ie(Ei, 1, 1)
        ms = time_graph(torch, stream, us, lambda: us.us_spmm_w4a4_ie(Ei, X, None, None, 1, Ya, None, wsg, 1, stream), 5)
        row["generic_N1_us"] = round(ms * 1e3, 2)
        ie[name] = row
    ie["reorder_host_s"] = round(reorder_s, 2)
    out["w4a4_ie_areas_4096"] = ie
    # rows that share sparsity patterns (groups of four with common column
    # scales before pruning, shuffled within each 16-row block) at 70 %:
    # plain 64 x 64 tiles against IE-BME 4 x 1 areas with the row reordering
    dc = wl.w4a4(4096, 4096, 16, 0.7, seed=0, rows="clustered")
    Wc = torch.from_numpy(dc["Wq"]).to(dev)
    swc = torch.from_numpy(dc["s_w"].view(np.int16)).to(dev)
    cl = {}
    Ep = us.us_encode(Wc, 64, 64, us.US_I4, us.US_ORDER_ROW)
    Ep.flags = us.US_BITMAP_STATIC
    permc = torch.from_numpy(us.us_reorder_rows(dc["Wq"], 16, 64, 4, 1, us.US_I4)).to(dev)
    Ec = us.us_encode_ie(Wc, 16, 64, 4, 1, us.US_I4, permc)
    Ec.E.flags = us.US_BITMAP_STATIC
    for name, E0, wb in (("plain_64x64", Ep, Ep.nbytes()), ("areas_4x1_16x64_reordered", Ec, Ec.E.nbytes() + permc.numel())):
        n0 = max(2, math.ceil(2.2 * l2 / wb))
        if name == "plain_64x64":
            cps0 = [E0] + [us.Encoded(E0.M, E0.K, 64, 64, E0.elem, E0.order, E0.bitmap.clone(), E0.tile_off.clone(),
                                      E0.values.clone(), E0.values_bytes, us.US_BITMAP_STATIC) for _ in range(n0 - 1)]
        else:
            cps0 = [E0] + [us.EncodedIE(us.Encoded(E0.E.M, E0.E.K, 16, 64, E0.E.elem, E0.E.order, E0.E.bitmap.clone(),
                                                   E0.E.tile_off.clone(), E0.E.values.clone(), E0.E.values_bytes,
                                                   us.US_BITMAP_STATIC), 4, 1, permc.clone()) for _ in range(n0 - 1)]
        row = {"weight_bytes": wb, "copies": n0}
        for N in (1, 16):
            X = torch.from_numpy(wl.pack_int4(dc["Xq"][:N])).to(dev)
            sxc = torch.from_numpy(dc["s_x"][:N].view(np.int16)).to(dev)
            Ya = torch.empty(N, 4096, dtype=torch.int32, device=dev)
            Yh = torch.empty(N, 4096, dtype=torch.int16, device=dev)
            if name == "plain_64x64":
                wsc = us.workspace(us.US_OP_SPMM_W4A4, E0, N)
                fn = lambda: [us.us_spmm_w4a4(E, X, swc, sxc, N, Ya, Yh, wsc, 0, stream) for E in cps0]
            else:
                wsc = us.workspace_ie(E0, N)
                fn = lambda: [us.us_spmm_w4a4_ie(E, X, swc, sxc, N, Ya, Yh, wsc, 0, stream) for E in cps0]
            ms = time_graph(torch, stream, us, fn, 10)
            t = ms * 1e3 / n0
            b = wb + N * 4096 // 2 + 2 * (4096 + N) + N * 4096 * 6
            row[f"N{N}"] = {"us_per_launch": round(t, 3), "bytes_per_call": b, "GB/s": round(b / (t * 1e-6) / 1e9, 1)}
        cl[name] = row
    out["w4a4_clustered_rows_4096_s70"] = cl
    # per-token activation quantisation, fp16 -> int4 + scale (reads 2NK, writes NK/2 + 2N bytes)
    qz = {}
    for N in (16, 2048):
        Xh = torch.from_numpy(np.random.default_rng(4).standard_normal((N, 4096)).astype(np.float16).view(np.int16)).to(dev)
        Xq = torch.empty(N, 2048, dtype=torch.uint8, device=dev)
        sq = torch.empty(N, dtype=torch.int16, device=dev)
        ms = time_graph(torch, stream, us, lambda: us.us_quantize_x(Xh, N, 4096, Xq, sq, stream), 20)
        byt = N * 4096 * 2 + N * 2048 + N * 2
        qz[str(N)] = {"us": round(ms * 1e3, 2), "GB/s": round(byt / (ms * 1e-3) / 1e9, 1),
                      "pct_hbm_measured": pct(byt / (ms * 1e-3) / 1e9, hbm_peak)}
    out["quantize_x_k4096"] = qz
    return out


if __name__ == "__main__":
    sys.exit(main())
