"""Benchmark of the W4A16 group-quantized linear layer on GB300.

One step = one decode pass of a 27B-class dense MLP through the layer:
x [1, 5120] -> gate/up projection (K=5120 -> N=17408, group 128) -> h [1, 17408]
-> down projection (K=17408 -> N=5120) -> out [1, 5120]; both are decode GEMVs.
The headline metric is the achieved HBM bandwidth of that step: algorithmic
bytes (every packed weight, scale, activation and output byte once) divided by
device time. Weights rotate through enough copies (> 4x the L2 size) that
every step streams them from HBM.

Side measurements in the same JSON line: the batched decode (M=4), the
prefill GEMM (M=4096, K=5120, N=17408; TFLOP/s) and the routed-expert layer
(E=128, 4096 tokens, top-8, group 32), when the library provides them.

The timed step makes the plain calls. The same step with the weights
declared static (W4A16_STATIC_WEIGHTS: each GEMV streams its weights before
the one ahead of it has finished) is reported beside it.

--impl reference times the CPU oracle (fp64, single thread) on the same
workload and metric. With --gpus N > 1 (torchrun), every rank runs an
independent replica (the layer needs no collective), timing is the max over
ranks and the value is the sum over ranks (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

DECODE = [(5120, 17408), (17408, 5120)]  # (K, N): gate/up then down
GROUP = 128


def decode_bytes(M: int) -> int:
    """Algorithmic bytes of one decode step: packed weights, scales, x and y once."""
    total = 0
    for K, N in DECODE:
        total += N * K // 2 + N * (K // GROUP) * 2 + M * K * 2 + M * N * 2
    return total


def moe_bytes(E, R, K, N, g):
    return E * N * K // 2 + E * N * (K // g) * 2 + R * K * 2 + R * N * 2


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [v.strip() for v in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- host records --

def host_info():
    """CPU model and logical core count of the machine the bench runs on."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    return {"cpu_model": model or platform.processor() or platform.machine(), "nproc": os.cpu_count(),
            "arch": platform.machine()}


def source_info():
    """The git commit when the tree has one, and a hash of the sources that run."""
    rev = None
    try:
        r = subprocess.run(["git", "-C", ROOT, "rev-parse", "HEAD"], capture_output=True, text=True, timeout=10)
        rev = r.stdout.strip() or None if r.returncode == 0 else None
    except (OSError, subprocess.SubprocessError):
        pass
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "w4a16_group_quantized_linear_gb300", "csrc")
    for name in sorted(os.listdir(csrc)) + ["../../include/w4a16.h", "../../bench.py"]:
        try:
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
        except OSError:
            pass
    return {"git": rev, "sources_sha256": h.hexdigest()[:16]}


def gpu_software(torch):
    drv = None
    try:
        drv = subprocess.run(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=10).stdout.strip().splitlines()[0]
    except (OSError, subprocess.SubprocessError, IndexError):
        pass
    return {"driver": drv, "cuda": torch.version.cuda, "torch": torch.__version__}


# ------------------------------------------------------------------ GPU arm --

def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


def max_over_ranks(ms: float, device, world: int) -> float:
    """The slowest rank's time (replicas run the same work; the job ends with the last)."""
    if world <= 1:
        return ms
    import torch

    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, ms_max: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return units_per_rank * world / (ms_max * 1e-3)


class Timer:
    """CUDA-event pairs around launches on the launching stream."""

    def __init__(self, torch):
        self.torch = torch
        self.pairs = []

    def around(self, fn):
        s = self.torch.cuda.Event(enable_timing=True)
        e = self.torch.cuda.Event(enable_timing=True)
        s.record()
        fn()
        e.record()
        self.pairs.append((s, e))

    def ms(self):
        return [s.elapsed_time(e) for s, e in self.pairs]


def run_gpu(args, rank, world):
    import torch

    import w4a16_group_quantized_linear_gb300 as w4

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w4.lib()
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20)
    hbm_peak, tc_peak, peak_kind = _peaks()

    # ---- weights: packed on the GPU by the library's quantizer, rotated copies
    M = 1
    step_bytes = decode_bytes(M)
    copies = max(2, -(-4 * l2 // (step_bytes - 2 * 10240)))
    g = workloads.rng(0)
    mats = []
    for K, N in DECODE:
        W = torch.from_numpy(workloads.weights(g, N, K)).to(dev)
        qw, s = w4.pack(W, GROUP)
        del W
        mats.append((qw, s))
    rot = [[(m[0].clone(), m[1].clone()) for m in mats] for _ in range(copies)]
    x = torch.from_numpy(workloads.activations(g, M, DECODE[0][0])).to(dev)
    h = torch.empty((M, DECODE[0][1]), dtype=torch.float16, device=dev)
    out = torch.empty((M, DECODE[1][1]), dtype=torch.float16, device=dev)

    def step(i, static=False):
        (qa, sa), (qb, sb) = rot[i % copies]
        w4.linear(x, qa, sa, GROUP, out=h, static_weights=static)
        w4.linear(h, qb, sb, GROUP, out=out, static_weights=static)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    w4.device_status()

    # ---- timed region: launches queued behind a spin so the GPU runs them back to
    # back (consecutive GEMVs overlap through programmatic dependent launch); CUDA
    # events only at the two ends, on the launching stream
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clocks:
        torch.cuda._sleep(int(1e7 + args.steps * 2e5))
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for i in range(args.steps):
            step(i)
        t1.record()
        torch.cuda.synchronize()
    ms_local = t0.elapsed_time(t1)
    ms_total = max_over_ranks(ms_local, dev, world)
    kernel_ms = ms_local / (2 * args.steps)  # mean GEMV launch duration in the stream
    per_launch_bytes = step_bytes / 2  # both GEMVs move the same algorithmic bytes
    achieved = per_launch_bytes / (kernel_ms * 1e-3) / 1e9
    value = job_throughput(step_bytes * args.steps, world, ms_total) / 1e9

    # ---- spread per call: 10 back-to-back regions of 20 steps each (CUDA events at the
    # two ends of every region); median and p95 of the per-GEMV mean, both modes
    def per_call(static):
        samples = []
        for rep_ in range(10):
            torch.cuda.synchronize()
            torch.cuda._sleep(int(2e6))
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            for i in range(20):
                step(rep_ * 20 + i, static)
            b.record()
            torch.cuda.synchronize()
            samples.append(a.elapsed_time(b) * 1e3 / 40)
        samples.sort()
        return {"median_us": statistics.median(samples), "p95_us": samples[int(0.95 * (len(samples) - 1) + 0.5)],
                "samples": len(samples), "how": "10 regions x 20 back-to-back steps (40 GEMVs), mean per GEMV each"}

    spread = per_call(False)
    static_mode = per_call(True)
    static_mode["GB/s"] = per_launch_bytes / (static_mode["median_us"] * 1e-6) / 1e9
    static_mode["frac_hbm"] = static_mode["GB/s"] / hbm_peak
    w4.device_status()

    # ---- end to end through the public API: pinned host x in, host result out.
    # A decode loop replays its step as a CUDA graph: the step (x copied in, the
    # two layers, the second writing the result into host memory) is captured
    # once per weight copy. If capture fails the same calls run eagerly, and the
    # line says so.
    xh = torch.from_numpy(workloads.activations(workloads.rng(1), M, DECODE[0][0])).pin_memory()
    oh = torch.empty((M, DECODE[1][1]), dtype=torch.float16).pin_memory()

    # x comes in by an async copy from pinned memory; the second layer stores its
    # output straight into pinned host memory (the API accepts a page-locked
    # output: the kernels write it through unified addressing), which is the
    # step's device-to-host transfer
    def e2e_step(i):
        x.copy_(xh, non_blocking=True)
        (qa, sa), (qb, sb) = rot[i % copies]
        w4.linear(x, qa, sa, GROUP, out=h)
        w4.linear(h, qb, sb, GROUP, out=oh)

    e2e_mode = "cuda_graph"
    run = e2e_step
    try:
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(cap):  # warm-up on the capture stream: its workspace exists before capture
            for i in range(copies):
                e2e_step(i)
        cap.synchronize()
        graphs = []
        for i in range(copies):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=cap):
                e2e_step(i)
            graphs.append(gr)
        run = lambda i: graphs[i % copies].replay()  # noqa: E731
        for i in range(3):
            run(i)
        torch.cuda.synchronize()
        w4.device_status()
    except (RuntimeError, w4.W4A16Error) as exc:
        e2e_mode = f"eager (graph capture failed: {type(exc).__name__})"
        run = e2e_step
        torch.cuda.synchronize()
    for i in range(3):
        run(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        run(i)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    w4.device_status()

    extra = {}
    if not args.decode_only:
        extra = side_measurements(args, torch, w4, dev, hbm_peak, tc_peak, l2)

    cs = clocks.summary()
    return dict(
        spread=spread, static_mode=static_mode, software=gpu_software(torch),
        value=value, ms_per_step=ms_total / args.steps, kernel_ms=kernel_ms, achieved=achieved,
        hbm_peak=hbm_peak, tc_peak=tc_peak, peak_kind=peak_kind, copies=copies,
        e2e=dict(value=step_bytes * args.steps * world / (e2e_ms * 1e-3) / 1e9, unit="GB/s",
                 h2d_bytes_per_step=xh.numel() * 2, d2h_bytes_per_step=oh.numel() * 2,
                 ms_per_step=e2e_ms / args.steps, mode=e2e_mode),
        clocks=cs, extra=extra, gpu=torch.cuda.get_device_name(dev), sms=props.multi_processor_count,
        launches=2 * args.steps, per_launch_bytes=per_launch_bytes)


def _time_launches(torch, fn, n, sleep_cycles=2e7):
    """Mean device time per launch of n back-to-back launches (CUDA events at the ends)."""
    torch.cuda.synchronize()
    torch.cuda._sleep(int(sleep_cycles))
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(n):
        fn(i)
    t1.record()
    torch.cuda.synchronize()
    return [t0.elapsed_time(t1) / n]


def side_measurements(args, torch, w4, dev, hbm_peak, tc_peak, l2):
    """Batched decode (M=4), prefill GEMM (M=4096) and routed experts, if supported."""
    out = {}
    g = workloads.rng(0)
    # batched decode np4: the gate/up shape, rotated copies
    K, N = DECODE[0]
    W = torch.from_numpy(workloads.weights(g, N, K)).to(dev)
    qw, s = w4.pack(W, GROUP)
    del W
    per = N * K // 2 + N * (K // GROUP) * 2
    copies = max(2, -(-4 * l2 // per))
    rot = [(qw.clone(), s.clone()) for _ in range(copies)]
    x4 = torch.from_numpy(workloads.activations(g, 4, K)).to(dev)
    y4 = torch.empty((4, N), dtype=torch.float16, device=dev)
    f = lambda i: w4.linear(x4, rot[i % copies][0], rot[i % copies][1], GROUP, out=y4)  # noqa: E731
    for i in range(5):
        f(i)
    ms = statistics.median(_time_launches(torch, f, 100))
    b = per + 4 * K * 2 + 4 * N * 2
    out["decode_m4"] = {"shape": [4, K, N], "us": ms * 1e3, "GB/s": b / (ms * 1e-3) / 1e9,
                        "frac_hbm": b / (ms * 1e-3) / 1e9 / hbm_peak}
    # small-batch continuum: M = 8, 16 (decode GEMV) and 32, 64 (narrow-tile GEMM)
    for Ms in (8, 16, 32, 64):
        xs_ = torch.from_numpy(workloads.activations(g, Ms, K)).to(dev)
        ys_ = torch.empty((Ms, N), dtype=torch.float16, device=dev)
        f = lambda i: w4.linear(xs_, rot[i % copies][0], rot[i % copies][1], GROUP, out=ys_)  # noqa: E731
        for i in range(5):
            f(i)
        ms = statistics.median(_time_launches(torch, f, 100))
        b = per + Ms * K * 2 + Ms * N * 2
        fl = 2.0 * Ms * N * K
        out[f"batch_m{Ms}"] = {"shape": [Ms, K, N], "us": ms * 1e3, "GB/s": b / (ms * 1e-3) / 1e9,
                               "frac_hbm": b / (ms * 1e-3) / 1e9 / hbm_peak, "TFLOP/s": fl / (ms * 1e-3) / 1e12}
    # fused gate + up pair with the SiLU * up epilogue (one launch, both matrices streamed)
    try:
        W2 = torch.from_numpy(workloads.weights(workloads.rng(7), N, K)).to(dev)
        qw2, s2 = w4.pack(W2, GROUP)
        del W2
        pairs = [(rot[i][0], rot[i][1], qw2.clone(), s2.clone()) for i in range(copies)]
        x1 = torch.from_numpy(workloads.activations(g, 1, K)).to(dev)
        y1 = torch.empty((1, N), dtype=torch.float16, device=dev)
        f = lambda i: w4.linear_gated(x1, *pairs[i % copies], GROUP, out=y1)  # noqa: E731
        for i in range(5):
            f(i)
        ms = statistics.median(_time_launches(torch, f, 100))
        b = 2 * per + K * 2 + N * 2
        out["decode_gated_m1"] = {"shape": [1, K, N], "us": ms * 1e3, "GB/s": b / (ms * 1e-3) / 1e9,
                                  "frac_hbm": b / (ms * 1e-3) / 1e9 / hbm_peak}
        del pairs
    except w4.W4A16Error as e:
        out["decode_gated_m1"] = {"unavailable": str(e)}
    del rot
    # prefill GEMM M=4096
    try:
        xp = torch.from_numpy(workloads.activations(g, 4096, K, outlier_frac=0.01)).to(dev)
        yp = torch.empty((4096, N), dtype=torch.float16, device=dev)
        f = lambda i: w4.linear(xp, qw, s, GROUP, out=yp)  # noqa: E731
        for i in range(3):
            f(i)
        ms = statistics.median(_time_launches(torch, f, 20))
        fl = 2.0 * 4096 * N * K
        out["prefill_m4096"] = {"shape": [4096, K, N], "us": ms * 1e3, "TFLOP/s": fl / (ms * 1e-3) / 1e12,
                                "frac_tc": fl / (ms * 1e-3) / 1e12 / tc_peak}
        xp5 = xp[:512].contiguous()
        yp5 = yp[:512]
        f = lambda i: w4.linear(xp5, qw, s, GROUP, out=yp5)  # noqa: E731
        for i in range(3):
            f(i)
        ms = statistics.median(_time_launches(torch, f, 50))
        fl = 2.0 * 512 * N * K
        out["prefill_m512"] = {"shape": [512, K, N], "us": ms * 1e3, "TFLOP/s": fl / (ms * 1e-3) / 1e12,
                               "frac_tc": fl / (ms * 1e-3) / 1e12 / tc_peak}
    except w4.W4A16Error as e:
        out["prefill"] = {"unavailable": str(e)}
    # fused gate + up with the SiLU * up epilogue (one GEMM over both matrices)
    # against the two projections as separate GEMMs, at M = 512 and 4096
    try:
        if "prefill_m512" not in out:
            raise w4.W4A16Error("the prefill GEMM did not run")
        W2 = torch.from_numpy(workloads.weights(workloads.rng(7), N, K)).to(dev)
        qu, su = w4.pack(W2, GROUP)
        del W2
        for Mg in (512, 4096):
            xg = xp[:Mg].contiguous()
            yg, yu = yp[:Mg], torch.empty((Mg, N), dtype=torch.float16, device=dev)
            fused = lambda i: w4.linear_gated(xg, qw, s, qu, su, GROUP, out=yg)  # noqa: E731

            def two(i):
                w4.linear(xg, qw, s, GROUP, out=yg)
                w4.linear(xg, qu, su, GROUP, out=yu)
            n = 50 if Mg == 512 else 10
            for i in range(3):
                fused(i)
                two(i)
            ms = statistics.median(_time_launches(torch, fused, n))
            ms2 = statistics.median(_time_launches(torch, two, n))
            fl = 2.0 * 2 * Mg * N * K
            out[f"prefill_gated_m{Mg}"] = {"shape": [Mg, K, N], "us": ms * 1e3, "us_two_gemms": ms2 * 1e3,
                                           "TFLOP/s": fl / (ms * 1e-3) / 1e12,
                                           "frac_tc": fl / (ms * 1e-3) / 1e12 / tc_peak}
            del yu
        w4.device_status()
        del qu, su
    except w4.W4A16Error as e:
        out["prefill_gated"] = {"unavailable": str(e)}
    # routed experts: E=128, 4096 tokens, top-8 (R = 32768 rows), group 32
    try:
        for name, (Km, Nm) in (("moe_gate_up", (2048, 512)), ("moe_down", (512, 2048))):
            W, xs, rt = workloads.moe(Km, Nm)
            E = W.shape[0]
            Wd = torch.from_numpy(W.reshape(E * Nm, Km)).to(dev)
            qm, sm = w4.pack(Wd, 32)
            del Wd, W
            qm, sm = qm.view(E, Nm, Km // 2), sm.view(E, Nm, Km // 32)
            xd = torch.from_numpy(xs).to(dev)
            off = torch.from_numpy(rt.offsets).to(dev)
            yd = torch.empty((xs.shape[0], Nm), dtype=torch.float16, device=dev)
            f = lambda i: w4.grouped_linear(xd, qm, sm, off, 32, out=yd)  # noqa: E731
            for i in range(3):
                f(i)
            ms = statistics.median(_time_launches(torch, f, 30))
            R = xs.shape[0]
            fl = 2.0 * R * Nm * Km
            b = moe_bytes(E, R, Km, Nm, 32)
            out[name] = {"E": E, "R": R, "K": Km, "N": Nm, "us": ms * 1e3, "TFLOP/s": fl / (ms * 1e-3) / 1e12,
                         "frac_tc": fl / (ms * 1e-3) / 1e12 / tc_peak, "GB/s": b / (ms * 1e-3) / 1e9,
                         "frac_hbm": b / (ms * 1e-3) / 1e9 / hbm_peak}
            del qm, sm, xd, yd
        w4.device_status()
    except w4.W4A16Error as e:
        out["moe"] = {"unavailable": str(e)}
    # routed-MoE dispatch around the grouped layer at the same workload: router
    # (softmax top-8 of 128), permutation + gather of x (K = 2048), weighted combine (N = 2048)
    try:
        T, E, k, Kh = workloads.MOE["tokens"], workloads.MOE["E"], workloads.MOE["top_k"], workloads.MOE["hidden"]
        gr = workloads.rng(7)
        logits = torch.from_numpy(workloads.router_logits(gr, T, E)).to(dev)
        xt = torch.from_numpy(workloads.activations(gr, T, Kh)).to(dev)
        ids, wts = w4.moe_route(logits, k)
        off, row_of, tok, xs = w4.moe_dispatch(ids, E, xt)
        ys = torch.from_numpy(workloads.activations(gr, T * k, Kh)).to(dev)
        P = T * k
        cases = {
            "moe_route": (lambda i: w4.moe_route(logits, k), T * E * 4 + P * 8),
            "moe_dispatch": (lambda i: w4.moe_dispatch(ids, E, xt), P * 4 * 2 + P * 8 + T * Kh * 2 + P * Kh * 2),
            "moe_combine": (lambda i: w4.moe_combine(ys, row_of, wts), P * Kh * 2 + T * Kh * 2 + P * 8),
        }
        for name, (f, b) in cases.items():
            for i in range(3):
                f(i)
            ms = statistics.median(_time_launches(torch, f, 30))
            out[name] = {"T": T, "E": E, "top_k": k, "K": Kh, "us": ms * 1e3, "GB/s": b / (ms * 1e-3) / 1e9,
                         "frac_hbm": b / (ms * 1e-3) / 1e9 / hbm_peak}
        w4.device_status()
        del logits, xt, ys, xs
    except w4.W4A16Error as e:
        out["moe_dispatch"] = {"unavailable": str(e)}
    # GGUF block formats (Q4_K, Q5_1): the decode GEMV at M = 1 on both decode
    # shapes, rotated copies so that successive launches miss in L2
    try:
        for fmt in ("q4_k", "q5_1"):
            for K, N in DECODE:
                gb = workloads.rng(9)
                blk = torch.from_numpy(workloads.raw_blocks(gb, fmt, N, K)).to(dev)
                per = blk.numel()
                nb = max(2, -(-4 * l2 // per))
                rotb = [blk] + [blk.clone() for _ in range(nb - 1)]
                xb = torch.from_numpy(workloads.activations(gb, 1, K)).to(dev)
                yb = torch.empty((1, N), dtype=torch.float16, device=dev)
                f = lambda i: w4.blocks_linear(fmt, xb, rotb[i % nb], out=yb)  # noqa: E731
                for i in range(5):
                    f(i)
                ms = statistics.median(_time_launches(torch, f, 100))
                b = per + K * 2 + N * 2
                out[f"blocks_{fmt}_m1_{K}x{N}"] = {"shape": [1, K, N], "us": ms * 1e3,
                                                   "GB/s": b / (ms * 1e-3) / 1e9,
                                                   "frac_hbm": b / (ms * 1e-3) / 1e9 / hbm_peak}
                del rotb, blk
        w4.device_status()
    except w4.W4A16Error as e:
        out["blocks"] = {"unavailable": str(e)}
    # the whole routed layer (4096 tokens, top-8 of 128 experts, hidden 2048, expert
    # width 512, group 32): route -> dispatch -> gate/up GEMM -> down GEMM -> combine,
    # with the token gather as a separate copy (dispatch writes x_sorted) or fused into
    # the gate/up GEMM's activation loads
    try:
        T, E, k, Kh, Ni = (workloads.MOE[key] for key in ("tokens", "E", "top_k", "hidden", "inter"))
        gr = workloads.rng(8)
        logits = torch.from_numpy(workloads.router_logits(gr, T, E)).to(dev)
        xt = torch.from_numpy(workloads.activations(gr, T, Kh)).to(dev)
        w_gu = torch.from_numpy(workloads.weights(gr, E * Ni, Kh)).to(dev)
        q_gu, s_gu = w4.pack(w_gu, 32)
        del w_gu
        w_dn = torch.from_numpy(workloads.weights(gr, E * Kh, Ni)).to(dev)
        q_dn, s_dn = w4.pack(w_dn, 32)
        del w_dn
        q_gu, s_gu = q_gu.view(E, Ni, Kh // 2), s_gu.view(E, Ni, Kh // 32)
        q_dn, s_dn = q_dn.view(E, Kh, Ni // 2), s_dn.view(E, Kh, Ni // 32)
        h = torch.empty((T * k, Ni), dtype=torch.float16, device=dev)
        ys = torch.empty((T * k, Kh), dtype=torch.float16, device=dev)

        def layer(fused):
            ids, wts = w4.moe_route(logits, k)
            if fused:
                off, row_of, tok, _ = w4.moe_dispatch(ids, E)
                w4.grouped_linear_gather(xt, tok, q_gu, s_gu, off, 32, out=h)
            else:
                off, row_of, tok, xs = w4.moe_dispatch(ids, E, xt)
                w4.grouped_linear(xs, q_gu, s_gu, off, 32, out=h)
            w4.grouped_linear(h, q_dn, s_dn, off, 32, out=ys)
            return w4.moe_combine(ys, row_of, wts)

        for name, fused in (("moe_layer_unfused", False), ("moe_layer_fused_gather", True)):
            for i in range(3):
                layer(fused)
            ms = statistics.median(_time_launches(torch, lambda i: layer(fused), 20))
            out[name] = {"T": T, "E": E, "top_k": k, "hidden": Kh, "inter": Ni, "us": ms * 1e3,
                         "TFLOP/s": 2 * 2.0 * T * k * Kh * Ni / (ms * 1e-3) / 1e12,
                         "steps": "route, dispatch" + ("" if fused else " with x gather") +
                                  ", gate/up GEMM" + (" gathering x" if fused else "") + ", down GEMM, combine"}
        w4.device_status()
        del q_gu, s_gu, q_dn, s_dn, h, ys, xt, logits
    except w4.W4A16Error as e:
        out["moe_layer"] = {"unavailable": str(e)}
    return out


# ------------------------------------------------------------ reference arm --

def _oracle_decode_setup():
    import oracle

    oracle.build()
    g = workloads.rng(0)
    mats = [oracle.quantize(workloads.weights(g, N, K), GROUP) for K, N in DECODE]
    x = workloads.activations(g, 1, DECODE[0][0])
    # the second layer's input (one untimed pass): a step that covers only part of
    # the first layer's outputs still feeds the second layer a full activation row
    h = oracle.linear(x, *mats[0], GROUP)[0].astype(np.float16)
    return oracle, mats, x, h


def _sample_bytes(rows):
    """Algorithmic bytes of a decode step that computes rows[i] outputs of layer i."""
    total = 0
    for (K, N), n in zip(DECODE, rows):
        total += n * K // 2 + n * (K // GROUP) * 2 + K * 2 + n * 2
    return total


def run_reference(steps: int, warmup: int, budget_s: float = 150.0):
    """The CPU oracle (fp64, one thread) on the decode step. A full step takes
    about a second on one core; when steps + warmup full steps would exceed
    about `budget_s`, every step computes the same leading fraction of both
    layers' outputs (a bounded sample of the same workload; the metric is
    bytes per second either way)."""
    oracle, mats, x, h = _oracle_decode_setup()
    t0 = time.perf_counter()
    oracle.linear(x, mats[0][0][:256], mats[0][1][:256], GROUP)  # probe: seconds per output row
    per_row = (time.perf_counter() - t0) / 256
    full_s = per_row * sum(N * K / DECODE[0][0] for K, N in DECODE)
    frac = min(1.0, budget_s / max(1e-9, (steps + warmup) * full_s))
    rows = [max(16, int(N * frac)) for _, N in DECODE]

    def step():
        oracle.linear(x, mats[0][0][:rows[0]], mats[0][1][:rows[0]], GROUP)
        oracle.linear(h, mats[1][0][:rows[1]], mats[1][1][:rows[1]], GROUP)

    for _ in range(warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    dt = time.perf_counter() - t0
    sample = (f"{steps} timed steps after {warmup} warm-up steps; each step = the decode step (M=1, "
              f"5120->17408->5120, group 128) on the first {rows[0]} and {rows[1]} output rows of the two "
              f"layers ({100 * frac:.1f} %), fp64, one thread")
    return _sample_bytes(rows) * steps / dt / 1e9, dt, sample


def cpu_baseline_sample(budget_s=12.0):
    """Oracle decode steps on one host core until about `budget_s` seconds pass."""
    oracle, mats, x, _ = _oracle_decode_setup()
    n, t0 = 0, time.perf_counter()
    while True:
        y1, _ = oracle.linear(x, *mats[0], GROUP)
        oracle.linear(y1.astype(np.float16), *mats[1], GROUP)
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    host = host_info()
    out = {"value": decode_bytes(1) * n / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": f"{n} full decode steps (M=1, 5120->17408->5120, group 128), fp64, one thread, {dt:.1f} s",
           "host": host}
    # the same oracle threaded over the output columns on every host core
    threads = max(1, host["nproc"] or 1)
    n, t0 = 0, time.perf_counter()
    while True:
        y1, _ = oracle.linear(x, *mats[0], GROUP, threads=threads)
        oracle.linear(y1.astype(np.float16), *mats[1], GROUP, threads=threads)
        n += 1
        if time.perf_counter() - t0 >= budget_s / 4:
            break
    dt = time.perf_counter() - t0
    out["threaded"] = {"value": decode_bytes(1) * n / dt / 1e9, "unit": "GB/s", "cores": threads,
                       "sample": f"{n} full decode steps, the oracle split over output columns on {threads} "
                                 f"threads, {dt:.1f} s"}
    out["extrapolated"] = oracle_other_configs(oracle)
    return out


def oracle_other_configs(oracle):
    """The oracle (one thread) on bounded samples of the prefill and routed-expert
    workloads, extrapolated linearly in the number of multiply-adds to the full
    problems. Labelled 'extrapolated': the full problems would take hours."""
    res = {}
    g = workloads.rng(11)
    # prefill: 64 token rows x the first 2048 output columns of K=5120 -> N=17408
    K, N, rows, cols = 5120, 17408, 64, 2048
    qw, s = oracle.quantize(workloads.weights(g, cols, K), GROUP)
    x = workloads.activations(g, rows, K, outlier_frac=0.01)
    t0 = time.perf_counter()
    oracle.linear(x, qw, s, GROUP)
    dt = time.perf_counter() - t0
    per_mac = dt / (rows * cols * K)
    for M in (512, 4096):
        t = per_mac * M * N * K
        res[f"prefill_m{M}"] = {"s": t, "TFLOP/s": 2.0 * M * N * K / t / 1e12,
                                "sample": f"{rows} rows x {cols} columns timed ({dt:.2f} s), extrapolated"}
    # routed experts: the rows of 2 experts (about 512 of 32768) at each projection's shape
    for name, (Km, Nm) in (("moe_gate_up", (2048, 512)), ("moe_down", (512, 2048))):
        rows = 512
        qw, s = oracle.quantize(workloads.weights(g, Nm, Km), 32)
        x = workloads.activations(g, rows, Km)
        t0 = time.perf_counter()
        oracle.linear(x, qw, s, 32)
        dt = time.perf_counter() - t0
        R = workloads.MOE["tokens"] * workloads.MOE["top_k"]
        t = dt * R / rows
        res[name] = {"s": t, "TFLOP/s": 2.0 * R * Nm * Km / t / 1e12,
                     "sample": f"{rows} rows of one expert's weights timed ({dt:.2f} s), extrapolated to R={R}"}
    return res


# ----------------------------------------------------------------- profile --

PROFILE_CASES = ("decode", "decode_down", "decode_m4", "decode_gated", "prefill", "prefill_m512", "prefill_gated",
                 "moe_gate_up", "moe_down", "moe_dispatch", "moe_gate_up_gather", "blocks_q4_k", "blocks_q4_k_down",
                 "blocks_q5_1", "blocks_q5_1_down")


def run_profile(case: str, launches: int):
    """A few launches of one workload, for ncu: no timing, no clocks, no oracle."""
    import torch

    import w4a16_group_quantized_linear_gb300 as w4

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w4.lib()
    g = workloads.rng(0)
    if case == "moe_dispatch":
        # router, dispatch (with the gather of x) and combine at the routed-expert workload
        T, E, k, Kh = workloads.MOE["tokens"], workloads.MOE["E"], workloads.MOE["top_k"], workloads.MOE["hidden"]
        logits = torch.from_numpy(workloads.router_logits(g, T, E)).to(dev)
        xt = torch.from_numpy(workloads.activations(g, T, Kh)).to(dev)
        ys = torch.from_numpy(workloads.activations(g, T * k, Kh)).to(dev)
        for _ in range(launches):
            ids, wts = w4.moe_route(logits, k)
            off, row_of, tok, xs = w4.moe_dispatch(ids, E, xt)
            w4.moe_combine(ys, row_of, wts)
    elif case == "decode_gated":
        K, N = DECODE[0]
        mats = [w4.pack(torch.from_numpy(workloads.weights(g, N, K)).to(dev), GROUP) for _ in range(8)]
        x = torch.from_numpy(workloads.activations(g, 1, K)).to(dev)
        y = torch.empty((1, N), dtype=torch.float16, device=dev)
        for i in range(launches):  # four gate/up pairs in turn: successive launches miss in L2
            j = 2 * (i % 4)
            w4.linear_gated(x, *mats[j], *mats[j + 1], GROUP, out=y)
    elif case == "prefill_gated":
        # the gate/up pair at M = 512 in one GEMM with the SiLU * up epilogue
        K, N = DECODE[0]
        qg, sg = w4.pack(torch.from_numpy(workloads.weights(g, N, K)).to(dev), GROUP)
        qu, su = w4.pack(torch.from_numpy(workloads.weights(g, N, K)).to(dev), GROUP)
        x = torch.from_numpy(workloads.activations(g, 512, K, outlier_frac=0.01)).to(dev)
        y = torch.empty((512, N), dtype=torch.float16, device=dev)
        for _ in range(launches):
            w4.linear_gated(x, qg, sg, qu, su, GROUP, out=y)
    elif case == "moe_gate_up_gather":
        # the gate/up projection reading its rows straight from the token-major x
        T, E, k, Kh, Ni = (workloads.MOE[key] for key in ("tokens", "E", "top_k", "hidden", "inter"))
        logits = torch.from_numpy(workloads.router_logits(g, T, E)).to(dev)
        xt = torch.from_numpy(workloads.activations(g, T, Kh)).to(dev)
        qm, sm = w4.pack(torch.from_numpy(workloads.weights(g, E * Ni, Kh)).to(dev), 32)
        qm, sm = qm.view(E, Ni, Kh // 2), sm.view(E, Ni, Kh // 32)
        ids, _ = w4.moe_route(logits, k)
        off, row_of, tok, _ = w4.moe_dispatch(ids, E)
        for _ in range(launches):
            w4.grouped_linear_gather(xt, tok, qm, sm, off, 32)
    elif case.startswith("blocks_"):
        # GGUF block-format GEMV, M = 1: blocks_q4_k / blocks_q5_1 on the gate/up
        # shape, *_down on the down shape
        fmt = "q4_k" if case.startswith("blocks_q4_k") else "q5_1"
        K, N = DECODE[1] if case.endswith("_down") else DECODE[0]
        copies = [torch.from_numpy(workloads.raw_blocks(g, fmt, N, K)).to(dev) for _ in range(4)]
        x = torch.from_numpy(workloads.activations(g, 1, K)).to(dev)
        y = torch.empty((1, N), dtype=torch.float16, device=dev)
        for i in range(launches):
            w4.blocks_linear(fmt, x, copies[i % 4], out=y)
    elif case.startswith("moe"):
        Km, Nm = (2048, 512) if case == "moe_gate_up" else (512, 2048)
        W, xs, rt = workloads.moe(Km, Nm)
        E = W.shape[0]
        qm, sm = w4.pack(torch.from_numpy(W.reshape(E * Nm, Km)).to(dev), 32)
        qm, sm = qm.view(E, Nm, Km // 2), sm.view(E, Nm, Km // 32)
        xd = torch.from_numpy(xs).to(dev)
        off = torch.from_numpy(rt.offsets).to(dev)
        yd = torch.empty((xs.shape[0], Nm), dtype=torch.float16, device=dev)
        for _ in range(launches):
            w4.grouped_linear(xd, qm, sm, off, 32, out=yd)
    else:
        K, N = DECODE[1] if case == "decode_down" else DECODE[0]
        M = {"decode": 1, "decode_down": 1, "decode_m4": 4, "prefill": 4096, "prefill_m512": 512}[case]
        qw, s = w4.pack(torch.from_numpy(workloads.weights(g, N, K)).to(dev), GROUP)
        copies = [(qw, s)] + [(qw.clone(), s.clone()) for _ in range(3)]  # successive launches miss in L2
        x = torch.from_numpy(workloads.activations(g, M, K, outlier_frac=0.01 if M > 16 else 0.0)).to(dev)
        y = torch.empty((M, N), dtype=torch.float16, device=dev)
        for i in range(launches):
            w4.linear(x, *copies[i % 4], GROUP, out=y)
    torch.cuda.synchronize()
    w4.device_status()
    print(f"profile {case}: {launches} launches done")


def measured_traffic(kernel_file: str, profile: str):
    """DRAM bytes per launch from a committed ncu summary, or None once the
    kernel source has changed since that capture (the summary records the
    sha256 of the source it was taken on)."""
    import hashlib

    path = os.path.join(ROOT, "profiles", profile)
    src = os.path.join(ROOT, "w4a16_group_quantized_linear_gb300", "csrc", kernel_file)
    try:
        text = open(path).read()
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    fields = dict(line.split(":", 1) for line in text.splitlines() if line.startswith(("source_sha256:", "dram_bytes_per_launch:")))
    if fields.get("source_sha256", "").strip() != sha:
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# -------------------------------------------------------------------- main --

METRIC = "decode GEMV achieved HBM GB/s (M=1, 27B-class gate/up + down, group 128)"


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--decode-only", action="store_true", help="skip the prefill / MoE side measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", choices=PROFILE_CASES, help="only run a few launches of one workload (for ncu)")
    ap.add_argument("--launches", type=int, default=6, help="launches in --profile mode")
    args = ap.parse_args()
    if args.profile:
        run_profile(args.profile, args.launches)
        return
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    config = {"workload": "decode step M=1: x[1,5120] -> W4A16 5120->17408 -> W4A16 17408->5120, group 128",
              "M": 1, "shapes_KN": DECODE, "group": GROUP, "l2": "weights rotate through >4x L2 of copies",
              "parallelism": "replicas" if world > 1 else "single GPU"}

    if args.impl == "reference":
        if rank != 0:
            return
        value, dt, sample = run_reference(args.steps, args.warmup)
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample,
                             "host": host_info()},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return

    if world > 1:
        import torch

        torch.distributed.init_process_group("nccl")
    r = run_gpu(args, rank, world)
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": r["value"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "accumulate": "f32", "weights": "int4, fp16 group scales",
        "data": "synthetic",
        "config": config,
        "roofline": {"bound": "hbm", "achieved": r["achieved"], "peak": r["hbm_peak"], "unit": "GB/s",
                     "frac": r["achieved"] / r["hbm_peak"],
                     "traffic": measured_traffic("gemv.cu", "gemv_decode_m1.md"),
                     "kernel": "gemv_decode_kernel<cluster 2|4> (group 128, M=1)", "peak_kind": r["peak_kind"],
                     "kernel_us": r["kernel_ms"] * 1e3, "algorithmic_bytes_per_launch": r["per_launch_bytes"]},
        "per_call": r["spread"], "static_weights_mode": r["static_mode"],
        "e2e": r["e2e"], "gpu_launches": r["launches"], "clocks": r["clocks"], "gpu": r["gpu"], "sms": r["sms"],
        "software": r["software"], "source": source_info(), "host": host_info(),
        "side": r["extra"],
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_sample()
    print(json.dumps(line))


if __name__ == "__main__":
    main()
