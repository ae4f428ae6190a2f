"""Benchmark of the W4A16 group-quantized GEMM on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Headline workload (one step): the decode set -- one token (M=1) through the
four INT4 projections of a ~4B-decoder layer, qkv 2560x4096, o_proj 4096x2560,
gate_up 2560x19456, down 9728x2560, group 128 ("Quantize the Target, Quantize
the Drafter", pith.science review: INT4 target and drafter, group size 128).
Metric: effective HBM GB/s = algorithmic bytes / time, with
bytes = K*N/2 + (K/128)*N*2.5 + 2*M*K + 2*M*N per GEMM.  Inputs are seeded
synthetic tensors with the workload's distributions (w4a16_inputs).

L2: the step rotates through 8 distinct copies of the packed weights (398 MB,
more than twice the 129 MB L2), so every step streams its weights from HBM,
as a forward pass through 8 different layers would.

Also printed in the same JSON line: the verify set (M=16) in GB/s, prefill
(M=2048) in TFLOP/s, each GEMM alone, the roofline of the dominant kernel,
the end-to-end number through the public API with host buffers, and the CPU
oracle timed on this host.  `--impl reference` times the CPU oracle (the only
reference implementation of this path) on the same metric.

Multi-GPU: the GEMM needs no exchange, so N GPUs run N independent replicas
(weak scaling); value = bytes of all ranks / slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import w4a16_inputs as wi  # noqa: E402

METRIC = "W4A16 GEMM effective HBM GB/s (M=1,16) and TFLOP/s (M≥2048), % of roofline"
COPIES = 8
CLOCK_WINDOW_S = 1.5
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


HEADLINE_FLAGS = 3  # W4A16_FLAG_PDL | W4A16_FLAG_STATIC_WEIGHTS


def gemm_bytes(M, K, N, group=128):
    G = K // group
    return K * N // 2 + G * N * 2 + G * N // 2 + 2 * M * K + 2 * M * N


def gemm_flops(M, K, N):
    return 2 * M * N * K


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# The sources a kernel is compiled from: a traffic figure measured by ncu stays
# valid while these are unchanged (each entry of profiles/traffic.json names them).
GEMV_SOURCES = ("common.cuh", "gemv.cu", "gemv_cs.cu")


def kernel_source_sha(names=GEMV_SOURCES):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "int4_weight_only_gemm_gb300", "csrc")
    for name in sorted(names):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_key, field="dram_bytes_per_step"):
    """DRAM bytes from a committed ncu summary, if the kernel sources still
    match the ones profiled; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    e = d.get(kernel_key)
    if not e or e.get("source_sha") != kernel_source_sha(tuple(e.get("sources", GEMV_SOURCES))):
        return None
    return e.get(field)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the GPU works."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle
# ---------------------------------------------------------------------------

def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    seed, items = wi.WORKLOADS["decode_m1"]
    probs = [wi.generate_named(s, M, seed) for (s, M) in items]
    total_steps = args.steps + args.warmup
    # Per-step sample: a window of w columns of every projection (four windows
    # per projection, taken in turn), w sized from a calibration of the step
    # time t(w) = a + b w so that the whole run stays near `budget` seconds.
    # Many short steps run single-threaded: a parallel region per call would
    # cost more than the call itself.
    budget = 60.0
    threads = 1 if total_steps > 200 else oracle.max_threads()

    def make_windows(w):
        windows = []
        for p in probs:
            ww = min(max(8, w // 8 * 8), p.N)
            sl = []
            for i in range(4):
                c0 = ((p.N - ww) * i // 4) // 8 * 8
                sl.append((p.x, np.ascontiguousarray(p.qweight[:, c0:c0 + ww]),
                           np.ascontiguousarray(p.scales[:, c0:c0 + ww]),
                           np.ascontiguousarray(p.qzeros[:, c0 // 8:(c0 + ww) // 8]), p.M, p.K, ww))
            windows.append(sl)
        return windows

    def step_time(windows, reps):
        oracle.gemm(*windows[0][0][:4], nthreads=threads)  # library load, thread start
        t0 = time.perf_counter()
        for i in range(reps):
            for sl in windows:
                oracle.gemm(*sl[i % 4][:4], nthreads=threads)
        return (time.perf_counter() - t0) / reps

    t8 = step_time(make_windows(8), 20)
    t64 = step_time(make_windows(64), 5)
    b = max((t64 - t8) / 56.0, 1e-9)
    a = max(t8 - 8 * b, 0.0)
    per_step = budget / max(total_steps, 1)
    w = int((per_step - a) / b) if per_step > a else 8
    windows = make_windows(w)
    step_bytes = sum(gemm_bytes(sl[0][4], sl[0][5], sl[0][6]) for sl in windows)
    for i in range(args.warmup):
        for sl in windows:
            c = sl[i % 4]
            oracle.gemm(c[0], c[1], c[2], c[3], nthreads=threads)
    t0 = time.perf_counter()
    for i in range(args.steps):
        for sl in windows:
            c = sl[i % 4]
            oracle.gemm(c[0], c[1], c[2], c[3], nthreads=threads)
    dt = time.perf_counter() - t0
    value = step_bytes * args.steps / dt / 1e9
    cols = [(items[j][0], windows[j][0][6], p.N) for j, p in enumerate(probs)]
    sample = (f"decode set M=1, each step a column window of every projection "
              f"({', '.join(f'{s} {w}/{n}' for s, w, n in cols)} columns), full K")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / max(args.steps, 1) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "decode_m1: qkv 2560x4096, o_proj 4096x2560, gate_up 2560x19456, "
                               "down 9728x2560, M=1, group 128", "implementation": "CPU oracle (fp64 triple loop)"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

class Workload:
    """A list of GEMMs resident on the GPU with COPIES weight copies each."""

    def __init__(self, w, torch, items, seed, copies, device):
        self.w, self.torch = w, torch
        self.gemms = []
        for (shape, M) in items:
            p = wi.generate_named(shape, M, seed)
            x, qw, sc, qz = w.to_device(p, device)
            qd = w.w4a16_pack(qw)
            # every copy has its own weights, scales and zero points, so that
            # all three stream from HBM as they would for distinct layers
            qds = [qd] + [qd.clone() for _ in range(copies - 1)]
            scs = [sc] + [sc.clone() for _ in range(copies - 1)]
            qzs = [qz] + [qz.clone() for _ in range(copies - 1)]
            del qw
            y = torch.empty((M, p.N), dtype=torch.bfloat16, device=device)
            need = w.w4a16_workspace_bytes_max(M, p.N, p.K)  # any path or token tile
            ws = w.new_workspace(need, device)
            self.gemms.append(dict(p=p, shape=shape, M=M, K=p.K, N=p.N, x=x, qds=qds, scs=scs, qzs=qzs, y=y, ws=ws,
                                   ws_bytes=ws.numel()))
        self.copies = copies
        self.bytes = sum(gemm_bytes(g["M"], g["K"], g["N"]) for g in self.gemms)
        self.flops = sum(gemm_flops(g["M"], g["K"], g["N"]) for g in self.gemms)

    def launch_step(self, copy, stream_ptr, only=None, flags=None, path=0):
        w = self.w
        n = 0
        for i, g in enumerate(self.gemms):
            if only is not None and i != only:
                continue
            st = w.w4a16_gemm_raw(g["x"].data_ptr(), g["qds"][copy].data_ptr(), g["scs"][copy].data_ptr(),
                                  g["qzs"][copy].data_ptr(), g["M"], g["N"], g["K"], 128, g["y"].data_ptr(),
                                  g["ws"].data_ptr(), g["ws_bytes"], path, stream_ptr, flags)
            if st != 0:
                raise RuntimeError(f"w4a16_gemm failed: {w.w4a16_status_str(st)}")
            n += 1
        return n

    def graphs(self, only=None, flags=None, path=0):
        """One graph per weight copy (a step each) and one for the whole rotation."""
        torch = self.torch
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for c in range(self.copies):  # warm-up outside capture
                self.launch_step(c, s.cuda_stream, only, flags, path)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        per_step = []
        for c in range(self.copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.launch_step(c, torch.cuda.current_stream().cuda_stream, only, flags, path)
            per_step.append(g)
        rot = torch.cuda.CUDAGraph()
        with torch.cuda.graph(rot):
            for c in range(self.copies):
                self.launch_step(c, torch.cuda.current_stream().cuda_stream, only, flags, path)
        torch.cuda.synchronize()
        return per_step, rot


def replay_steps(per_step, rot, copies, start, count):
    """Replays exactly `count` steps beginning at step index `start`."""
    i = start
    end = start + count
    while i < end and i % copies:
        per_step[i % copies].replay()
        i += 1
    while i + copies <= end:
        rot.replay()
        i += copies
    while i < end:
        per_step[i % copies].replay()
        i += 1


def time_graph_steps(torch, per_step, rot, copies, steps, warmup, barrier=None):
    replay_steps(per_step, rot, copies, 0, warmup)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    replay_steps(per_step, rot, copies, warmup, steps)
    e1.record()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    return e0.elapsed_time(e1)  # ms


def measure_e2e(w, torch, wl, steps):
    """Through the public binding with host buffers: per step, the step's
    activations (one pinned host buffer holding the four GEMMs' inputs) go to
    the device in one copy, the four GEMMs run, their outputs (one device
    buffer) come back to pinned host memory in one copy, and the host waits."""
    xs = [g["x"] for g in wl.gemms]
    ys = [g["y"] for g in wl.gemms]
    xn = [t.numel() for t in xs]
    yn = [t.numel() for t in ys]
    # 16-byte aligned slices (8 bf16) of one buffer per direction
    xo = [0]
    for n in xn:
        xo.append(xo[-1] + (n + 7) // 8 * 8)
    yo = [0]
    for n in yn:
        yo.append(yo[-1] + (n + 7) // 8 * 8)
    hx = torch.zeros(xo[-1], dtype=torch.bfloat16).pin_memory()
    for j, t in enumerate(xs):
        hx[xo[j]:xo[j] + xn[j]].copy_(t.reshape(-1).cpu())
    hy = torch.empty(yo[-1], dtype=torch.bfloat16).pin_memory()
    dx = torch.empty(xo[-1], dtype=torch.bfloat16, device=xs[0].device)
    dy = torch.empty(yo[-1], dtype=torch.bfloat16, device=xs[0].device)
    dxs = [dx[xo[j]:xo[j] + xn[j]].view(xs[j].shape) for j in range(len(xs))]
    dys = [dy[yo[j]:yo[j] + yn[j]].view(ys[j].shape) for j in range(len(ys))]
    h2d = hx.numel() * 2
    d2h = hy.numel() * 2
    stream = torch.cuda.current_stream()

    def one(i):
        c = i % wl.copies
        dx.copy_(hx, non_blocking=True)
        for j, g in enumerate(wl.gemms):
            w.w4a16_gemm(dxs[j], g["qds"][c], g["scs"][c], g["qzs"][c], out=dys[j], workspace=g["ws"],
                         flags=HEADLINE_FLAGS)
        hy.copy_(dy, non_blocking=True)
        stream.synchronize()

    for i in range(min(20, steps)):
        one(i)
    t0 = time.perf_counter()
    for i in range(steps):
        one(i)
    dt = time.perf_counter() - t0
    return wl.bytes * steps / dt / 1e9, h2d, d2h, dt / steps * 1e3


def cpu_baseline(min_seconds=8.0, one_core_seconds=3.0):
    """The oracle on the host cores: all of them (OpenMP default), then one."""
    import oracle
    seed, items = wi.WORKLOADS["decode_m1"]
    probs = [wi.generate_named(s, M, seed) for (s, M) in items]
    step_bytes = sum(gemm_bytes(p.M, p.K, p.N) for p in probs)
    cores = oracle.max_threads()

    def timed(limit, nthreads):
        n = 0
        t0 = time.perf_counter()
        while True:
            for p in probs:
                oracle.gemm(p.x, p.qweight, p.scales, p.qzeros, nthreads=nthreads)
            n += 1
            dt = time.perf_counter() - t0
            if dt >= limit or n >= 200:
                return n, dt

    n, dt = timed(min_seconds, 0)
    n1, dt1 = timed(one_core_seconds, 1)  # last: the thread count set here persists
    return {"value": step_bytes * n / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"the full decode set (4 projections, M=1) repeated {n} times, {dt:.1f} s",
            "one_core": {"value": step_bytes * n1 / dt1 / 1e9, "cores": 1,
                         "sample": f"the same set repeated {n1} times, {dt1:.1f} s"}}


def measure_requant(w, torch, device, hbm, reps=200):
    """Grid-preserving re-quantization of the gate_up weights (2560 x 19456)
    straight into the device layout, two weight copies alternating (> L2)."""
    K, N = wi.shape_kn("gate_up")
    p = wi.generate(1, K, N, seed=5, shape_index=2)
    ws = [torch.from_numpy(wi.random_weights(K, N, seed=5 + i).view(np.int16)).to(device).view(torch.bfloat16)
          for i in range(2)]
    sc = torch.from_numpy(p.scales.view(np.int16)).to(device).view(torch.float16)
    qz = torch.from_numpy(p.qzeros.view(np.int32)).to(device)
    outs = [torch.empty((K // 8, N), dtype=torch.int32, device=device) for _ in range(2)]
    for i in range(10):
        w.w4a16_requant_pack(ws[i % 2], sc, qz, out=outs[i % 2])
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(reps):
        w.w4a16_requant_pack(ws[i % 2], sc, qz, out=outs[i % 2])
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / reps
    G = K // 128
    nbytes = K * N * 2 + G * N * 2 + G * N // 2 + K * N // 2
    return {"us": us, "GB/s": nbytes / us / 1e3, "frac": nbytes / us / 1e3 / hbm,
            "bytes": nbytes, "shape": f"{K}x{N}", "launch": "stream loop of launches (no graph)"}


def measure_gate_up_silu(w, torch, device, hbm, bf16_peak):
    """The fused gate/up projection with its SiLU-multiply epilogue on the
    decoder's 2560 x 19456 shape (H = 9728) at M = 1, 16 and 2048, beside the
    plain gate_up GEMM of the same weights: CUDA graphs over rotating weight
    copies (> L2), as for the decode step."""
    K, N = wi.shape_kn("gate_up")
    H = N // 2
    out = {}
    for M, copies, n, seed in ((1, COPIES, 2000, 1), (16, COPIES, 2000, 2), (2048, 2, 20, 3)):
        p = wi.generate(M, K, N, seed=seed, shape_index=2)
        x, qw, sc, qz = w.to_device(p, device)
        fused = [w.w4a16_pack_gate_up(qw) for _ in range(copies)]
        plain = [w.w4a16_pack(qw) for _ in range(copies)]
        scs = [sc] + [sc.clone() for _ in range(copies - 1)]
        qzs = [qz] + [qz.clone() for _ in range(copies - 1)]
        del qw
        ws = w.new_workspace(w.w4a16_workspace_bytes(M, N, K), device)
        y_f = torch.empty((M, H), dtype=torch.bfloat16, device=device)
        y_p = torch.empty((M, N), dtype=torch.bfloat16, device=device)
        res = {}
        for name, qds, call in (
                ("fused", fused, lambda c: w.w4a16_gemm_gate_up_silu(x, fused[c], scs[c], qzs[c], out=y_f, workspace=ws)),
                ("plain", plain, lambda c: w.w4a16_gemm(x, plain[c], scs[c], qzs[c], out=y_p, workspace=ws))):
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                for c in range(len(qds)):
                    call(c)
            torch.cuda.current_stream().wait_stream(s)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for c in range(len(qds)):
                    call(c)
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            reps = max(1, n // copies)
            e0.record()
            for _ in range(reps):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            res[name] = e0.elapsed_time(e1) * 1e3 / (reps * copies)
            del g
        G = K // 128
        fbytes = K * N // 2 + G * N * 2 + G * N // 2 + M * K * 2 + M * H * 2
        entry = {"us": res["fused"], "plain_gate_up_us": res["plain"], "GB/s": fbytes / res["fused"] / 1e3}
        if M <= 16:
            entry["frac"] = entry["GB/s"] / hbm
        else:
            entry["TFLOP/s"] = gemm_flops(M, K, N) / res["fused"] / 1e6
            entry["frac"] = entry["TFLOP/s"] / bf16_peak
        # a separate activation pass would write y [M][2H] in bf16 and read it back
        entry["intermediate_bytes_avoided"] = M * N * 2 * 2 - M * H * 2
        out[f"M={M}"] = entry
        del x, sc, qz, fused, plain, ws, y_f, y_p
        torch.cuda.empty_cache()
    out["shape"] = f"K={K}, 2H={N} (H={H})"
    return out


# ---------------------------------------------------------------------------
# the M sweep (config 4) and the dispatch candidates
# ---------------------------------------------------------------------------

SWEEP_M = (1, 2, 4, 8, 16, 32, 64, 128, 8192)
# the dispatch table also measures prefill-sized M between 128 and 8192
TUNE_M = (1, 2, 4, 8, 16, 32, 64, 128, 256, 2048, 8192)
L2_BYTES = 129 << 20
PATH_NAMES = {1: "gemv", 2: "tc", 3: "gemv_splitk", 4: "gemv_cs"}


def sweep_items(vocab_ms=(1, 16), ms=SWEEP_M):
    """(shape, M) pairs of the sweep: the four projections at every M of `ms`,
    the vocabulary head at `vocab_ms`."""
    items = [(s, m) for m in ms for s in wi.LAYER]
    return items + [("vocab", m) for m in vocab_ms]


def candidates(M):
    """Kernel configurations the dispatch table chooses from at this M:
    (name, path, flags); the token tiles the tensor-core kernel may use here."""
    out = []
    if M <= 8:
        out += [("gemv_splitk", 3, 1), ("gemv_cs", 4, 1)]
    for nt in (16, 32, 64, 128, 192):
        if nt <= max(16, 2 * M) and (M > 8 or nt == 16) and (M < 2048 or nt >= 64):
            out.append((f"tc{nt}", 2, 1 | (nt << 8)))
    return out


def time_gemm(w, torch, p, device, path, flags, reps_target_ms=20.0):
    """Microseconds per launch of one GEMM: a CUDA graph launches it over a
    rotation of weight copies whose total exceeds twice the L2 (so every
    launch streams its weights from HBM), replayed after a warm-up."""
    x, qw, sc, qz = w.to_device(p, device)
    qd = w.w4a16_pack(qw)
    del qw
    wbytes = gemm_bytes(p.M, p.K, p.N)
    copies = int(min(64, max(2, -(-int(2.1 * L2_BYTES) // wbytes))))
    qds = [qd] + [qd.clone() for _ in range(copies - 1)]
    scs = [sc] + [sc.clone() for _ in range(copies - 1)]
    qzs = [qz] + [qz.clone() for _ in range(copies - 1)]
    y = torch.empty((p.M, p.N), dtype=torch.bfloat16, device=device)
    ws = w.new_workspace(w.w4a16_workspace_bytes_max(p.M, p.N, p.K), device)
    nbytes = ws.numel()

    def launch_all(stream_ptr):
        for q, sq, zq in zip(qds, scs, qzs):
            st = w.w4a16_gemm_raw(x.data_ptr(), q.data_ptr(), sq.data_ptr(), zq.data_ptr(), p.M, p.N, p.K, 128,
                                  y.data_ptr(), ws.data_ptr(), nbytes, path, stream_ptr, flags)
            if st != 0:
                raise RuntimeError(f"w4a16_gemm path {path} flags {flags}: {w.w4a16_status_str(st)}")

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        launch_all(s.cuda_stream)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        launch_all(torch.cuda.current_stream().cuda_stream)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    once = max(e0.elapsed_time(e1), 1e-3)
    reps = int(max(2, min(200, reps_target_ms / once)))
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (reps * copies)
    del g, qds, scs, qzs, qd, x, y, ws
    return us, copies


def roofline_us(M, K, N, hbm, bf16_peak):
    return max(gemm_bytes(M, K, N) / (hbm * 1e3), gemm_flops(M, K, N) / (bf16_peak * 1e6))


def measure_sweep(w, torch, device, hbm, bf16_peak):
    """Config 4: every (shape, M) of the sweep through the library's own
    kernel choice (path AUTO); per GEMM us, GB/s, TFLOP/s and the fraction of
    the roofline max(bytes / HBM, flops / bf16 peak), and the sums over the
    four projections of a layer."""
    out = {}
    for shape, M in sweep_items():
        p = wi.generate_named(shape, M, 4)
        us, copies = time_gemm(w, torch, p, device, 0, 1)
        rl = roofline_us(M, p.K, p.N, hbm, bf16_peak)
        e = out.setdefault(f"M={M}", {})
        e[shape] = {"us": us, "GB/s": gemm_bytes(M, p.K, p.N) / us / 1e3,
                    "TFLOP/s": gemm_flops(M, p.K, p.N) / us / 1e6, "frac": rl / us,
                    "path": PATH_NAMES.get(w.w4a16_auto_path(M, p.N, p.K), "?"), "weight_copies": copies}
        torch.cuda.empty_cache()
    for key, e in out.items():
        M = int(key[2:])
        if all(s in e for s in wi.LAYER):
            us = sum(e[s]["us"] for s in wi.LAYER)
            rl = sum(roofline_us(M, *wi.shape_kn(s), hbm, bf16_peak) for s in wi.LAYER)
            e["layer"] = {"us": us, "frac": rl / us}
    return out


def tune_dispatch(path_out, ms=TUNE_M):
    """Times every dispatch candidate at every point of the sweep (the vocabulary
    head at M <= 128 as well) and writes the measurements that
    int4_weight_only_gemm_gb300/csrc/gen_dispatch.py turns into the table."""
    import torch
    import int4_weight_only_gemm_gb300 as w
    w.load_library()
    device = torch.device("cuda", 0)
    props = torch.cuda.get_device_properties(device)
    entries = []
    for shape, M in sweep_items(vocab_ms=tuple(m for m in (1, 2, 4, 8, 16, 32, 64, 128) if m in ms), ms=ms):
        p = wi.generate_named(shape, M, 4)
        for name, path, flags in candidates(M):
            us, _ = time_gemm(w, torch, p, device, path, flags)
            entries.append({"shape": shape, "K": p.K, "N": p.N, "M": M, "config": name, "us": round(us, 3)})
            print(json.dumps(entries[-1]), flush=True)
        torch.cuda.empty_cache()
    doc = {"what": "microseconds per launch of each dispatch candidate (CUDA graphs over rotating copies of the "
                   "weights, scales and zero points, > 2x L2); written by bench.py --tune-dispatch",
           "device": props.name, "sms": props.multi_processor_count,
           "when": time.strftime("%Y-%m-%dT%H:%M:%SZ", time.gmtime()), "entries": entries}
    with open(path_out, "w") as f:
        json.dump(doc, f, indent=1)



def measure_swa(w, torch, device, hbm, bf16_peak):
    """Sliding-window decode attention of the drafter on the long scenario's
    context (8192 prompt + 256 generated = 8448 positions), window 1024 and
    2048, a 16-token draft block and a single query; 32 query heads over 8
    key/value heads of width 128.  CUDA graphs over 8 copies of the caches
    (277 MB, more than twice the L2).  Algorithmic bytes: the keys and values
    of every head's window once, plus q and out; flops 4 * 128 per (query,
    head, visible key)."""
    Hq, Hkv, d, L = 32, 8, 128, 8448
    out = {}
    r = np.random.default_rng(12)
    kc = [torch.randn((Hkv, L, d), device=device).to(torch.bfloat16) for _ in range(COPIES)]
    vt = [torch.randn((Hkv, d, L), device=device).to(torch.bfloat16) for _ in range(COPIES)]
    for nq in (16, 1):
        q = torch.from_numpy(r.standard_normal((nq, Hq, d), dtype=np.float32)).to(device).to(torch.bfloat16)
        o = torch.empty_like(q)
        for W in (1024, 2048):
            ws = w.new_workspace(w.w4a16_swa_workspace_bytes(nq, Hq, Hkv, L, W), device)

            def launch_all():
                for c in range(COPIES):
                    w.w4a16_swa_attention(q, kc[c], vt[c], L, W, False, out=o, workspace=ws)

            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                launch_all()
            torch.cuda.current_stream().wait_stream(s)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                launch_all()
            for _ in range(5):
                g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = 200
            e0.record()
            for _ in range(reps):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / (reps * COPIES)
            keys = min(L, W + nq - 1)                      # the block's window, per key/value head
            visible = sum(min(W, L - nq + i + 1) for i in range(nq))  # keys seen by each query
            nbytes = Hkv * keys * d * 2 * 2 + 2 * nq * Hq * d * 2
            flops = 4 * d * visible * Hq
            rl = max(nbytes / (hbm * 1e3), flops / (bf16_peak * 1e6))
            out[f"nq={nq} W={W}"] = {"us": us, "GB/s": nbytes / us / 1e3, "TFLOP/s": flops / us / 1e6,
                                     "frac": rl / us, "bytes": nbytes, "flops": flops,
                                     "bound": "hbm" if nbytes / hbm > flops / bf16_peak * 1e-3 else "tensor"}
            del g, ws
        del q, o
    del kc, vt
    torch.cuda.empty_cache()
    out["shape"] = f"Hq={Hq}, Hkv={Hkv}, d={d}, L={L}, causal; value cache transposed per head"
    return out


def max_over_ranks(dist, torch, value: float, device) -> float:
    """The largest of the ranks' values (the slowest rank's time); the value
    itself without a process group."""
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_case(case, reps):
    """One seeded GEMM of the named layer shape, launched `reps` times back to
    back on the current stream (the workload of the ncu summaries)."""
    import torch
    import int4_weight_only_gemm_gb300 as w
    parts = case.split(":")
    shape, M = parts[0], int(parts[1])
    path = int(parts[2]) if len(parts) > 2 else 0
    p = wi.generate_named(shape, M, 1)
    x, qw, sc, qz = w.to_device(p)
    qd = w.w4a16_pack(qw)
    del qw
    y = torch.empty((M, p.N), dtype=torch.bfloat16, device="cuda")
    ws = w.new_workspace(w.w4a16_workspace_bytes(M, p.N, p.K, path=path), "cuda")
    for _ in range(reps):
        w.w4a16_gemm(x, qd, sc, qz, path=path, workspace=ws, out=y)
    torch.cuda.synchronize()
    st = w.w4a16_last_device_status()
    if st != 0:
        raise RuntimeError(f"device status {w.w4a16_status_str(st)}")
    print(json.dumps({"case": case, "reps": reps, "path": path, "ok": True}), flush=True)


def run_swa_case(case, reps):
    """One sliding-window attention call of the swa_decode_attention scenario
    (Hq = 32, Hkv = 8, d = 128, L = 8448, causal), launched `reps` times back
    to back (the workload of the attention ncu summary)."""
    import torch
    import int4_weight_only_gemm_gb300 as w
    nq, W = (int(v) for v in case.split(":"))
    Hq, Hkv, d, L = 32, 8, 128, 8448
    g = torch.Generator(device="cuda").manual_seed(12)
    kc = torch.randn((Hkv, L, d), device="cuda", generator=g).to(torch.bfloat16)
    vt = torch.randn((Hkv, d, L), device="cuda", generator=g).to(torch.bfloat16)
    q = torch.randn((nq, Hq, d), device="cuda", generator=g).to(torch.bfloat16)
    o = torch.empty_like(q)
    ws = w.new_workspace(w.w4a16_swa_workspace_bytes(nq, Hq, Hkv, L, W), "cuda")
    for _ in range(reps):
        w.w4a16_swa_attention(q, kc, vt, L, W, False, out=o, workspace=ws)
    torch.cuda.synchronize()
    st = w.w4a16_last_device_status()
    if st != 0:
        raise RuntimeError(f"device status {w.w4a16_status_str(st)}")
    print(json.dumps({"swa_case": case, "reps": reps, "ok": True}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50000)
    ap.add_argument("--warmup", type=int, default=1000)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true", help="skip the M=16 / M=2048 / per-GEMM extras")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end host-buffer measurement")
    ap.add_argument("--case", default="",
                    help="SHAPE:M[:PATH] -- run that one GEMM --reps times and exit (for profilers); "
                         "PATH 0 = auto, 1 = split-K GEMV, 2 = tensor-core kernel")
    ap.add_argument("--swa-case", default="",
                    help="NQ:W -- run one sliding-window attention call (the swa_decode_attention "
                         "scenario) --reps times and exit (for profilers)")
    ap.add_argument("--requant-case", action="store_true",
                    help="run the re-quantize + pack of the gate_up weights --reps times and exit (for profilers)")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--no-sweep", action="store_true", help="skip the M sweep")
    ap.add_argument("--only", default="", help="comma-separated extras to run (default: all)")
    ap.add_argument("--tune-dispatch", default="",
                    help="OUT.json -- time every dispatch candidate over the sweep, write them and exit")
    ap.add_argument("--tune-m", default="", help="comma-separated M values for --tune-dispatch (default: all)")
    args = ap.parse_args()
    if args.case:
        run_case(args.case, args.reps)
        return
    if args.swa_case:
        run_swa_case(args.swa_case, args.reps)
        return
    if args.requant_case:
        import torch
        import int4_weight_only_gemm_gb300 as w
        r = measure_requant(w, torch, "cuda", 1.0, reps=args.reps)
        st = w.w4a16_last_device_status()
        if st != 0:
            raise RuntimeError(f"device status {w.w4a16_status_str(st)}")
        print(json.dumps({"requant_case": r["shape"], "reps": args.reps, "ok": True}), flush=True)
        return
    if args.tune_dispatch:
        ms = tuple(int(v) for v in args.tune_m.split(",")) if args.tune_m else TUNE_M
        tune_dispatch(args.tune_dispatch, ms)
        return
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    import int4_weight_only_gemm_gb300 as w
    w.load_library()  # raises if the CUDA library is missing: there is no fallback
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    def barrier():
        if dist is not None:
            dist.barrier()

    peaks, peak_src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    bf16_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))

    seed1, items1 = wi.WORKLOADS["decode_m1"]
    wl = Workload(w, torch, items1, seed1, COPIES, device)
    # The four GEMMs as a programmatic-dependent chain whose weights are
    # constant (W4A16_FLAG_PDL | W4A16_FLAG_STATIC_WEIGHTS): each GEMM may start
    # streaming its weights before the preceding one completes.
    per_step, rot = wl.graphs(flags=HEADLINE_FLAGS)
    with ClockSampler(local_rank) as clk:
        time.sleep(0.3)  # nvidia-smi's first sample
        ms = time_graph_steps(torch, per_step, rot, COPIES, args.steps, args.warmup, barrier)
        # A short timed region can end between two samples: the same step
        # graphs keep replaying for CLOCK_WINDOW_S seconds after it, so the
        # clocks are sampled under the same load.
        reps = max(1, int(CLOCK_WINDOW_S * 1e3 / max(ms / args.steps * COPIES, 1e-3)))
        for _ in range(reps):
            rot.replay()
        torch.cuda.synchronize()
    clocks = clk.summary()
    clocks["window"] = f"the timed steps plus {reps * COPIES} more steps of the same graphs (~{CLOCK_WINDOW_S} s)"
    launches_in_graphs = len(wl.gemms) * args.steps  # graph replays do not pass through the library
    ms = max_over_ranks(dist, torch, ms, device)
    ms_step = ms / args.steps
    value = wl.bytes * args.steps * world / (ms / 1e3) / 1e9

    extra = {}
    failed = []  # extras that raised: the error goes into the line, later GPU extras are skipped

    def guarded(name, fn):
        if args.only and name not in args.only.split(","):
            return
        if failed:
            extra[name] = {"skipped": f"after the failure of {failed[0]}"}
            return
        try:
            fn()
        except Exception as exc:
            extra[name] = {"error": repr(exc)[:400]}
            if "CUDA" in repr(exc) or "cuda" in type(exc).__name__.lower() or "Accelerator" in type(exc).__name__:
                failed.append(name)  # the context is unusable: no more GPU work

    def ex_decode_per_gemm():
        # each projection alone (graph of the 8-copy rotation of that GEMM)
        per = {}
        for i, g in enumerate(wl.gemms):
            ps, rt = wl.graphs(only=i)
            n = max(200, min(args.steps, 20000))
            t_ms = time_graph_steps(torch, ps, rt, COPIES, n, 50)
            b = gemm_bytes(g["M"], g["K"], g["N"])
            per[g["shape"]] = {"us": t_ms / n * 1e3, "GB/s": b * n / (t_ms / 1e3) / 1e9,
                               "frac": b * n / (t_ms / 1e3) / 1e9 / hbm}
        extra["decode_m1_per_gemm"] = per

    def ex_decode_flags():
        # the decode set under each launch-flag combination
        fl = {}
        for flags, name, path in ((0, "plain", 0), (1, "pdl", 0), (3, "pdl_static_weights", 0),
                                  (1, "pdl_all_column_sliced", 4), (3, "pdl_static_all_column_sliced", 4),
                                  (3, "pdl_static_all_split_k", 3)):
            ps, rt = wl.graphs(flags=flags, path=path)
            n = max(200, min(args.steps, 20000))
            t_ms = time_graph_steps(torch, ps, rt, COPIES, n, 50)
            fl[name] = {"us_per_step": t_ms / n * 1e3, "GB/s": wl.bytes * n / (t_ms / 1e3) / 1e9,
                        "path": PATH_NAMES.get(path, "auto")}
        extra["decode_m1_flags"] = fl

    def ex_workload(name, unit):
        seed, items = wi.WORKLOADS[name]
        small = unit == "GB/s"
        copies = COPIES if small else 2
        wl2 = Workload(w, torch, items, seed, copies, device)
        n = 4000 if small else 40
        # the step as the headline's: PDL chain with static weights; the plain
        # PDL chain beside it
        ps, rt = wl2.graphs()
        t_pdl = time_graph_steps(torch, ps, rt, copies, n, 10)
        del ps, rt
        ps, rt = wl2.graphs(flags=HEADLINE_FLAGS)
        t_ms = time_graph_steps(torch, ps, rt, copies, n, 10)
        if unit == "GB/s":
            v = wl2.bytes * n / (t_ms / 1e3) / 1e9
            frac = v / hbm
        else:
            v = wl2.flops * n / (t_ms / 1e3) / 1e12
            frac = v / bf16_peak
        per2 = {}
        for i, g in enumerate(wl2.gemms):
            ps1, rt1 = wl2.graphs(only=i)
            n1 = 2000 if small else 20
            t1 = time_graph_steps(torch, ps1, rt1, copies, n1, 5)
            per2[g["shape"]] = {"us": t1 / n1 * 1e3,
                                "GB/s": gemm_bytes(g["M"], g["K"], g["N"]) * n1 / (t1 / 1e3) / 1e9,
                                "TFLOP/s": gemm_flops(g["M"], g["K"], g["N"]) * n1 / (t1 / 1e3) / 1e12}
            del ps1, rt1
        extra[name] = {"value": v, "unit": unit, "frac": frac, "ms_per_step": t_ms / n,
                       "launch": "PDL chain, static weights (flags 3)", "ms_per_step_pdl_only": t_pdl / n,
                       "workload": ", ".join(f"{s} M={M}" for s, M in items), "per_gemm": per2}
        del ps, rt, wl2
        torch.cuda.empty_cache()

    def ex_verify_batched():
        # batched speculative verify: b draft blocks of 16 tokens through the
        # four projections of the layer, PDL-chained in one graph per step
        vb = {}
        for b in (1, 2, 3, 4):
            M = 16 * b
            wl3 = Workload(w, torch, [(s, M) for s in wi.LAYER], 2, COPIES, device)
            ps, rt = wl3.graphs(flags=HEADLINE_FLAGS)
            n = 2000
            t_ms = time_graph_steps(torch, ps, rt, COPIES, n, 10)
            us = t_ms / n * 1e3
            vb[f"M={M}"] = {"us_per_step": us, "GB/s": wl3.bytes / us / 1e3, "frac": wl3.bytes / us / 1e3 / hbm,
                            "tokens/s": M / us * 1e6}
            del ps, rt, wl3
            torch.cuda.empty_cache()
        extra["verify_batched"] = vb

    if rank == 0 and not args.no_extra:
        guarded("decode_m1_per_gemm", ex_decode_per_gemm)
        guarded("decode_m1_flags", ex_decode_flags)
        guarded("verify_m16", lambda: ex_workload("verify_m16", "GB/s"))
        guarded("prefill_m2048", lambda: ex_workload("prefill_m2048", "TFLOP/s"))
        guarded("requant_pack_gate_up",
                lambda: extra.__setitem__("requant_pack_gate_up", measure_requant(w, torch, device, hbm)))
        guarded("gate_up_silu", lambda: extra.__setitem__(
            "gate_up_silu", measure_gate_up_silu(w, torch, device, hbm, bf16_peak)))
        guarded("verify_batched", ex_verify_batched)
        guarded("swa_decode_attention",
                lambda: extra.__setitem__("swa_decode_attention", measure_swa(w, torch, device, hbm, bf16_peak)))
        if not args.no_sweep:
            guarded("sweep", lambda: extra.__setitem__("sweep", measure_sweep(w, torch, device, hbm, bf16_peak)))

    e2e = None
    if not args.no_e2e and not failed:
        e2e_v, h2d, d2h, e2e_ms = measure_e2e(w, torch, wl, min(2000, max(50, args.steps // 10)))
        e2e = {"value": e2e_v, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms, "api": "int4_weight_only_gemm_gb300.w4a16_gemm (C ABI w4a16_gemm_path)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline()

    if rank == 0:
        achieved = wl.bytes / (ms_step / 1e3) / 1e9
        traffic = profiled_traffic("gemv_decode_m1_step")
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "decode_m1: one token through qkv 2560x4096, o_proj 4096x2560, "
                                   "gate_up 2560x19456, down 9728x2560; group 128; int4 weights, bf16 x/y",
                       "global_batch": 1, "parallelism": f"replicas x{world}",
                       "l2": f"rotating {COPIES} copies of weights, scales and zero points "
                             f"({COPIES * wl.bytes / 1e6:.0f} MB > 2x L2)",
                       "bytes_per_step": wl.bytes,
                       "launch": "CUDA graph of the 8-copy rotation; PDL chain, static weights (flags 3)"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "traffic": traffic,
                         "kernel": "the GEMV of each of the step's four GEMMs (the dispatch table's form)",
                         "peak_source": f"{peak_src} hbm_gbs"},
            "e2e": e2e,
            "gpu_launches": launches_in_graphs,
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        # the tensor-core kernel's roofline on its dominant GEMM (gate_up) of the
        # verify and prefill steps: achieved = algorithmic bytes or flops of one
        # launch / its in-graph time
        for key, tkey, bound in (("verify_m16", "tc_verify_m16_gate_up", "hbm"),
                                 ("prefill_m2048", "tc_prefill_m2048_gate_up", "tensor")):
            e = extra.get(key)
            if not e or "per_gemm" not in e or "gate_up" not in e["per_gemm"]:
                continue
            M = 16 if key == "verify_m16" else 2048
            K, N = wi.shape_kn("gate_up")
            us = e["per_gemm"]["gate_up"]["us"]
            if bound == "hbm":
                ach, pk, unit = gemm_bytes(M, K, N) / us / 1e3, hbm, "GB/s"
            else:
                ach, pk, unit = gemm_flops(M, K, N) / us / 1e6, bf16_peak, "TFLOP/s"
            line[f"roofline_{key}"] = {"bound": bound, "achieved": ach, "peak": pk, "unit": unit, "frac": ach / pk,
                                       "traffic": profiled_traffic(tkey, "dram_bytes_per_launch"),
                                       "kernel": f"tc_gemm_kernel<{16 if M == 16 else 192}> on gate_up "
                                                 f"{K}x{N}, M={M}", "peak_source": f"{peak_src}"}
        line.update(extra)
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
