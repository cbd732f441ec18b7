"""Benchmark of the ternary-weight x int8 layer step on GB300.

One step = the three products of one ternary layer at M=16384 rows, N=3456,
K=1280 (the pages' largest forward shape, with the two backward products at
the same shape):
    C  = A . W        t3_gemm_fwd     (int8 x ternary -> int32)
    dX = dY . W^T     t3_gemm_bwd_dx  (int8 x ternary -> int32)
    dW = A^T . dY     t3_gemm_bwd_dw  (int8 x int8    -> int32)
The metric counts 2*M*N*K operations per product (zeros included), as the
pages do.  Inputs are synthetic and seeded (t3_synth), resident in HBM before
the timed region; the step moves ~410 MB, far more than the 129 MB L2, so no
explicit L2 flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the plain int64 loops) on a bounded
sample of rows of the same workload, on the host cores.
Multi-GPU runs (torchrun) are independent replicas: the products have no
exchange step on one layer, so nothing is communicated on the data path.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import t3_synth  # noqa: E402

METRIC = "TOPS (2·M·N·K/s) ternary×int8 fwd/dX/dW; % of int8 tensor peak / HBM roofline"
UNIT = "TOPS"
M, N, K = 16384, 3456, 1280
SEED = 2
OPS_PER_PRODUCT = 2 * M * N * K
WORKLOAD = f"ternary layer step fwd+dX+dW, M={M} N={N} K={K}"
FALLBACK_TFLOPS = 1900.0
STATED_INT8_TOPS = 4500.0   # the dense int8 tensor rate the target was stated against
PAGES_CONTEXT = "pages: fwd 16384x3456x1280 at 171 TOPS on an RTX 4090 (other hardware, fwd only)"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-pack", action="store_true",
                    help="skip the device-packer sweep (HBM-bound, reported beside the step)")
    ap.add_argument("--no-small-m", action="store_true",
                    help="skip the small-M forward sweep (for launch-list captures)")
    ap.add_argument("--step-only", action="store_true",
                    help="time the layer step (and its end-to-end form) only: no scaled, "
                         "quantizer, packer or small-M legs (for launch-list captures)")
    ap.add_argument("--small-m-only", metavar="M,N,K", default=None,
                    help="time one small-M forward configuration of the sweep and exit "
                         "(for profiler captures)")
    ap.add_argument("--hslm-only", metavar="M,N,K", default=None,
                    help="time the three products at one of the HSLM shapes and exit "
                         "(for profiler captures)")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def max_over_ranks(x, pg, device):
    """The largest of every rank's x (a time): the whole job takes as long as
    its slowest rank.  pg is torch.distributed (initialised) or None."""
    if pg is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_tops(ms_per_step, world):
    """Whole-job throughput: every rank runs one layer step (three products)
    per step, so the units all ranks processed over the slowest rank's time."""
    return 3 * OPS_PER_PRODUCT * world / (ms_per_step * 1e-3) / 1e12


def make_host_inputs():
    g = t3_synth.rng(SEED)
    A = t3_synth.int8_uniform(g, (M, K))
    w = t3_synth.ternary(g, (K, N))
    dY = t3_synth.int8_uniform(g, (M, N))
    return A, w, dY


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {}, "fallback"


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.index), "-lms", "100"],
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

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


SMALL_M = [(m, n, k) for (n, k) in ((3456, 1280), (8192, 8192)) for m in (1, 8, 27)]


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic_layer_step_16384x3456x1280.md")


def csrc_digest():
    """sha256 over the CUDA sources, in name order: a captured traffic figure
    only describes the kernels it was taken from."""
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "ternary_weight_int8_t3_gb300", "csrc")
    for name in sorted(os.listdir(d)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(d, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def dram_traffic(product):
    """DRAM bytes (read + write) per launch of `product` from the committed ncu
    summary, or None when it is absent or the kernels changed since."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    digest, per = None, {}
    with open(TRAFFIC_FILE) as f:
        for line in f:
            line = line.strip().strip("`")
            if line.startswith("csrc_sha256:"):
                digest = line.split(":", 1)[1].strip()
            elif line.startswith("dram_bytes_per_launch:"):
                for item in line.split(":", 1)[1].split(","):
                    k, v = item.strip().split("=")
                    per[k] = int(v)
    if digest != csrc_digest():
        return None
    return per.get(product)


def bench_small_m(t3, torch, dev, stream, hbm_gbs, reps=30, configs=None):
    """Small-M forward sweep: bytes moved (packed weights + activations + the
    int32 output) per call over its device time.  Enough distinct copies of Wp
    rotate through the calls that no copy is still in the 129 MB L2.  The calls
    are captured once in a CUDA graph and replayed, so the device time is not
    hidden behind host launch overhead (a call is a kernel that zeroes C plus
    the product kernel)."""
    out = []
    for (m, n, k) in (configs or SMALL_M):
        wl = t3_synth.BY_NAME[f"skinny_m{m}_n{n}_k{k}"]
        A, w, _ = t3_synth.make_inputs(wl)
        wp = t3.t3_pack_ternary(w)
        copies = max(2, -(-2 * 129 * 2**20 // wp.nbytes))
        wp_d = torch.from_numpy(wp).to(dev)
        wps = [wp_d.clone() for _ in range(copies)]
        A_d = torch.from_numpy(A).to(dev)
        C = torch.empty((m, n), dtype=torch.int32, device=dev)
        for i in range(3):
            t3.t3_gemm_fwd(A_d, wps[i % copies], K=k, C=C, stream=stream)
        torch.cuda.synchronize(dev)
        mode = "graph"
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for i in range(reps):
                    t3.t3_gemm_fwd(A_d, wps[i % copies], K=k, C=C)
            run = g.replay
        except Exception:  # capture unsupported here: time the eager calls
            mode = "eager"
            def run():
                for i in range(reps):
                    t3.t3_gemm_fwd(A_d, wps[i % copies], K=k, C=C, stream=stream)
        run()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        us = e0.elapsed_time(e1) * 1e3 / reps
        nbytes = wp.nbytes + A.nbytes + m * n * 4
        gbs = nbytes / (us * 1e-6) / 1e9
        out.append({"M": m, "N": n, "K": k, "us_per_call": round(us, 3), "bytes": nbytes,
                    "GBps": round(gbs, 1), "frac_hbm": round(gbs / hbm_gbs, 3),
                    "TOPS": round(2 * m * n * k / (us * 1e-6) / 1e12, 2), "timing": mode})
        del wps
    return out


def launch_floor_us(torch, dev, reps=30):
    """Per-call floor of the small-M timing: a one-element fill kernel
    captured `reps` times in a CUDA graph and replayed, so that each call
    costs only a launch and an empty grid's run, timed like the small-M calls."""
    x = torch.zeros(1, dtype=torch.int32, device=dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(reps):
            x.fill_(i)
    g.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize(dev)
    return round(e0.elapsed_time(e1) * 1e3 / reps, 3)


PACK_SHAPES = [(1280, 3456), (8192, 8192)]


def bench_scaled(t3, torch, dev, stream, A_d, wp_d, dY_d, K, reps=10):
    """The layer step's three products with scaled float output (row scales
    per output row, column scales per output column): fwd and dX scale in the
    pair pipeline's epilogue, dW converts its exact int32 result in place."""
    M, N = A_d.shape[0], wp_d.shape[0]
    g = torch.Generator(device="cpu").manual_seed(99)
    def sc(n):
        return (torch.randn(n, generator=g) * 0.01).to(dev)
    rs_m, cs_n, cs_k, rs_k = sc(M), sc(N), sc(K), sc(K)
    C = torch.empty((M, N), dtype=torch.float32, device=dev)
    dX = torch.empty((M, K), dtype=torch.float32, device=dev)
    dW = torch.empty((K, N), dtype=torch.float32, device=dev)
    dW16 = torch.empty((K, N), dtype=torch.bfloat16, device=dev)
    ws = torch.empty((K, N), dtype=torch.int32, device=dev)
    calls = {
        "fwd": lambda: t3.t3_gemm_fwd_scaled(A_d, wp_d, K, rs_m, cs_n, t3.T3_OUT_F32, C=C, stream=stream),
        "dx": lambda: t3.t3_gemm_bwd_dx_scaled(dY_d, wp_d, K, rs_m, cs_k, t3.T3_OUT_F32, dX=dX,
                                               stream=stream),
        "dw": lambda: t3.t3_gemm_bwd_dw_scaled(A_d, dY_d, rs_k, cs_n, t3.T3_OUT_F32, dW=dW,
                                               stream=stream),
        # bf16 dW: the exact int32 product goes through a caller-owned workspace
        "dw_bf16_workspace": lambda: t3.t3_gemm_bwd_dw_scaled(
            A_d, dY_d, rs_k, cs_n, t3.T3_OUT_BF16, dW=dW16, workspace=ws, stream=stream),
    }
    out = {}
    for name, call in calls.items():
        for _ in range(3):
            call()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            call()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / reps
        out[name] = {"us": round(ms * 1e3, 1), "TOPS": round(OPS_PER_PRODUCT / (ms * 1e-3) / 1e12, 1)}
    return out


def bench_device_pack(t3, torch, dev, stream, hbm_gbs, reps=20):
    """Device packer sweep: bytes moved (w in, Wp out) per call over its device
    time.  Enough distinct copies of w rotate through the calls that no copy is
    still in the 129 MB L2; the calls are replayed from a CUDA graph."""
    out = []
    for (k, n) in PACK_SHAPES:
        g = t3_synth.rng(4242 + k + n)
        w = t3_synth.ternary(g, (k, n))
        copies = max(2, -(-2 * 129 * 2**20 // w.nbytes))
        w_d = torch.from_numpy(w).to(dev)
        ws = [w_d.clone() for _ in range(copies)]
        wp = torch.empty((n, (k + 3) // 4), dtype=torch.uint8, device=dev)
        for i in range(3):
            t3.t3_pack_ternary_device(ws[i % copies], wp, stream=stream)
        torch.cuda.synchronize(dev)
        g_ = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_):
            for i in range(reps):
                t3.t3_pack_ternary_device(ws[i % copies], wp)
        g_.replay()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g_.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        us = e0.elapsed_time(e1) * 1e3 / reps
        nbytes = w.nbytes + wp.numel()
        gbs = nbytes / (us * 1e-6) / 1e9
        out.append({"K": k, "N": n, "us_per_call": round(us, 3), "bytes": nbytes,
                    "GBps": round(gbs, 1), "frac_hbm": round(gbs / hbm_gbs, 3), "timing": "graph"})
        del ws
    return out


def bench_quantize(t3, torch, dev, stream, hbm_gbs, M, K, reps=20):
    """Row quantizer at the layer's activation shape: bytes moved (bf16 in,
    int8 and row scales out) per call over its device time, inputs rotated
    past the L2, calls replayed from a CUDA graph."""
    g = torch.Generator(device="cpu").manual_seed(7)
    x = (torch.randn((M, K), generator=g) * 3).to(torch.bfloat16).to(dev)
    copies = max(2, -(-2 * 129 * 2**20 // (x.numel() * 2)))
    xs = [x.clone() for _ in range(copies)]
    q = torch.empty((M, K), dtype=torch.int8, device=dev)
    sc = torch.empty((M,), dtype=torch.float32, device=dev)
    for i in range(3):
        t3.t3_quantize_rows_bf16(xs[i % copies], q, sc, stream=stream)
    torch.cuda.synchronize(dev)
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        for i in range(reps):
            t3.t3_quantize_rows_bf16(xs[i % copies], q, sc)
    gr.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    gr.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    us = e0.elapsed_time(e1) * 1e3 / reps
    nbytes = M * K * 2 + M * K + M * 4
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"M": M, "K": K, "us_per_call": round(us, 3), "bytes": nbytes, "GBps": round(gbs, 1),
            "frac_hbm": round(gbs / hbm_gbs, 3), "timing": "graph"}


def bench_fused_quant(t3, torch, dev, stream, wp_d, reps=10):
    """The row quantizer and the forward at the layer shape, two ways: the
    quantizer kernel and then the forward on its int8 output (two passes over
    the bf16 activations, int8 written and read back), and the quantizer fused
    into the forward (a scales-only pass, then the forward's converters
    quantize the bf16 tiles).  bf16 inputs rotate past the L2."""
    g = torch.Generator(device="cpu").manual_seed(11)
    x = (torch.randn((M, K), generator=g) * 3).to(torch.bfloat16).to(dev)
    copies = max(2, -(-2 * 129 * 2**20 // (x.numel() * 2)))
    xs = [x.clone() for _ in range(copies)]
    q = torch.empty((M, K), dtype=torch.int8, device=dev)
    sc = torch.empty((M,), dtype=torch.float32, device=dev)
    inv = torch.empty((M,), dtype=torch.float32, device=dev)
    C = torch.empty((M, N), dtype=torch.int32, device=dev)

    def unfused(i):
        t3.t3_quantize_rows_bf16(xs[i % copies], q, sc, stream=stream)
        t3.t3_gemm_fwd(q, wp_d, K=K, C=C, stream=stream)

    def fused(i):
        t3.t3_gemm_fwd_bf16(xs[i % copies], wp_d, C=C, row_scale=sc, row_inv=inv, stream=stream)

    out = {}
    for name, call in (("quantize_then_fwd", unfused), ("fused_fwd_bf16", fused)):
        for i in range(3):
            call(i)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(reps):
            call(i)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        us = e0.elapsed_time(e1) * 1e3 / reps
        out[name] = {"us": round(us, 1), "TOPS": round(OPS_PER_PRODUCT / (us * 1e-6) / 1e12, 1)}
    return out


# The pages' own forward timings of the shapes in their throughput table, in
# ms per call on an RTX 4090 (launch overhead included): "t27c PTX backend:
# ternary x int8 GEMM kernel emitted by a .t27 spec", section "Measured: RTX
# 4090".  Context for the same shapes timed here, not a target.
PAGES_FWD_MS = {(4096, 3456, 1280): 0.2211, (4096, 1280, 3456): 0.2538,
                (4096, 1280, 1280): 0.0997, (16384, 3456, 1280): 0.8487,
                (16384, 1280, 3456): 0.8345, (16384, 1280, 1280): 0.3359}


def bench_configs(t3, torch, dev, stream, peak, reps=20,
                  names=("fwd_square_4096", "bwd_1782x3456x1280")):
    """The other full-size workloads, each product timed on its own: the
    square forward 4096^3 (weights P(0) = 1/2) and the backward of the pages'
    1782-row layer (dX over N = 3456, dW over the 1782 rows), or the workloads
    named.  Enough sets of buffers rotate through the calls that none is still
    in the 129 MB L2."""
    out = {}
    for name in names:
        wl = t3_synth.BY_NAME[name]
        A, w, dY = t3_synth.make_inputs(wl)
        wp = t3.t3_pack_ternary(w)
        m, n, k = wl.M, wl.N, wl.K
        prods = {"fwd": (m * k + wp.nbytes + 4 * m * n)} if wl.op == "fwd" else {
            "dx": m * n + wp.nbytes + 4 * m * k, "dw": m * k + m * n + 4 * k * n}
        for prod, nbytes in prods.items():
            sets = max(2, -(-2 * 129 * 2**20 // nbytes))
            bufs = []
            for _ in range(sets):
                if prod == "fwd":
                    bufs.append((torch.from_numpy(A).to(dev), torch.from_numpy(wp).to(dev),
                                 torch.empty((m, n), dtype=torch.int32, device=dev)))
                elif prod == "dx":
                    bufs.append((torch.from_numpy(dY).to(dev), torch.from_numpy(wp).to(dev),
                                 torch.empty((m, k), dtype=torch.int32, device=dev)))
                else:
                    bufs.append((torch.from_numpy(A).to(dev), torch.from_numpy(dY).to(dev),
                                 torch.empty((k, n), dtype=torch.int32, device=dev)))

            def call(b):
                x, y, o = b
                if prod == "fwd":
                    t3.t3_gemm_fwd(x, y, K=k, C=o, stream=stream)
                elif prod == "dx":
                    t3.t3_gemm_bwd_dx(x, y, k, dX=o, stream=stream)
                else:
                    t3.t3_gemm_bwd_dw(x, y, dW=o, stream=stream)
            for i in range(max(3, sets)):
                call(bufs[i % sets])
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(reps):
                call(bufs[i % sets])
            e1.record(stream)
            torch.cuda.synchronize(dev)
            us = e0.elapsed_time(e1) * 1e3 / reps
            tops = 2 * m * n * k / (us * 1e-6) / 1e12
            out[f"{prod} {m}x{n}x{k}"] = {"us": round(us, 2), "TOPS": round(tops, 1),
                                          "frac": round(tops / peak, 3), "buffer_sets": sets}
            del bufs
    return out


# The layer widths of the pages' HSLM backward measurements (243 and 729, at
# 27 and 1782 rows): rows of 243 and 729 bytes, not word-aligned.
HSLM_SHAPES = [(m, n, k) for m in (27, 1782) for (n, k) in ((729, 243), (243, 729))]


def bench_hslm(t3, torch, dev, peak, reps=20, max_sets=64, shapes=None):
    """fwd, dX and dW at the HSLM widths, each product's calls captured in a
    CUDA graph and replayed (these products take microseconds: without the
    graph the host's launch rate would be timed).  Up to `max_sets` buffer
    sets rotate through the calls; `set_bytes` x `buffer_sets` says whether
    that rotation outgrows the 129 MB L2 (the 27-row shapes stay resident)."""
    out = {}
    for (m, n, k) in (shapes or HSLM_SHAPES):
        g = t3_synth.rng(m + n + k)
        A = t3_synth.int8_uniform(g, (m, k))
        dY = t3_synth.int8_uniform(g, (m, n))
        wp = t3.t3_pack_ternary(t3_synth.ternary(g, (k, n)))
        set_bytes = A.nbytes + dY.nbytes + wp.nbytes + 4 * (m * n + m * k + k * n)
        sets = int(min(max_sets, max(2, -(-2 * 129 * 2**20 // set_bytes))))
        bufs = [(torch.from_numpy(A).to(dev), torch.from_numpy(dY).to(dev), torch.from_numpy(wp).to(dev),
                 torch.empty((m, n), dtype=torch.int32, device=dev),
                 torch.empty((m, k), dtype=torch.int32, device=dev),
                 torch.empty((k, n), dtype=torch.int32, device=dev)) for _ in range(sets)]
        row = {"buffer_sets": sets, "set_bytes": set_bytes}
        for prod in ("fwd", "dx", "dw"):
            def call(b):
                a_d, dy_d, wp_d, c_d, dx_d, dw_d = b
                if prod == "fwd":
                    t3.t3_gemm_fwd(a_d, wp_d, K=k, C=c_d)
                elif prod == "dx":
                    t3.t3_gemm_bwd_dx(dy_d, wp_d, k, dX=dx_d)
                else:
                    t3.t3_gemm_bwd_dw(a_d, dy_d, dW=dw_d)
            for i in range(3):
                call(bufs[i % sets])
            torch.cuda.synchronize(dev)
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr):
                for i in range(reps):
                    call(bufs[i % sets])
            gr.replay()
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            gr.replay()
            e1.record()
            torch.cuda.synchronize(dev)
            us = e0.elapsed_time(e1) * 1e3 / reps
            tops = 2 * m * n * k / (us * 1e-6) / 1e12
            row[prod] = {"us": round(us, 2), "TOPS": round(tops, 2), "frac": round(tops / peak, 4)}
            del gr
        out[f"{m}x{n}x{k}"] = row
        del bufs
    return out


def cpu_baseline(A, w, dY, target_s=15.0):
    """The oracle, as it stands, on a bounded sample of rows of each product."""
    import oracle
    wp = oracle.pack(w)
    total_ops, total_t, sample = 0, 0.0, []
    per_op = target_s / 3.0
    for name in ("fwd", "dx", "dw"):
        rows_probe = 32 if name != "dw" else 4
        def run(nrows):
            rows = np.linspace(0, (M if name != "dw" else K) - 1, nrows).astype(np.int64)
            t0 = time.perf_counter()
            if name == "fwd":
                oracle.fwd(A, wp, rows)
                ops = 2 * nrows * N * K
            elif name == "dx":
                oracle.dx(dY, wp, K, rows)
                ops = 2 * nrows * N * K
            else:
                oracle.dw(A, dY, rows)
                ops = 2 * nrows * N * M
            return ops, time.perf_counter() - t0
        ops, t = run(rows_probe)
        nrows = max(rows_probe, int(rows_probe * per_op / max(t, 1e-4)))
        nrows = min(nrows, M if name != "dw" else K)
        ops, t = run(nrows)
        total_ops += ops
        total_t += t
        sample.append(f"{name}: {nrows} output rows")
    return {"value": total_ops / total_t / 1e12, "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle", "sample": "; ".join(sample) + f" of the {WORKLOAD} ({total_t:.1f} s)"}


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: each step a bounded row sample."""
    if rank != 0:
        return
    import oracle
    A, w, dY = make_host_inputs()
    wp = oracle.pack(w)
    rows_fwd = np.linspace(0, M - 1, 6).astype(np.int64)
    rows_dw = np.linspace(0, K - 1, 6).astype(np.int64)
    ops_step = 2 * len(rows_fwd) * N * K * 2 + 2 * len(rows_dw) * N * M

    def step():
        oracle.fwd(A, wp, rows_fwd)
        oracle.dx(dY, wp, K, rows_fwd)
        oracle.dw(A, dY, rows_dw)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = ops_step * args.steps / el / 1e12
    sample = (f"per step: fwd and dX on {len(rows_fwd)} rows each, dW on {len(rows_dw)} rows, "
              f"of the {WORKLOAD}")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": sample},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, local_rank, world = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    import ternary_weight_int8_t3_gb300 as t3

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    if args.hslm_only:
        cfg = tuple(int(x) for x in args.hslm_only.split(","))
        if cfg not in HSLM_SHAPES:
            raise SystemExit(f"--hslm-only: {cfg} is not one of {HSLM_SHAPES}")
        peak = read_peaks()[0].get("bf16_tflops", 1900.0)
        print(json.dumps({"hslm_shapes": bench_hslm(t3, torch, dev, peak, shapes=[cfg])}))
        return

    if args.small_m_only:
        cfg = tuple(int(x) for x in args.small_m_only.split(","))
        if cfg not in SMALL_M:
            raise SystemExit(f"--small-m-only: {cfg} is not one of {SMALL_M}")
        peaks, _ = read_peaks()
        hbm = peaks.get("hbm_gbs", 6800.0)
        calls = bench_small_m(t3, torch, dev, torch.cuda.current_stream(dev), hbm,
                              configs=[cfg])
        print(json.dumps({"small_m": {"hbm_peak_GBps": hbm, "calls": calls}}))
        return

    A, w, dY = make_host_inputs()
    wp = t3.t3_pack_ternary(w)
    A_d = torch.from_numpy(A).to(dev)
    wp_d = torch.from_numpy(wp).to(dev)
    dY_d = torch.from_numpy(dY).to(dev)
    C = torch.empty((M, N), dtype=torch.int32, device=dev)
    dX = torch.empty((M, K), dtype=torch.int32, device=dev)
    dW = torch.empty((K, N), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        t3.t3_gemm_fwd(A_d, wp_d, K=K, C=C, stream=stream)
        t3.t3_gemm_bwd_dx(dY_d, wp_d, K, dX=dX, stream=stream)
        t3.t3_gemm_bwd_dw(A_d, dY_d, dW=dW, stream=stream)

    def barrier():
        torch.cuda.synchronize(dev)
        if pg is not None:
            pg.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(max(args.warmup, 3)):
        step()
    barrier()

    # ---- device-resident timed region, per-product events on the launch stream
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks:
        barrier()
        start.record(stream)
        for i in range(args.steps):
            e = ev[i]
            e[0].record(stream)
            t3.t3_gemm_fwd(A_d, wp_d, K=K, C=C, stream=stream)
            e[1].record(stream)
            t3.t3_gemm_bwd_dx(dY_d, wp_d, K, dX=dX, stream=stream)
            e[2].record(stream)
            t3.t3_gemm_bwd_dw(A_d, dY_d, dW=dW, stream=stream)
            e[3].record(stream)
        stop.record(stream)
        barrier()
    elapsed_ms = start.elapsed_time(stop)
    per = {"fwd": [], "dx": [], "dw": []}
    for e in ev:
        per["fwd"].append(e[0].elapsed_time(e[1]))
        per["dx"].append(e[1].elapsed_time(e[2]))
        per["dw"].append(e[2].elapsed_time(e[3]))
    rc, detail = t3.t3_last_device_error()
    if rc != t3.T3_OK:
        raise RuntimeError(f"device wait timed out during the bench ({detail:#x})")

    elapsed_max = max_over_ranks(elapsed_ms, pg, dev)

    # ---- end to end: pinned host inputs in, results out, every step
    A_h = torch.from_numpy(A).pin_memory()
    wp_h = torch.from_numpy(wp).pin_memory()
    dY_h = torch.from_numpy(dY).pin_memory()
    C_h = torch.empty((M, N), dtype=torch.int32).pin_memory()
    dX_h = torch.empty((M, K), dtype=torch.int32).pin_memory()
    dW_h = torch.empty((K, N), dtype=torch.int32).pin_memory()
    e2e_steps = max(3, min(args.steps, 10))
    # Pipelined over steps: each step copies its inputs in and all three results
    # out, on streams of their own, so that copies overlap the kernels and each
    # other; two sets of device buffers alternate, and events order every reuse
    # (inputs are overwritten only after the kernels that read them finished,
    # outputs only after the copy out of their previous contents finished).
    sets = [(A_d, wp_d, dY_d, C, dX, dW),
            (torch.empty_like(A_d), torch.empty_like(wp_d), torch.empty_like(dY_d),
             torch.empty_like(C), torch.empty_like(dX), torch.empty_like(dW))]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_names = ("a_in", "dy_in", "c_done", "dx_done", "kern_done", "out_done")
    evs = [{n: torch.cuda.Event() for n in ev_names} for _ in sets]
    used = [False, False]

    def e2e_step(i):
        b = i % 2
        a_d, w_d, y_d, c_d, x_d, g_d = sets[b]
        e = evs[b]
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(e["kern_done"])  # the last kernels reading this set
            a_d.copy_(A_h, non_blocking=True)
            w_d.copy_(wp_h, non_blocking=True)
            e["a_in"].record(s_in)
            y_d.copy_(dY_h, non_blocking=True)
            e["dy_in"].record(s_in)
        stream.wait_event(e["a_in"])
        if used[b]:
            stream.wait_event(e["out_done"])  # the last copy out of this set's outputs
        t3.t3_gemm_fwd(a_d, w_d, K=K, C=c_d, stream=stream)
        e["c_done"].record(stream)
        stream.wait_event(e["dy_in"])
        t3.t3_gemm_bwd_dx(y_d, w_d, K, dX=x_d, stream=stream)
        e["dx_done"].record(stream)
        t3.t3_gemm_bwd_dw(a_d, y_d, dW=g_d, stream=stream)
        e["kern_done"].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(e["c_done"])
            C_h.copy_(c_d, non_blocking=True)
            s_out.wait_event(e["dx_done"])
            dX_h.copy_(x_d, non_blocking=True)
            s_out.wait_event(e["kern_done"])
            dW_h.copy_(g_d, non_blocking=True)
            e["out_done"].record(s_out)
        used[b] = True

    def e2e_join():
        for sd in (s_in, s_out):
            ev_j = torch.cuda.Event()
            ev_j.record(sd)
            stream.wait_event(ev_j)

    e2e_step(0)
    e2e_step(1)
    e2e_join()
    torch.cuda.synchronize()
    barrier()
    s2, t2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s2.record(stream)
    s_in.wait_event(s2)
    s_out.wait_event(s2)
    for i in range(e2e_steps):
        e2e_step(i)
    e2e_join()
    t2.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = max_over_ranks(s2.elapsed_time(t2) / e2e_steps, pg, dev)
    h2d = A.nbytes + wp.nbytes + dY.nbytes
    d2h = (M * N + M * K + K * N) * 4

    if rank != 0:
        if pg is not None:
            pg.destroy_process_group()
        return

    ms_step = elapsed_max / args.steps
    value = job_tops(ms_step, world)
    avg = {k: sum(v) / len(v) for k, v in per.items()}
    op_tops = {k: OPS_PER_PRODUCT / (avg[k] * 1e-3) / 1e12 for k in avg}
    dominant = max(avg, key=avg.get)
    peaks, peak_src = read_peaks()
    long_region = elapsed_ms > 1000.0
    if peak_src == "measured":
        peak = peaks.get("bf16_tflops_sustained" if long_region else "bf16_tflops", FALLBACK_TFLOPS)
        peak_note = ("sustained" if long_region else "burst") + " bf16 dense of measured; f16 runs at the bf16 rate"
    else:
        peak, peak_note = FALLBACK_TFLOPS, "bf16 dense of fallback; f16 runs at the bf16 rate"
    traffic = dram_traffic(dominant)
    kname = {"fwd": "t3_gemm_fwd", "dx": "t3_gemm_bwd_dx", "dw": "t3_gemm_bwd_dw"}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K, "seed": SEED,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "arith": "int8 x ternary (and int8 x int8) -> exact int32 via f16 tcgen05 operands, f32 TMEM accumulation",
                   "l2": "per-step traffic ~410 MB > 129 MB L2; no flush",
                   "context": PAGES_CONTEXT},
        "per_product_tops": op_tops,
        "per_product_ms": avg,
        "roofline": {"kernel": kname[dominant], "bound": "tensor", "achieved": op_tops[dominant],
                     "peak": peak, "unit": "TFLOP/s", "frac": op_tops[dominant] / peak,
                     "traffic": traffic, "peak_source": peak_note,
                     "stated_int8_peak": STATED_INT8_TOPS,
                     "frac_of_stated_int8_peak": op_tops[dominant] / STATED_INT8_TOPS,
                     "peak_choice": "ptxas rejects tcgen05.mma kind::i8 for sm_103a, so the "
                                    "products run as exact f16 tensor-core MMAs and the f16/bf16 "
                                    "peak is their roofline; the stated ~4.5 POPS int8 rate does "
                                    "not exist on this chip"},
        "gpu_launches": 4 * args.steps,  # fwd, dX, dW zeroing + dW product
        "e2e": {"value": job_tops(e2e_ms, world), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "pinned host buffers; every step copies its inputs in and C, dX, dW out "
                       "on streams of their own, overlapping the kernels and each other (two "
                       "device buffer sets alternate)"},
        "clocks": clocks.summary(),
    }
    hbm = peaks.get("hbm_gbs", 6800.0) if peak_src == "measured" else 6800.0
    if not args.step_only:
        line["scaled_f32"] = bench_scaled(t3, torch, dev, stream, A_d, wp_d, dY_d, K)
        line["quantize_rows"] = bench_quantize(t3, torch, dev, stream, hbm, M, K)
        line["quantized_fwd_bf16"] = bench_fused_quant(t3, torch, dev, stream, wp_d)
    if not args.step_only:
        line["configs"] = bench_configs(t3, torch, dev, stream, peak)
        pages = bench_configs(t3, torch, dev, stream, peak,
                              names=[f"fwd_{m}x{n}x{k}" for (m, n, k) in t3_synth.PAGES_FWD_SHAPES])
        pages[f"fwd {M}x{N}x{K}"] = {"us": round(avg["fwd"] * 1e3, 2),
                                     "TOPS": round(op_tops["fwd"], 1),
                                     "frac": round(op_tops["fwd"] / peak, 3),
                                     "timing": "the layer step's forward"}
        for key, v in pages.items():
            shape = tuple(int(x) for x in key.split()[1].split("x"))
            v["pages_rtx4090_us"] = round(PAGES_FWD_MS[shape] * 1e3, 1)
        line["pages_fwd_shapes"] = pages
        line["hslm_shapes"] = bench_hslm(t3, torch, dev, peak)
    if not (args.no_pack or args.step_only):
        line["device_pack"] = {"hbm_peak_GBps": hbm, "calls": bench_device_pack(t3, torch, dev, stream, hbm)}
    if not (args.no_small_m or args.step_only):
        line["small_m"] = {"hbm_peak_GBps": hbm, "calls": bench_small_m(t3, torch, dev, stream, hbm),
                           "launch_floor_us": launch_floor_us(torch, dev)}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(A, w, dY)
    print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
