#!/usr/bin/env python
"""Benchmark of the GB300 TetraJet-v2 NVFP4 linear path.

One step = the ~370M-class decoder-layer linear set on 16384 tokens (QKV
1024->3072, out-proj 1024->1024, SwiGLU gate/up 1024->2x4096, down 4096->1024;
10% of each layer's input channels kept in FP8 by OutControl), forward + dX + dW
through the C ABI, followed by one OsciReset pass over 369,098,752 fp32 master
weights (cosine learning-rate schedule 1e-3 -> 1e-5 over 200 steps, reset
threshold lr < 1e-4 and risk > 4).

value  = linear-set fwd+bwd algorithmic TFLOP/s (6 * M * sum N*K per step) over
         the time of the linear calls, inputs resident in HBM;
e2e    = the same with X and dY copied host->device from pinned memory and dW
         copied back every step;
parts  = per-call times; the OsciReset pass and the quantize sweep in GB/s.
Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "NVFP4 linear fwd+bwd TFLOP/s & quantize GB/s, as fraction of GB300 roofline"
WORKLOAD = ("layer_set_370M: decoder-layer linear set QKV 1024->3072, out 1024->1024, gate/up 1024->8192, "
            "down 4096->1024 on 16384 tokens, 10% FP8 outlier channels, fwd+dX+dW; plus OsciReset over "
            "369,098,752 fp32 master weights per step")
TOKENS = 16384
OUTLIER_PCT = 10
LR_THR, RISK_THR = 1e-4, 4.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def linear_flops(M=TOKENS):
    from nvfp4_bit_fully_gb300.workloads import LAYER_SET

    return 6.0 * M * sum(n * k for _, n, k in LAYER_SET)


def osci_bytes_per_elem():
    # read w, w_prev, dist_Q, dist_M (4 B each) + previous Q (0.5 + 1/16 + 4/128 B);
    # write w_prev, dist_Q, dist_M + new Q + 1 mask bit (w itself only on reset)
    q = 0.5 + 1.0 / 16 + 4.0 / 128
    return (16 + q) + (12 + q + 1.0 / 8)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1].split()[0]))
                    smax.append(float(parts[2].split()[0]))
                    power.append(float(parts[3].split()[0]))
                except ValueError:
                    continue
                for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                                     parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# the step
# ---------------------------------------------------------------------------
class Timeline:
    """CUDA events around every C-ABI call of a step, on the launching stream."""

    def __init__(self, stream):
        self.stream = stream
        self.records = []

    def time(self, name, fn):
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(self.stream)
        out = fn()
        e.record(self.stream)
        self.records.append((name, s, e))
        return out

    def summary(self):
        agg = {}
        for name, s, e in self.records:
            agg.setdefault(name, []).append(s.elapsed_time(e))
        return {k: (float(np.sum(v)), len(v)) for k, v in agg.items()}


# kernel behind each step call (for per-kernel aggregation of the live event times)
CALL_KERNEL = {
    "quant_x": "k_quant_split (OutControl split of X)", "quant_dy_row": "k_quant_rows (NVFP4 + MXFP8 of dY)",
    "quant_dy_col": "k_quant_cols (NVFP4 + MXFP8 of dY)",
    "requant_w": "k_realign_pair (re-align NVFP4 + slice)", "requant_x": "k_realign_pair (re-align NVFP4 + slice)",
    "gemm_fwd": "k_gemm_nvfp4", "gemm_dx": "k_gemm_nvfp4", "gemm_dw": "k_gemm_nvfp4",
    "osci_reset": "k_osci_reset",
}


class Linear:
    """One linear of the layer set: inputs, calibrated outlier set, forward weight
    operands and every output / intermediate buffer, all resident in HBM.

    run() issues the step as the individual C-ABI calls that tj_linear_fwd /
    tj_linear_bwd_dx / tj_linear_bwd_dw make internally (same kernels, same order),
    so every kernel gets its own CUDA events in the timed region."""

    def __init__(self, tj, wl, name, N, K, dev, seed):
        self.name, self.N, self.K = name, N, K
        self.X, self.W, self.dY = wl.device_layer_set_linear(name, N, K, seed=seed, M=TOKENS, device=dev)
        W = self.W
        self.k = (OUTLIER_PCT * K + 99) // 100
        # OutControl calibration: 4 warm-up batches with fixed heavy channels (cold path)
        sumsq = torch.zeros(K, dtype=torch.float64, device=dev)
        for b in range(4):
            xb = wl.device_calibration_batch(K, TOKENS, 20, b, seed, 700 + K, dev)
            tj.outlier_calibrate(xb, sumsq)
            del xb
        self.oi, self.ni = tj.outlier_calibrate(None, sumsq, finalize=True, k=self.k)
        self.wq = tj.quantize_nvfp4(W, sel=self.ni)
        self.w8 = tj.quantize_mxfp8(W, sel=self.oi)
        M, kn, k = TOKENS, K - self.k, self.k
        self.xq, self.x8 = tj.NVFP4.empty(M, kn, dev), tj.MXFP8.empty(M, k, dev)
        self.s_dy, self.s_w = tj.NVFP4.empty(M, N, dev), tj.NVFP4.empty(kn, N, dev)
        self.q8_dy, self.q8_w = tj.MXFP8.empty(M, N, dev), tj.MXFP8.empty(k, N, dev)
        self.s_dyt, self.s_x = tj.NVFP4.empty(N, M, dev), tj.NVFP4.empty(kn, M, dev)
        self.q8_dyt, self.q8_x = tj.MXFP8.empty(N, M, dev), tj.MXFP8.empty(k, M, dev)
        self.Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        self.dX = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
        self.dW = torch.empty(N, K, dtype=torch.float32, device=dev)
        self.ws_dx = torch.empty(tj.workspace_size(tj.TJ_OP_BWD_DX, M, N, K, k), dtype=torch.uint8, device=dev)
        self.ws_dw = torch.empty(tj.workspace_size(tj.TJ_OP_BWD_DW, M, N, K, k), dtype=torch.uint8, device=dev)
        self.flops = 6.0 * M * N * K
        # algorithmic work of every call: (FP4 flops, FP8 flops) or bytes
        f4 = lambda a, b, c: 2.0 * a * b * c
        # operand and output bytes of each GEMM launch (NVFP4 / MXFP8 operands, bf16 Y and dX,
        # fp32 dW)
        self.gemm_bytes = {
            "gemm_fwd": (M + N) * (kn * NV_B + k * MX_B) + M * N * 2,
            "gemm_dx": M * N * (NV_B + MX_B) + N * (kn * NV_B + k * MX_B) + M * K * 2,
            "gemm_dw": N * M * (NV_B + MX_B) + M * (kn * NV_B + k * MX_B) + N * K * 4,
        }
        self.work = {
            "gemm_fwd": (f4(M, N, kn), f4(M, N, k)), "gemm_dx": (f4(M, kn, N), f4(M, k, N)),
            "gemm_dw": (f4(N, kn, M), f4(N, k, M)),
            "quant_x": M * kn * (2 + NV_B) + M * k * (2 + MX_B),
            "quant_dy_row": M * N * (2 + NV_B + MX_B), "quant_dy_col": M * N * (2 + NV_B + MX_B),
            "requant_w": 2 * kn * N * NV_B + 2 * k * N * MX_B, "requant_x": 2 * kn * M * NV_B + 2 * k * M * MX_B,
        }
        # lane instructions of each quantize call (per-element counts x elements, for the issue
        # roofline); a re-alignment pair launch counts the elements of the NVFP4 operand and of
        # its slice together (its count is measured at the same 10% slice share)
        li = LANE_INSTR_PER_ELEM
        self.lane_instr = {"quant_x": li["split"] * M * K, "quant_dy_row": li["rows"] * M * N,
                           "quant_dy_col": li["cols"] * M * N,
                           "requant_w": li["realign_pair"] * (kn + k) * N,
                           "requant_x": li["realign_pair"] * (kn + k) * M}

    def run(self, tj, seed, tl, stream):
        T = lambda name, fn: tl.time(self.name + "." + name, fn)
        s = stream
        SR = tj.TJ_SR
        # forward (tj_linear_fwd)
        # the OutControl split of X: NVFP4 normal channels + MXFP8 outlier channels, one read
        T("quant_x", lambda: tj.quantize_split(self.X, self.ni, self.oi, out=self.xq, out8=self.x8, stream=s))
        T("gemm_fwd", lambda: tj.gemm_nvfp4(self.xq, self.wq, self.x8, self.w8, out=self.Y, stream=s))
        # input gradient (tj_linear_bwd_dx)
        # dY rows: the SR + RHT operand of dX and the MXFP8 rows of dY from one read
        T("quant_dy_row", lambda: tj.quantize_nvfp4_mxfp8(self.dY, mode=SR, rht=True, seed=seed, tag=tj.TAG_DY_ROW,
                                                          rht_tag=tj.TAG_RHT_DX, out=self.s_dy, out8=self.q8_dy,
                                                          stream=s))
        # W-hat^T and its slice re-aligned in one launch
        T("requant_w", lambda: tj.requantize_nvfp4_mxfp8(self.wq, self.w8, SR, True, seed, tj.TAG_WT, tj.TAG_RHT_DX,
                                                         out=self.s_w, out8=self.q8_w, stream=s))
        # the FP4 product and its FP8 outlier slice in one launch
        T("gemm_dx", lambda: tj.gemm_pair(self.s_dy, self.s_w, self.q8_dy, self.q8_w, alpha=2.0 ** -7, out=self.dX,
                                          out8=self.dX, col_map=self.ni, col_map8=self.oi, stream=s))
        # weight gradient (tj_linear_bwd_dw)
        T("quant_dy_col", lambda: tj.quantize_nvfp4_mxfp8(self.dY, along_cols=True, mode=SR, rht=True, seed=seed,
                                                          tag=tj.TAG_DY_COL, rht_tag=tj.TAG_RHT_DW, out=self.s_dyt,
                                                          out8=self.q8_dyt, stream=s))
        T("requant_x", lambda: tj.requantize_nvfp4_mxfp8(self.xq, self.x8, SR, True, seed, tj.TAG_XT, tj.TAG_RHT_DW,
                                                         out=self.s_x, out8=self.q8_x, stream=s))
        T("gemm_dw", lambda: tj.gemm_pair_f32(self.s_dyt, self.s_x, self.q8_dyt, self.q8_x, self.dW, self.ni, self.oi,
                                              alpha=2.0 ** -7, stream=s))

    def run_api(self, tj, seed, stream):
        """The same step through the user-facing calls (tj_linear_fwd / bwd_dx / bwd_dw)."""
        tj.linear_fwd(self.X, self.wq, self.w8, self.ni, self.oi, xq=self.xq, x8=self.x8, out=self.Y, stream=stream)
        tj.linear_bwd_dx(self.dY, self.wq, self.w8, self.ni, self.oi, seed=seed, workspace=self.ws_dx, out=self.dX,
                         stream=stream)
        tj.linear_bwd_dw(self.dY, self.xq, self.x8, self.ni, self.oi, seed=seed, workspace=self.ws_dw, out=self.dW,
                         stream=stream)


class OsciState:
    """OsciReset state of the master weights: w, w_prev, dist_Q, dist_M, Q double buffer, mask."""

    def __init__(self, tj, wl, n, dev, seed):
        self.w = wl.device_master_weights(n, seed=seed, device=dev)
        self.bytes = n * osci_bytes_per_elem()
        rows, cols = self.w.shape
        self.w_prev = self.w.clone()
        self.dq = torch.zeros_like(self.w)
        self.dm = torch.zeros_like(self.w)
        self.q = [tj.quantize_nvfp4(self.w), tj.NVFP4.empty(rows, cols, dev)]
        self.mask = torch.empty(rows * ((cols + 31) // 32), dtype=torch.int32, device=dev)
        self.n = rows * cols

    def run(self, tj, lr, tl, stream):
        tl.time("osci_reset", lambda: tj.osci_reset(self.w, self.w_prev, self.dq, self.dm, self.q[0], self.q[1],
                                                    self.mask, lr, LR_THR, RISK_THR, True, stream=stream))
        self.q.reverse()


# DRAM bytes per element measured by ncu (dram__bytes_read + write of one capture of the
# current kernel version, divided by its elements), for the HBM-bound kernels; kernels not
# listed report traffic None.  k_osci_reset: 1913.3 MB over 67,108,864 weights.
TRAFFIC_BYTES_PER_ELEM = {"k_osci_reset": 28.55}
# DRAM bytes per launch of the GEMM: the twelve launches of one timed step of the layer set
# at 16384 tokens read 939.9 MB and wrote 363.6 MB (one-pass ncu capture of the current
# kernel), 108.6 MB per launch on average.  Valid for the default workload only.
TRAFFIC_BYTES_PER_LAUNCH = {"k_gemm_nvfp4": 108.6e6}
# Lane instructions per element of the issue-bound quantize kernels (smsp__thread_inst_executed
# of one ncu capture of the current kernel versions, `bench.py --only quant`, divided by the
# elements each launch processes: dY elements for the row / column passes, input elements of
# X for the split, elements of the re-aligned tensors for the re-alignments: the NVFP4 operand
# alone, its slice alone, and both for the pair launch, at 921 + 103 channels).  With them each
# kernel entry reports an issue roofline: lane instructions / (SMs x 128 lanes x SM clock x
# time), the fraction of the SMs' instruction issue the kernel uses.
LANE_INSTR_PER_ELEM = {"rows": 40.89, "cols": 46.29, "split": 27.11, "realign_nv": 48.11, "realign_mx": 28.12,
                      "realign_pair": 47.15}
NV_B = 0.5 + 1.0 / 16 + 4.0 / 128      # bytes per NVFP4 element (codes + E4M3 + FP32 scales)
MX_B = 1.0 + 1.0 / 32                   # bytes per MXFP8 element (E4M3 + UE8M0)


# ---------------------------------------------------------------------------
# secondary measurements (outside the timed step loop)
# ---------------------------------------------------------------------------
def time_kernel(fn, stream, reps=50, flush=None, warmup=10):
    """Median device ms of fn() over reps launches, the L2 flushed before each
    (outside the events).  Every rep is enqueued before the first is waited on,
    so host launch latency never shows up as device time."""
    for _ in range(warmup):
        fn()
    evs = []
    for _ in range(reps):
        if flush is not None:
            with torch.cuda.stream(stream):
                flush.zero_()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn()
        e.record(stream)
        evs.append((s, e))
    torch.cuda.synchronize()
    return float(np.median([s.elapsed_time(e) for s, e in evs]))


def quantize_sweep(tj, dev, stream, hbm_peak, flush):
    """The quantize-only sweep: 4096x1024, 8192x2048, 16384x4096 bf16 inputs, RTN and SR,
    row-wise and transposed alignment; bytes = 2 (read) + 0.59375 (write) per element."""
    from nvfp4_bit_fully_gb300 import workloads as wl

    out = []
    for rows, cols in ((4096, 1024), (8192, 2048), (16384, 4096)):
        x = wl.device_heavy_columns((rows, cols), 1.0, 30.0, math.ceil(cols / 100), 0, 11, dev)
        for along in (False, True):
            q = tj.NVFP4.empty(cols if along else rows, rows if along else cols, dev)
            for mode in (tj.TJ_RTN, tj.TJ_SR):
                ms = time_kernel(lambda: tj.quantize_nvfp4(x, along_cols=along, mode=mode, seed=1, tag=1, out=q,
                                                           stream=stream), stream, 50, flush)
                gbs = rows * cols * (2 + 0.59375) / (ms * 1e-3) / 1e9
                out.append({"shape": [rows, cols], "align": "col" if along else "row",
                            "mode": "SR" if mode else "RTN", "ms": round(ms, 4), "GB/s": round(gbs, 1),
                            "frac": round(gbs / hbm_peak, 3)})
        del x
    return out


def adamw_osci_alone(tj, osci, stream, hbm_peak):
    """The fused training-step pass (AdamW + OsciReset + forward-W quantize, tj_adamw_osci_reset)
    over the same master weights, with a synthetic gradient, timed alone.  Its state is a copy,
    so the step's OsciReset trajectory is untouched."""
    g = torch.randn_like(osci.w) * 1e-2
    m = torch.zeros_like(osci.w)
    v = torch.zeros_like(osci.w)
    w = osci.w.clone()
    w_prev, dq, dm = osci.w_prev.clone(), osci.dq.clone(), osci.dm.clone()
    step = [0]

    def fn():
        step[0] += 1
        tj.adamw_osci_reset(w, g, m, v, w_prev, dq, dm, osci.q[0], osci.q[1], osci.mask, 5e-5, 0.9, 0.95, 1e-8,
                            0.1, step[0], LR_THR, RISK_THR, True, stream=stream)

    ms = time_kernel(fn, stream, 20, warmup=3)
    # read w, g, m, v, w_prev, dist_Q, dist_M + previous Q; write w, m, v, w_prev, dist_Q,
    # dist_M + new Q + 1 mask bit
    nbytes = osci.n * (4 * 7 + NV_B + 4 * 6 + NV_B + 1.0 / 8)
    del g, m, v, w, w_prev, dq, dm
    return {"params": osci.n, "ms": round(ms, 4), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1),
            "frac": round(nbytes / (ms * 1e-3) / 1e9 / hbm_peak, 3), "bytes_per_weight": round(nbytes / osci.n, 4)}


def gemm_alone(tj, lin, stream, fp4_peak, fp8_peak):
    """The largest forward GEMM (FP4 part + FP8 slice in one tile) timed alone."""
    M, N, K, k = TOKENS, lin.N, lin.K, lin.k
    ms = time_kernel(lambda: tj.gemm_nvfp4(lin.xq, lin.wq, lin.x8, lin.w8, out=lin.Y, stream=stream), stream, 50)
    f4 = 2.0 * M * N * (K - k)
    f8 = 2.0 * M * N * k
    t_star = f4 / (fp4_peak * 1e12) + f8 / (fp8_peak * 1e12)          # time at the dtype-weighted peak
    return {"shape": [M, N, K], "k_fp8": k, "ms": round(ms, 4), "TFLOP/s": round((f4 + f8) / (ms * 1e-3) / 1e12, 1),
            "frac_of_peak": round(t_star / (ms * 1e-3), 3)}


def _gemm_frac(f4, f8, ms, fp4_peak, fp8_peak):
    t_star = f4 / (fp4_peak * 1e12) + f8 / (fp8_peak * 1e12)          # time at the dtype-weighted peak
    return {"ms": round(ms, 4), "TFLOP/s": round((f4 + f8) / (ms * 1e-3) / 1e12, 1), "frac": round(t_star / (ms * 1e-3), 4)}


def cfg3_fwd(tj, dev, stream, fp4_peak, fp8_peak):
    """Forward NVFP4 linear with OutControl at its own shape: X 16384 x 1024 (the fifth
    calibration-distribution batch), W 4096 x 1024 N(0, 0.02); the 10% FP8 channels come
    from the calibration kernel over 4 warm-up batches with 20 fixed heavy channels x40.
    Timed through tj_linear_fwd (OutControl split of X + FP4 GEMM with its FP8 slice)."""
    from nvfp4_bit_fully_gb300 import workloads as wl

    M, K, N, seed = TOKENS, 1024, 4096, 1
    k = (OUTLIER_PCT * K + 99) // 100
    sumsq = torch.zeros(K, dtype=torch.float64, device=dev)
    for b in range(4):
        xb = wl.device_calibration_batch(K, M, 20, b, seed, 21, dev)
        torch.cuda.synchronize()
        tj.outlier_calibrate(xb, sumsq, stream=stream)
        torch.cuda.synchronize()
        del xb
    oi, ni = tj.outlier_calibrate(None, sumsq, finalize=True, k=k, stream=stream)
    X = wl.device_calibration_batch(K, M, 20, 4, seed, 21, dev)
    g = wl._cuda_gen(seed, 22, dev)
    W = (torch.randn(N, K, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    torch.cuda.synchronize()
    wq, w8 = tj.quantize_nvfp4(W, sel=ni, stream=stream), tj.quantize_mxfp8(W, sel=oi, stream=stream)
    xq, x8 = tj.NVFP4.empty(M, K - k, dev), tj.MXFP8.empty(M, k, dev)
    Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    f4, f8 = 2.0 * M * N * (K - k), 2.0 * M * N * k
    torch.cuda.synchronize()                 # inputs were drawn on torch's current stream
    ms = time_kernel(lambda: tj.linear_fwd(X, wq, w8, ni, oi, xq=xq, x8=x8, out=Y, stream=stream), stream)
    ms_gemm = time_kernel(lambda: tj.gemm_nvfp4(xq, wq, x8, w8, out=Y, stream=stream), stream)
    out = {"shape": [M, N, K], "k_fp8": k, "linear_fwd": _gemm_frac(f4, f8, ms, fp4_peak, fp8_peak),
           "gemm": _gemm_frac(f4, f8, ms_gemm, fp4_peak, fp8_peak)}
    out["slice_formats"] = slice_formats(tj, dev, stream, X, W, ni, oi, k, fp4_peak, fp8_peak)
    del X, W, xq, x8, Y, wq, w8
    return out


def slice_formats(tj, dev, stream, X, W, ni, oi, k, fp4_peak, fp8_peak):
    """The same layer with the FP8 slice (E4M3 x E4M3) and with the FP6 x FP4 slice (X in
    E2M3, W in E2M1; the backward gives dY the partner format, so dX's slice is E2M3 x E2M1
    and dW's E2M1 x E2M3): forward through tj_linear_fwd, the forward GEMM alone, and the
    two backward calls with dY 16384 x 4096 heavy-tailed rows.  The f8f6f4 MMA runs FP6 and
    FP4 slice operands at the FP8 rate, so the peak weighting is the FP8 slice's."""
    from nvfp4_bit_fully_gb300 import workloads as wl

    M, K = X.shape
    N = W.shape[0]
    f4, f8 = 2.0 * M * N * (K - k), 2.0 * M * N * k
    dY = wl.device_student_t_rows(M, N, 1e-3, 3, 3, 33, dev)
    torch.cuda.synchronize()
    res = {}
    for name, fx, fw in (("fp8_x_fp8", tj.TJ_MX_E4M3, tj.TJ_MX_E4M3), ("e2m3_x_e2m1", tj.TJ_MX_E2M3, tj.TJ_MX_E2M1)):
        wq, w8 = tj.quantize_nvfp4(W, sel=ni, stream=stream), tj.quantize_mxfp8(W, sel=oi, stream=stream, fmt=fw)
        xq, x8 = tj.NVFP4.empty(M, K - k, dev), tj.MXFP8.empty(M, k, dev, fx)
        Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        dX = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
        dW = torch.empty(N, K, dtype=torch.float32, device=dev)
        ws_dx = torch.empty(tj.workspace_size(tj.TJ_OP_BWD_DX, M, N, K, k), dtype=torch.uint8, device=dev)
        ws_dw = torch.empty(tj.workspace_size(tj.TJ_OP_BWD_DW, M, N, K, k), dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()
        seeds = iter(range(10**6))
        ms_f = time_kernel(lambda: tj.linear_fwd(X, wq, w8, ni, oi, xq=xq, x8=x8, out=Y, stream=stream), stream)
        ms_g = time_kernel(lambda: tj.gemm_nvfp4(xq, wq, x8, w8, out=Y, stream=stream), stream)
        ms_dx = time_kernel(lambda: tj.linear_bwd_dx(dY, wq, w8, ni, oi, seed=next(seeds), workspace=ws_dx, out=dX,
                                                     stream=stream), stream)
        ms_dw = time_kernel(lambda: tj.linear_bwd_dw(dY, xq, x8, ni, oi, seed=next(seeds), workspace=ws_dw, out=dW,
                                                     stream=stream), stream)
        f4b = 2.0 * M * (K - k) * N
        res[name] = {"linear_fwd": _gemm_frac(f4, f8, ms_f, fp4_peak, fp8_peak),
                     "gemm_fwd": _gemm_frac(f4, f8, ms_g, fp4_peak, fp8_peak),
                     "linear_bwd_dx": _gemm_frac(f4b, f8, ms_dx, fp4_peak, fp8_peak),
                     "linear_bwd_dw": _gemm_frac(f4b, f8, ms_dw, fp4_peak, fp8_peak),
                     "slice_code_bytes_x": x8.codes.numel(), "slice_code_bytes_w": w8.codes.numel()}
        del wq, w8, xq, x8, Y, dX, dW, ws_dx, ws_dw
    del dY
    return res


def cfg4_bwd(tj, dev, stream, fp4_peak, fp8_peak):
    """Backward NVFP4 linear with RHT and SR at its own shape: dY 16384 x 4096 with
    heavy-tailed rows (1e-3 |t_3| N(0, 1)), W 4096 x 1024 N(0, 0.02), X 16384 x 1024 N(0, 1)
    with 1% of the columns x30; W-hat and X-hat from the RTN forward quantization, no
    outlier channels.  Timed through tj_linear_bwd_dx and tj_linear_bwd_dw (each: dY
    quantizer, operand re-alignment, FP4 GEMM)."""
    from nvfp4_bit_fully_gb300 import workloads as wl

    M, N, K, seed = TOKENS, 4096, 1024, 2
    dY = wl.device_student_t_rows(M, N, 1e-3, 3, seed, 31, dev)
    g = wl._cuda_gen(seed, 32, dev)
    W = (torch.randn(N, K, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    X = wl.device_heavy_columns((M, K), 1.0, 30.0, math.ceil(K / 100), seed, 11, dev)
    torch.cuda.synchronize()
    wq, xq = tj.quantize_nvfp4(W, stream=stream), tj.quantize_nvfp4(X, stream=stream)
    dX = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
    dW = torch.empty(N, K, dtype=torch.float32, device=dev)
    ws_dx = torch.empty(tj.workspace_size(tj.TJ_OP_BWD_DX, M, N, K, 0), dtype=torch.uint8, device=dev)
    ws_dw = torch.empty(tj.workspace_size(tj.TJ_OP_BWD_DW, M, N, K, 0), dtype=torch.uint8, device=dev)
    f4 = 2.0 * M * N * K
    torch.cuda.synchronize()                 # inputs were drawn on torch's current stream
    seeds = iter(range(10**6))
    ms_dx = time_kernel(lambda: tj.linear_bwd_dx(dY, wq, seed=next(seeds), workspace=ws_dx, out=dX, stream=stream),
                        stream)
    ms_dw = time_kernel(lambda: tj.linear_bwd_dw(dY, xq, seed=next(seeds), workspace=ws_dw, out=dW, stream=stream),
                        stream)
    out = {"shape": {"dY": [M, N], "W": [N, K], "X": [M, K]}, "linear_bwd_dx": _gemm_frac(f4, 0.0, ms_dx, fp4_peak, fp8_peak),
           "linear_bwd_dw": _gemm_frac(f4, 0.0, ms_dw, fp4_peak, fp8_peak)}
    del dY, W, X, wq, xq, dX, dW, ws_dx, ws_dw
    return out


def fp8_layer_set(tj, linears, stream, fp8_peak, nvfp4_linear_ms):
    """The FP8 linear baseline (tj_fp8_linear_*: MXFP8 operands, no RHT / SR / outlier
    split) over the same layer set, inputs and outputs: forward, dX and dW of the four
    linears per step.  The weights' MXFP8 forms (W along K, W^T along N) are made once,
    outside the timed region, as the NVFP4 forward weights are.  nvfp4_speedup = FP8
    step time / NVFP4 linear step time (the pages' metric: >1 means NVFP4 is faster)."""
    dev = linears[0].X.device
    bufs = []
    for lin in linears:
        M, N, K = TOKENS, lin.N, lin.K
        bufs.append({
            "w8": tj.quantize_mxfp8(lin.W, stream=stream), "wt8": tj.quantize_mxfp8(lin.W, along_cols=True, stream=stream),
            "x8": tj.MXFP8.empty(M, K, dev), "xt8": tj.MXFP8.empty(K, M, dev),
            "ws_dx": torch.empty(tj.workspace_size(tj.TJ_OP_FP8_BWD_DX, M, N, K, 0), dtype=torch.uint8, device=dev),
            "ws_dw": torch.empty(tj.workspace_size(tj.TJ_OP_FP8_BWD_DW, M, N, K, 0), dtype=torch.uint8, device=dev)})
    torch.cuda.synchronize()

    def step():
        for lin, b in zip(linears, bufs):
            tj.fp8_linear_fwd(lin.X, b["w8"], x8=b["x8"], xt8=b["xt8"], out=lin.Y, stream=stream)
            tj.fp8_linear_bwd_dx(lin.dY, b["wt8"], workspace=b["ws_dx"], out=lin.dX, stream=stream)
            tj.fp8_linear_bwd_dw(lin.dY, b["xt8"], workspace=b["ws_dw"], out=lin.dW, stream=stream)

    ms = time_kernel(step, stream, 20, warmup=3)
    flops = sum(l.flops for l in linears)
    tflops = flops / (ms * 1e-3) / 1e12
    del bufs
    return {"ms_per_step": round(ms, 4), "TFLOP/s": round(tflops, 1), "frac_of_fp8_peak": round(tflops / fp8_peak, 4),
            "nvfp4_speedup": round(ms / nvfp4_linear_ms, 3),
            "recipe": "MXFP8 (E4M3, UE8M0 per 1x32 along each GEMM's contraction axis, RTN) for X, W, dY; "
                      "fp32 accumulation; launches per linear: fwd 3 (X rows, X^T columns, GEMM), dX 2, dW 2"}


# ---------------------------------------------------------------------------
# the oracle as a CPU baseline (bounded sample of the same workload)
# ---------------------------------------------------------------------------
def oracle_sample(tokens, names=None):
    """Oracle fwd+bwd of the linear set (or the named linears) on `tokens` tokens;
    returns (seconds, flops)."""
    from nvfp4_bit_fully_gb300 import workloads as wl
    from oracle import calib as OC
    from oracle import linear as OL

    secs = 0.0
    flops = 0.0
    for name, N, K in wl.LAYER_SET:
        if names is not None and name not in names:
            continue
        X, W, dY = wl.layer_set_linear(name, N, K, seed=3, M=tokens)
        Xf, Wf, dYf = X.float().numpy(), W.float().numpy(), dY.float().numpy()
        t0 = time.perf_counter()
        k = OC.outlier_count(K, OUTLIER_PCT)
        outl, _ = OC.top_k_channels(OC.accumulate_sumsq(Xf, np.zeros(K)), k)
        _, fx, fw = OL.forward(Xf, Wf, outl)
        OL.bwd_dx(dYf, fw, outl, 7)
        OL.bwd_dw(dYf, fx, outl, 7)
        secs += time.perf_counter() - t0
        flops += 6.0 * tokens * N * K
    return secs, flops


def oracle_sample_one_thread(tokens):
    """oracle_sample in a fresh interpreter whose BLAS runs on one thread; (seconds, flops) or None."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    code = "import bench; s, f = bench.oracle_sample(%d); print(s, f)" % tokens
    try:
        r = subprocess.run([sys.executable, "-c", code], cwd=os.path.dirname(os.path.abspath(__file__)), env=env,
                           capture_output=True, text=True, timeout=600)
        s, f = r.stdout.split()[-2:]
        return float(s), float(f)
    except Exception:
        return None


def cpu_baseline():
    secs, flops = oracle_sample(128)
    out = {"value": round(flops / secs / 1e12, 6), "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
           "sample": "oracle fwd+dX+dW (calibration, quantize, RHT+SR, re-alignment, fp64 GEMMs) of all four "
                     "linears of the set on 128 of the 16384 tokens; %.1f s of CPU time (numpy elementwise "
                     "single-threaded, fp64 matmul via multithreaded BLAS)" % secs}
    one = oracle_sample_one_thread(128)
    if one is not None:
        out["one_thread"] = {"value": round(one[1] / one[0] / 1e12, 6), "cores": 1,
                             "sample": "the same sample with BLAS on one thread; %.1f s" % one[0]}
    return out


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(world, v):
    """Largest value over the ranks (the timed region ends when the slowest replica ends)."""
    if world == 1:
        return v
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world, flops_per_replica_step, steps, max_ms):
    """Throughput of the whole job: the work of every replica over the slowest replica's time."""
    return world * flops_per_replica_step * steps / (max_ms * 1e-3) / 1e12


def run_reference(args, world, rank):
    """--impl reference: the oracle (CPU) timed on bounded samples of the same workload."""
    if rank != 0:
        return 0
    for _ in range(args.warmup):
        oracle_sample(128, ("out",))
    secs, flops = 0.0, 0.0
    for _ in range(args.steps):
        s, f = oracle_sample(128, ("out",))
        secs += s
        flops += f
    value = flops / secs / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * secs / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (fp32 quantizer)",
            "data": "synthetic", "config": {"workload": WORKLOAD, "sample_per_step": "out-proj 1024->1024, 128 tokens"},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": "each step: oracle fwd+dX+dW of the out-proj linear (1024->1024, 10% FP8 "
                                       "outliers) on 128 of the 16384 tokens"},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def profiling_case(which):
    """Small cases for profiler captures (a few hundred MB on the device), each kernel
    launched twice: the second launch is the one to capture.
    gemm : the gate/up forward GEMM, 16384 x 8192, K = 921 FP4 + 103 FP8 slice, bf16 out.
    quant: at the dY shape 16384 x 4096: the row and column passes (NVFP4 SR + RHT and
           MXFP8); at 16384 x 1024: the OutControl split of X (103 outlier channels), the
           re-alignment of X-hat^T (921 channels, SR + RHT) and of its FP8 slice, as two
           launches and as one pair launch."""
    import __graft_entry__

    __graft_entry__.build()
    from nvfp4_bit_fully_gb300 import tj

    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    M, K, k = TOKENS, 1024, 103
    X = torch.randn(M, K, generator=g, device=dev).to(torch.bfloat16)
    oi = torch.arange(0, K, 10, device=dev, dtype=torch.int32)[:k]
    keep = torch.ones(K, dtype=torch.bool, device=dev)
    keep[oi.long()] = False
    ni = torch.nonzero(keep).squeeze(1).to(torch.int32)
    xq, x8 = tj.quantize_split(X, ni, oi)
    if which == "gemm":
        N = 8192
        W = (torch.randn(N, K, generator=g, device=dev) * 0.02).to(torch.bfloat16)
        wq, w8 = tj.quantize_nvfp4(W, sel=ni), tj.quantize_mxfp8(W, sel=oi)
        Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        calls = [lambda: tj.gemm_nvfp4(xq, wq, x8, w8, out=Y)]
    else:
        N = 4096
        dY = (torch.randn(M, N, generator=g, device=dev) * 1e-3).to(torch.bfloat16)
        s_dy, q8 = tj.NVFP4.empty(M, N, dev), tj.MXFP8.empty(M, N, dev)
        s_dyt, q8t = tj.NVFP4.empty(N, M, dev), tj.MXFP8.empty(N, M, dev)
        s_x, q8x = tj.NVFP4.empty(K - k, M, dev), tj.MXFP8.empty(k, M, dev)
        calls = [
            lambda: tj.quantize_nvfp4_mxfp8(dY, mode=tj.TJ_SR, rht=True, seed=3, tag=tj.TAG_DY_ROW,
                                            rht_tag=tj.TAG_RHT_DX, out=s_dy, out8=q8),
            lambda: tj.quantize_nvfp4_mxfp8(dY, along_cols=True, mode=tj.TJ_SR, rht=True, seed=3, tag=tj.TAG_DY_COL,
                                            rht_tag=tj.TAG_RHT_DW, out=s_dyt, out8=q8t),
            lambda: tj.quantize_split(X, ni, oi, out=xq, out8=x8),
            lambda: tj.requantize_nvfp4(xq, tj.TJ_SR, True, 3, tj.TAG_XT, tj.TAG_RHT_DW, out=s_x),
            lambda: tj.requantize_mxfp8(x8, out=q8x),
            lambda: tj.requantize_nvfp4_mxfp8(xq, x8, tj.TJ_SR, True, 3, tj.TAG_XT, tj.TAG_RHT_DW, out=s_x, out8=q8x),
        ]
    torch.cuda.synchronize()
    for f in calls:
        for _ in range(2):
            f()
    torch.cuda.synchronize()
    tj.device_status()
    print(json.dumps({"profiling_case": which, "launches": 2 * len(calls)}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the quantize sweep / GEMM-alone / e2e parts")
    ap.add_argument("--osci-params", type=int, default=0, help="override the OsciReset size (profiling only)")
    ap.add_argument("--only", choices=["all", "osci", "linear", "gemm", "quant"], default="all",
                    help="run one part of the step, or one profiling case (gemm, quant), for small profiler "
                         "captures; not a bench line")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.only in ("gemm", "quant"):
        return profiling_case(args.only)

    import __graft_entry__

    __graft_entry__.build()
    from nvfp4_bit_fully_gb300 import tj
    from nvfp4_bit_fully_gb300 import workloads as wl

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    stream = torch.cuda.Stream(device=dev)
    peaks, peak_src = load_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    bf16_burst = float(peaks["bf16_tflops"])
    fp4_peak, fp8_peak = bf16_burst * 13.5 / 2.25, bf16_burst * 4.5 / 2.25      # nominal dtype ratios

    with torch.cuda.stream(stream):
        linears = [Linear(tj, wl, n, N, K, dev, seed=3 + rank) for n, N, K in wl.LAYER_SET] \
            if args.only != "osci" else []
        osci_n = args.osci_params or wl.OSCI_PARAMS
        osci = OsciState(tj, wl, osci_n, dev, seed=3 + rank) if args.only != "linear" else None
    torch.cuda.synchronize()

    step_counter = [0]

    def step(tl):
        t = step_counter[0]
        seed = 1000 + t
        for lin in linears:
            lin.run(tj, seed, tl, stream)
        if osci is not None:
            osci.run(tj, float(wl.cosine_lr(t % 200)), tl, stream)
        step_counter[0] += 1

    for _ in range(args.warmup):
        step(Timeline(stream))
    torch.cuda.synchronize()
    tj.device_status()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.25)
    tl = Timeline(stream)
    barrier(world)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(args.steps):
        step(tl)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    tj.device_status()

    total_ms = max_over_ranks(world, t_start.elapsed_time(t_end))
    summ = tl.summary()
    if args.only != "all":
        if rank == 0:
            print(json.dumps({"profiling_case": args.only, "ms_per_step": total_ms / args.steps,
                              "parts": {k: v[0] / v[1] for k, v in summ.items()}}), flush=True)
        return 0
    lin_ms = max_over_ranks(world, sum(v[0] for k, v in summ.items() if k != "osci_reset"))
    osci_ms = summ["osci_reset"][0] / summ["osci_reset"][1]
    flops_step = sum(l.flops for l in linears)
    value = whole_job_tflops(world, flops_step, args.steps, lin_ms)
    osci_gbs = osci.bytes / (osci_ms * 1e-3) / 1e9
    # per call: average ms and throughput against its algorithmic work
    parts = {}
    kern = {}                       # kernel -> [total ms, flops4, flops8, bytes, launches]
    kern_instr = {}                 # kernel -> lane instructions over the timed steps (quantize kernels)
    for name, (ms_tot, n) in sorted(summ.items()):
        call = name.split(".")[-1]
        p = {"ms": round(ms_tot / n, 4)}
        agg = kern.setdefault(CALL_KERNEL[call], [0.0, 0.0, 0.0, 0.0, 0])
        if call != "osci_reset":
            lin_i = next(l for l in linears if l.name == name.split(".")[0]).lane_instr.get(call)
            if lin_i is not None:
                kern_instr[CALL_KERNEL[call]] = kern_instr.get(CALL_KERNEL[call], 0.0) + lin_i * n
        agg[0] += ms_tot
        agg[4] += n
        if call == "osci_reset":
            p["GB/s"] = round(osci_gbs, 1)
            agg[3] += osci.bytes * n
        else:
            lin = next(l for l in linears if l.name == name.split(".")[0])
            w = lin.work[call]
            if isinstance(w, tuple):
                p["TFLOP/s"] = round((w[0] + w[1]) / (ms_tot / n * 1e-3) / 1e12, 1)
                agg[1] += w[0] * n
                agg[2] += w[1] * n
                agg[3] += lin.gemm_bytes[call] * n          # operands and output, for the traffic ratio
            else:
                p["GB/s"] = round(w / (ms_tot / n * 1e-3) / 1e9, 1)
                agg[3] += w * n
        parts[name] = p
    kernels = {}
    for kname, (ms_tot, f4, f8, by, n) in kern.items():
        e = {"launches_per_step": n // args.steps, "ms_per_step": round(ms_tot / args.steps, 4),
             "share": round(ms_tot / (total_ms * world / world), 3)}
        if f4 + f8 > 0:
            t_star = f4 / (fp4_peak * 1e12) + f8 / (fp8_peak * 1e12)       # time at the dtype-weighted peak
            e.update({"TFLOP/s": round((f4 + f8) / (ms_tot * 1e-3) / 1e12, 1),
                      "frac": round(t_star / (ms_tot * 1e-3), 4)})
        else:
            e.update({"GB/s": round(by / (ms_tot * 1e-3) / 1e9, 1), "frac": round(by / (ms_tot * 1e-3) / 1e9 / hbm_peak, 3)})
            if kname in kern_instr and clk.get("sm_mhz"):
                lanes_per_s = num_sms * 128 * float(clk["sm_mhz"]) * 1e6
                e["issue_roofline"] = {"lane_instr_per_step": round(kern_instr[kname] / args.steps),
                                       "frac": round(kern_instr[kname] / (lanes_per_s * ms_tot * 1e-3), 3)}
        kernels[kname] = e
    # dominant kernel of the step (largest total time), with its roofline
    dom = max(kern.items(), key=lambda kv: kv[1][0])[0]
    ms_tot, f4, f8, by, n = kern[dom]
    if f4 + f8 > 0:
        peak_mix = (f4 + f8) / (f4 / fp4_peak + f8 / fp8_peak)           # dtype-weighted peak, TFLOP/s
        achieved = (f4 + f8) / (ms_tot * 1e-3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 1), "peak": round(peak_mix, 1),
                "unit": "TFLOP/s", "frac": round(achieved / peak_mix, 4),
                "traffic": (round(TRAFFIC_BYTES_PER_LAUNCH[dom]) if dom in TRAFFIC_BYTES_PER_LAUNCH else None),
                "algorithmic_bytes_per_launch": round(by / n) if by else None,
                "algorithmic_flops_per_launch": round((f4 + f8) / n),
                "peak_source": "%s bf16 burst %.1f x nominal fp4 (x6) / fp8 (x2) ratios, weighted by the FP4 / FP8 "
                               "flop mix" % (peak_src, bf16_burst)}
    else:
        achieved = by / (ms_tot * 1e-3) / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 3),
                "traffic": (round(TRAFFIC_BYTES_PER_ELEM[dom] * osci.n) if dom in TRAFFIC_BYTES_PER_ELEM else None),
                "algorithmic_bytes_per_launch": round(by / n), "peak_source": peak_src + " hbm_gbs"}
    # every recorded call of the timed region launches exactly one kernel of the library
    # (per linear: split + GEMM, dY rows + re-alignment pair + GEMM pair, dY columns +
    # re-alignment pair + GEMM pair; then one OsciReset)
    launches = len(tl.records)

    extras = {}
    if not args.no_extras and rank == 0:
        flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)   # 512 MB > L2
        extras["quantize_sweep"] = quantize_sweep(tj, dev, stream, hbm_peak, flush)
        big = max(linears, key=lambda l: l.N * l.K)
        extras["gemm_fwd_alone"] = gemm_alone(tj, big, stream, fp4_peak, fp8_peak)
        del flush
        extras["fp8_layer_set"] = fp8_layer_set(tj, linears, stream, fp8_peak, lin_ms / args.steps)
        extras["cfg3_fwd"] = cfg3_fwd(tj, dev, stream, fp4_peak, fp8_peak)
        extras["cfg4_bwd"] = cfg4_bwd(tj, dev, stream, fp4_peak, fp8_peak)
        if osci is not None:
            extras["adamw_osci_reset"] = adamw_osci_alone(tj, osci, stream, hbm_peak)
    e2e = None
    if not args.no_extras:
        e2e = measure_e2e(tj, linears, stream, max(3, args.steps // 4), world)

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 1), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4 (e2m1 x e4m3 x fp32 scales) + fp8 slice, fp32 acc",
                "data": "synthetic (seeded CUDA generator; shapes and distributions of the pages' OLMo-2 370M linears)",
                "config": {"workload": WORKLOAD, "tokens": TOKENS, "outlier_pct": OUTLIER_PCT,
                           "osci_reset_params": osci.n, "parallelism": "replicas" if world > 1 else "single GPU",
                           "l2": "no flush: per-step working set ~13 GB (OsciReset state 10.8 GB) >> 129 MB L2"},
                "linear_ms_per_step": round(lin_ms / args.steps, 4),
                "osci_reset": {"ms": round(osci_ms, 4), "GB/s": round(osci_gbs, 1), "frac": round(osci_gbs / hbm_peak, 3)},
                "roofline": roof, "kernels": kernels, "parts": parts, "gpu_launches": launches, "clocks": clk}
        line.update(extras)
        if e2e is not None:
            line["e2e"] = e2e
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline()
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def measure_e2e(tj, linears, stream, steps, world):
    """Same metric through the public API with host buffers: X and dY of every linear copied
    host->device from pinned memory and every dW copied back, inside the timed region.  The
    copies run on two more streams (host->device, device->host), pipelined with the compute.
    - Each linear's inputs are copied as soon as the previous step's use of the same device
      buffers has finished, so they overlap the compute of the linears before it.
    - Each dW leaves as soon as its linear's backward has written it.
    - Events order every copy against the compute that reads or writes the same buffer."""
    hx = [l.X.cpu().pin_memory() for l in linears]
    hdy = [l.dY.cpu().pin_memory() for l in linears]
    hdw = [torch.empty(l.dW.shape, dtype=l.dW.dtype).pin_memory() for l in linears]
    h2d = sum(t.numel() * t.element_size() for t in hx + hdy)
    d2h = sum(t.numel() * t.element_size() for t in hdw)
    cs = torch.cuda.Stream(device=stream.device)        # host -> device
    ds = torch.cuda.Stream(device=stream.device)        # device -> host
    n = len(linears)
    ev_in = [torch.cuda.Event() for _ in range(n)]      # inputs of linear i on the device
    ev_done = [torch.cuda.Event() for _ in range(n)]    # linear i's calls finished (inputs free, dW written)
    ev_out = [torch.cuda.Event() for _ in range(n)]     # dW of linear i copied back (dW free)
    started = [False] * n

    def one(seed):
        for i, l in enumerate(linears):
            if started[i]:
                cs.wait_event(ev_done[i])
            with torch.cuda.stream(cs):
                l.X.copy_(hx[i], non_blocking=True)
                l.dY.copy_(hdy[i], non_blocking=True)
            ev_in[i].record(cs)
        for i, l in enumerate(linears):
            stream.wait_event(ev_in[i])
            if started[i]:
                stream.wait_event(ev_out[i])
            with torch.cuda.stream(stream):
                l.run_api(tj, seed, stream)
            ev_done[i].record(stream)
            ds.wait_event(ev_done[i])
            with torch.cuda.stream(ds):
                hdw[i].copy_(l.dW, non_blocking=True)
            ev_out[i].record(ds)
            started[i] = True

    for w in range(2):
        one(5000 + w)
    torch.cuda.synchronize()
    barrier(world)
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(stream)
    cs.wait_event(s)
    ds.wait_event(s)
    for t in range(steps):
        one(6000 + t)
    for c in (cs, ds):
        end_c = torch.cuda.Event()
        end_c.record(c)
        stream.wait_event(end_c)
    e.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(world, s.elapsed_time(e))
    return {"value": round(whole_job_tflops(world, sum(l.flops for l in linears), steps, ms), 1), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": round(ms / steps, 4),
            "copies": "host->device and device->host streams, pipelined with the compute"}


if __name__ == "__main__":
    sys.exit(main())
