"""Synthetic ablations of the TetraJet-v2 components, run through the library.

The pages report ablations measured in pretraining (technical summary §4): removing
OsciReset, OutControl in the forward and the backward pass, and robustness to the
oscillation threshold and to the step at which tracking starts.  Without a corpus or
trained weights, this harness restates them on synthetic tensors whose behaviour the
components target, and measures what each component changes:

OsciReset (§2.B), on a synthetic optimiser trajectory: every master weight descends
towards its own target with a sign step of the (cosine-decayed) learning rate plus
noise, so once the learning rate is small it keeps crossing back and forth over its
target; targets are placed near quantization-bin boundaries, where that crossing
flips the quantized weight.  Per configuration (OsciReset off; reset threshold r;
tracking start step) it reports the resets, the flips of the quantized weights between
bins (code changes) over the last steps, the oscillation the method suppresses, and
the final distance of the quantized weights from the quantized targets.

OutControl (§2.C), on activations with a few heavy channels: for each outlier
fraction p it calibrates the channel set, runs the layer's forward and backward
through tj_linear_fwd / tj_linear_bwd_dx / tj_linear_bwd_dw over several seeds,
and reports the forward error against the unquantized product, and the bias (error
of the mean over seeds) and per-seed error of dX and dW.

Slice formats (§5 names FP6 x FP4 mixed precision as a future direction): at a 10%
outlier fraction, the same layer with the FP8 slice and with FP6 x FP4 slices (X in
E2M3 or E3M2 with W in E2M1, and the reverse), reporting the slice product's own error,
the layer's forward error and the error of the mean dX / dW on the outlier channels.

Usage:  python -m nvfp4_bit_fully_gb300.ablation [--out ablation.json] [--small]
Needs a CUDA GPU and the built library (there is no CPU fallback).
"""
import argparse
import json
import math

import numpy as np

OSCI_THRESHOLDS = (2.0, 4.0, 8.0, 16.0)
OSCI_START_STEPS = (0, 100, 150, 180)
OUTLIER_PCTS = (0, 1, 5, 10, 20)
# slice element formats (x, w): the FP8 slice and the FP6 x FP4 variants (tj.h tj_mx_format)
SLICE_FORMATS = (("e4m3 x e4m3", 0, 0), ("e2m3 x e2m1", 3, 5), ("e3m2 x e2m1", 4, 5), ("e2m1 x e2m3", 5, 3))
LR_THR = 1e-4


# ---------------------------------------------------------------------------
# host metrics (plain numpy; pinned by CPU tests)
# ---------------------------------------------------------------------------
def rel_err(got, ref):
    """Frobenius-norm error of `got` relative to `ref`."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got - ref))


def bias_and_spread(samples, ref):
    """For estimates `samples` [S, ...] of `ref`: the relative error of their mean (the
    bias, up to the sampling noise of the mean) and the mean relative error of one
    sample.  An unbiased estimator's first value falls like 1/sqrt(S) of the second."""
    samples = np.asarray(samples, dtype=np.float64)
    return {"bias": rel_err(samples.mean(axis=0), ref),
            "per_seed": float(np.mean([rel_err(s, ref) for s in samples])), "seeds": int(samples.shape[0])}


def flips(history):
    """Number of changes between consecutive snapshots of quantized values [T, ...]."""
    h = np.asarray(history)
    return int((h[1:] != h[:-1]).sum()) if h.shape[0] > 1 else 0


def unpack_codes(raw, rows, cols):
    """E2M1 codes [rows, cols] of an NVFP4 code buffer [rows_p][cols_p / 2] (two codes per
    byte, the even element in the low nibble), with the sign of a zero magnitude cleared:
    the quantized bin of each element."""
    cols_p = (cols + 127) // 128 * 128
    b = np.asarray(raw, dtype=np.uint8).reshape(-1, cols_p // 2)[:rows]
    c = np.empty((rows, cols_p), dtype=np.uint8)
    c[:, 0::2] = b & 15
    c[:, 1::2] = b >> 4
    c = c[:, :cols]
    return np.where((c & 7) == 0, 0, c)


def cosine_lr(step, total, lr_max=1e-3, lr_min=1e-5):
    return lr_min + 0.5 * (lr_max - lr_min) * (1.0 + math.cos(math.pi * step / total))


def osci_configs():
    """The OsciReset sweep: off, every threshold from step 0, the default threshold 4 from
    every start step."""
    cfgs = [{"name": "off", "track": False, "risk_thr": 4.0, "start": 0}]
    cfgs += [{"name": "r=%g" % r, "track": True, "risk_thr": r, "start": 0} for r in OSCI_THRESHOLDS]
    cfgs += [{"name": "start=%d" % s, "track": True, "risk_thr": 4.0, "start": s} for s in OSCI_START_STEPS if s]
    return cfgs


def synthetic_targets(rng, rows, cols, bin_edge_frac=0.5):
    """Target weights N(0, 0.02), a fraction of which is moved onto the boundary between two
    E2M1 bins of one unit (amax / 6) of its 128-block (the oscillation-prone weights)."""
    t = rng.standard_normal((rows, cols)).astype(np.float32) * np.float32(0.02)
    blk = np.abs(t.reshape(rows, -1, 128)).max(axis=2, keepdims=True)       # outer-block maxima
    s = blk / np.float32(6.0)                                               # ~ one E2M1 unit at the block top
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float32)
    # every element but its block's maximum (which keeps the block's scale) may move
    pick = (rng.random((rows, cols)) < bin_edge_frac) & (np.abs(t) != np.repeat(blk, 128, axis=2).reshape(rows, cols))
    m = mids[rng.integers(0, len(mids), (rows, cols))].reshape(rows, -1, 128)
    edge = (np.sign(t).reshape(rows, -1, 128) * m * s).reshape(rows, cols).astype(np.float32)
    return np.where(pick, edge, t).astype(np.float32)


# ---------------------------------------------------------------------------
# GPU runs through the library
# ---------------------------------------------------------------------------
def run_osci(tj, torch, rows, cols, steps, seed, cfg, window=20):
    """One OsciReset configuration on the synthetic trajectory; returns its metrics."""
    dev = torch.device("cuda")
    rng = np.random.default_rng(seed)
    target = torch.from_numpy(synthetic_targets(rng, rows, cols)).to(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    w = (target + torch.randn(rows, cols, generator=g, device=dev) * 0.01).contiguous()
    w_prev = w.clone()
    dq = torch.zeros_like(w)
    dm = torch.zeros_like(w)
    q = [tj.quantize_nvfp4(w), tj.NVFP4.empty(rows, cols, dev)]
    mask = torch.empty(rows * ((cols + 31) // 32), dtype=torch.int32, device=dev)
    resets, hist = 0, []
    for t in range(steps):
        lr = cosine_lr(t, steps)
        step = torch.sign(w - target) + 0.5 * torch.randn(rows, cols, generator=g, device=dev)
        w.sub_(lr * step)
        track = cfg["track"] and t >= cfg["start"]
        if t == cfg["start"] and cfg["track"]:            # tracking starts: distances from here
            w_prev.copy_(w)
            dq.zero_()
            dm.zero_()
        tj.osci_reset(w, w_prev, dq, dm, q[0], q[1], mask, lr, LR_THR, cfg["risk_thr"], track)
        if track:
            bits = mask.view(torch.int32).cpu().numpy().view(np.uint32)
            resets += int(np.unpackbits(bits.view(np.uint8)).sum())
        q.reverse()
        if t >= steps - window:                          # the bins (codes) of the step's Q
            hist.append(unpack_codes(q[0].codes.cpu().numpy(), rows, cols))
    qt = tj.dequantize_nvfp4(tj.quantize_nvfp4(target)).cpu().numpy()
    final = tj.dequantize_nvfp4(q[0]).cpu().numpy()
    torch.cuda.synchronize()
    return {"config": cfg["name"], "resets": resets, "resets_per_weight": resets / (rows * cols),
            "flips_last_%d_steps" % window: flips(hist), "flip_rate": flips(hist) / (rows * cols * (len(hist) - 1)),
            "final_q_vs_q_target": rel_err(final, qt)}


def run_outctl(tj, torch, M, N, K, pct, seeds, base_seed):
    """One outlier fraction: calibration, forward error, gradient bias and spread."""
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(base_seed)
    heavy = torch.randperm(K, generator=g, device=dev)[:max(1, K // 50)]

    def batch():
        x = torch.randn(M, K, generator=g, device=dev)
        x[:, heavy] *= 40.0
        return x.to(torch.bfloat16)

    k = (pct * K + 99) // 100
    sumsq = torch.zeros(K, dtype=torch.float64, device=dev)
    for _ in range(2):
        tj.outlier_calibrate(batch(), sumsq)
    X = batch()
    W = (torch.randn(N, K, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    dY = (torch.randn(M, N, generator=g, device=dev) * 1e-3).to(torch.bfloat16)
    Xf, Wf, dYf = X.double(), W.double(), dY.double()
    y_ref = (Xf @ Wf.T).cpu().numpy()
    dx_ref = (dYf @ Wf).cpu().numpy()
    dw_ref = (dYf.T @ Xf).cpu().numpy()
    if k:
        oi, ni = tj.outlier_calibrate(None, sumsq, finalize=True, k=k)
        wq, w8 = tj.quantize_nvfp4(W, sel=ni), tj.quantize_mxfp8(W, sel=oi)
    else:
        oi = ni = w8 = None
        wq = tj.quantize_nvfp4(W)
    y, xq, x8 = tj.linear_fwd(X, wq, w8, ni, oi, out_dtype=torch.float32)
    dxs, dws = [], []
    for s in range(seeds):
        dxs.append(tj.linear_bwd_dx(dY, wq, w8, ni, oi, seed=base_seed * 1000 + s, out_dtype=torch.float32).cpu().numpy())
        dws.append(tj.linear_bwd_dw(dY, xq, x8, ni, oi, seed=base_seed * 1000 + s).cpu().numpy())
    torch.cuda.synchronize()
    # the quantized forward operands set the target of the backward estimates: dX estimates
    # dY W-hat, dW estimates dY^T X-hat (§2.A), so their bias is measured against those
    w_hat = _dequant_operand(tj, torch, wq, w8, ni, oi, N, K)
    x_hat = _dequant_operand(tj, torch, xq, x8, ni, oi, M, K)
    return {"outlier_pct": pct, "k": int(k), "fwd_rel_err": rel_err(y.cpu().numpy(), y_ref),
            "dx": bias_and_spread(dxs, dY.double().cpu().numpy() @ w_hat),
            "dw": bias_and_spread(dws, dY.double().cpu().numpy().T @ x_hat),
            "dx_vs_unquantized": rel_err(np.mean(dxs, axis=0), dx_ref),
            "dw_vs_unquantized": rel_err(np.mean(dws, axis=0), dw_ref)}


def run_slice_formats(tj, torch, M, N, K, pct, seeds, base_seed):
    """The layer of run_outctl at one outlier fraction with each slice format pair."""
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(base_seed)
    heavy = torch.randperm(K, generator=g, device=dev)[:max(1, K // 50)]

    def batch():
        x = torch.randn(M, K, generator=g, device=dev)
        x[:, heavy] *= 40.0
        return x.to(torch.bfloat16)

    k = (pct * K + 99) // 100
    sumsq = torch.zeros(K, dtype=torch.float64, device=dev)
    for _ in range(2):
        tj.outlier_calibrate(batch(), sumsq)
    oi, ni = tj.outlier_calibrate(None, sumsq, finalize=True, k=k)
    X = batch()
    W = (torch.randn(N, K, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    dY = (torch.randn(M, N, generator=g, device=dev) * 1e-3).to(torch.bfloat16)
    Xf, Wf, dYf = X.double(), W.double(), dY.double()
    o = oi.long()
    y_ref = (Xf @ Wf.T).cpu().numpy()
    slice_ref = (Xf[:, o] @ Wf[:, o].T).cpu().numpy()
    dx_ref = (dYf @ Wf[:, o]).cpu().numpy()
    dw_ref = (dYf.T @ Xf[:, o]).cpu().numpy()
    wq = tj.quantize_nvfp4(W, sel=ni)
    rows = []
    for name, fx, fw in SLICE_FORMATS:
        w8 = tj.quantize_mxfp8(W, sel=oi, fmt=fw)
        y, xq, x8 = tj.linear_fwd(X, wq, w8, ni, oi, out_dtype=torch.float32, fmt_x8=fx)
        ys = tj.gemm_mxfp8(x8, w8)
        dxs, dws = [], []
        for s in range(seeds):
            dxs.append(tj.linear_bwd_dx(dY, wq, w8, ni, oi, seed=base_seed * 1000 + s,
                                        out_dtype=torch.float32)[:, o].cpu().numpy())
            dws.append(tj.linear_bwd_dw(dY, xq, x8, ni, oi, seed=base_seed * 1000 + s)[:, o].cpu().numpy())
        torch.cuda.synchronize()
        rows.append({"slice": name, "k": int(k), "slice_fwd_rel_err": rel_err(ys.cpu().numpy(), slice_ref),
                     "fwd_rel_err": rel_err(y.cpu().numpy(), y_ref),
                     "dx_outlier_cols_vs_unquantized": rel_err(np.mean(dxs, axis=0), dx_ref),
                     "dw_outlier_cols_vs_unquantized": rel_err(np.mean(dws, axis=0), dw_ref),
                     "slice_code_bytes": int(x8.codes.numel() + w8.codes.numel())})
    return rows


def _dequant_operand(tj, torch, q, q8, ni, oi, rows, K):
    """fp64 values of a forward operand [rows, K] from its NVFP4 part (normal channels)
    and FP8 slice (outlier channels), in the original channel order."""
    full = np.zeros((rows, K))
    nv = tj.dequantize_nvfp4(q).double().cpu().numpy()
    if ni is None:
        full[:, :] = nv
        return full
    full[:, ni.cpu().numpy()] = nv
    full[:, oi.cpu().numpy()] = tj.dequantize_mxfp8(q8).double().cpu().numpy()
    return full


def run(out_path, small=False):
    import torch

    from nvfp4_bit_fully_gb300 import tj

    tj.load()
    if small:
        rows, cols, steps, M, N, K, seeds = 64, 256, 40, 256, 256, 512, 4
    else:
        rows, cols, steps, M, N, K, seeds = 1024, 1024, 200, 4096, 1024, 1024, 16
    table = {"osci_reset": [run_osci(tj, torch, rows, cols, steps, 7, c) for c in osci_configs()],
             "outcontrol": [run_outctl(tj, torch, M, N, K, p, seeds, 11) for p in OUTLIER_PCTS],
             "slice_formats": run_slice_formats(tj, torch, M, N, K, 10, seeds, 13),
             "setup": {"osci": {"weights": rows * cols, "steps": steps, "lr": "cosine 1e-3 -> 1e-5", "lr_thr": LR_THR},
                       "outcontrol": {"M": M, "N": N, "K": K, "seeds": seeds, "heavy_channels": max(1, K // 50)}}}
    with open(out_path, "w") as f:
        json.dump(table, f, indent=1)
    return table


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--out", default="ablation.json")
    ap.add_argument("--small", action="store_true", help="a minute-scale version of the sweep")
    args = ap.parse_args()
    table = run(args.out, args.small)
    print(json.dumps({k: v for k, v in table.items() if k != "setup"}, indent=1))


if __name__ == "__main__":
    main()
