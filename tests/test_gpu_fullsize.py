"""GPU parity at the full workload sizes, on sampled outputs.

The full tensors run through the library in the same calls and shapes as the
benchmark; the oracle then recomputes a sample of the outputs one by one:
- 16384 tokens through each linear of the ~370M-class decoder-layer set, with OutControl calibrated on four batches;
- the forward-with-OutControl case (16384 x 1024 -> 4096);
- the backward RHT + SR case (dY 16384 x 4096, W 4096 x 1024);
- the quantize-only sweep at 16384 x 4096;
- OsciReset, alone and fused with the AdamW step, over the benchmark's 369,098,752 master weights.

Every sampled operand row, of a quantized operand the step produced, has to match bit for bit:
- X-hat rows and their FP8 slice;
- S_dY rows, Q8(dY) rows;
- S_W / S_X rows, the re-aligned W-hat^T / X-hat^T;
- the transposed dY operands;
- the FP8 re-alignments.

Each sampled product entry must lie within 2e-3 * sum|a||b| of the oracle's fp64 product (plus
half a bf16 ulp for bf16 outputs).

Sampling keeps the oracle's work small.  A double-block RTN quantization depends only on its own
128-element segment, so a column of W-hat or X-hat needs only the 128-channel block holding it.
SR depends on the element index, which the oracle takes as row ids.  Samples include the first
and last rows, the first and last (ragged) channel blocks and the last outlier channel.
"""
import math

import numpy as np
import pytest
import torch

from layouts import (assert_gemm_close, carve_workspace, mxfp8_to_logical, nvfp4_padding_is_zero,
                     nvfp4_to_logical)
from nvfp4_bit_fully_gb300 import workloads as wl
from oracle import calib as OC
from oracle import linear as OL
from oracle import quant as Q

pytestmark = pytest.mark.gpu

TOKENS = 16384


@pytest.fixture(scope="module")
def tj():
    from nvfp4_bit_fully_gb300 import tj as _tj

    _tj.load()
    return _tj


def _f32(t):
    return t.float().cpu().numpy()


def _rows_equal(got, ref, rows, what):
    """got: logical arrays of the whole GPU operand; ref: oracle arrays of the sampled rows."""
    for name, g, r in zip(("codes", "scales", "outer scales"), got, ref):
        g = np.asarray(g)[rows]
        r = np.asarray(r)
        assert g.shape == r.shape, (what, name, g.shape, r.shape)
        if not np.array_equal(g, r):
            bad = np.argwhere(g != r)
            i = tuple(bad[0])
            raise AssertionError("%s %s differ at %d positions; first (sample row %d, col %d): gpu %r oracle %r"
                                 % (what, name, len(bad), i[0], i[1], g[i], r[i]))


def _nv_deq_cols(A, cols, cs):
    """Columns cs (indices into `cols`) of the fp32 RTN double-block X-hat / W-hat of A[:, cols],
    as rows [len(cs), rows of A]: only the 128-channel blocks holding them are quantized."""
    blocks = {}
    out = []
    for c in cs:
        b0 = (int(c) // Q.OUTER) * Q.OUTER
        if b0 not in blocks:
            blocks[b0] = Q.dequantize_nvfp4_f32(*Q.quantize_nvfp4(A[:, cols[b0: b0 + Q.OUTER]], Q.RTN))
        out.append(blocks[b0][:, int(c) - b0])
    return np.stack(out)


def _mx_deq_cols(A, cols, js):
    """Columns js of the fp32 MXFP8 slice of A[:, cols] (their 32-channel groups only), as rows."""
    groups = {}
    out = []
    for j in js:
        g0 = (int(j) // 32) * 32
        if g0 not in groups:
            groups[g0] = Q.dequantize_mxfp8_f32(*Q.quantize_mxfp8(A[:, cols[g0: g0 + 32]]))
        out.append(groups[g0][:, int(j) - g0])
    return np.stack(out)


def _abs_nv(qa, qb, alpha=1.0):
    return alpha * (np.abs(Q.dequantize_nvfp4_f64(*qa)) @ np.abs(Q.dequantize_nvfp4_f64(*qb)).T)


def _abs_mx(qa, qb):
    return np.abs(Q.dequantize_mxfp8_f64(*qa)) @ np.abs(Q.dequantize_mxfp8_f64(*qb)).T


def _samples(n, count, rng):
    s = set(rng.choice(n, size=min(count, n), replace=False).tolist()) | {0, n - 1}
    return np.array(sorted(s), dtype=np.int64)


def _channel_samples(k_n, rng):
    """Normal-channel samples from the first block, one middle block and the last (ragged) block."""
    nb = (k_n + Q.OUTER - 1) // Q.OUTER
    blocks = sorted({0, nb // 2, nb - 1})
    s = set()
    for b in blocks:
        lo, hi = b * Q.OUTER, min(k_n, (b + 1) * Q.OUTER)
        s |= set(rng.choice(np.arange(lo, hi), size=min(4, hi - lo), replace=False).tolist())
    s.add(k_n - 1)
    return np.array(sorted(s), dtype=np.int64)


def _run_steps(tj, X, W, dY, ni, oi, k, seed):
    """The benchmark's call sequence for one linear (the kernels tj_linear_fwd / bwd_dx /
    bwd_dw launch, one C-ABI call each), into fresh buffers."""
    M, K = X.shape
    N = W.shape[0]
    kn = K - k
    d = X.device
    r = {}
    r["wq"], r["w8"] = tj.quantize_nvfp4(W, sel=ni), tj.quantize_mxfp8(W, sel=oi)
    r["xq"], r["x8"] = tj.NVFP4.empty(M, kn, d), tj.MXFP8.empty(M, k, d)
    tj.quantize_split(X, ni, oi, out=r["xq"], out8=r["x8"])
    r["Y"] = torch.empty(M, N, dtype=torch.bfloat16, device=d)
    tj.gemm_nvfp4(r["xq"], r["wq"], r["x8"], r["w8"], out=r["Y"])
    SR = tj.TJ_SR
    r["s_dy"], r["q8_dy"] = tj.NVFP4.empty(M, N, d), tj.MXFP8.empty(M, N, d)
    tj.quantize_nvfp4_mxfp8(dY, mode=SR, rht=True, seed=seed, tag=tj.TAG_DY_ROW, rht_tag=tj.TAG_RHT_DX,
                            out=r["s_dy"], out8=r["q8_dy"])
    r["s_w"] = tj.requantize_nvfp4(r["wq"], SR, True, seed, tj.TAG_WT, tj.TAG_RHT_DX)
    r["q8_w"] = tj.requantize_mxfp8(r["w8"])
    r["dX"] = torch.empty(M, K, dtype=torch.bfloat16, device=d)
    tj.gemm_pair(r["s_dy"], r["s_w"], r["q8_dy"], r["q8_w"], alpha=2.0 ** -7, out=r["dX"], out8=r["dX"],
                 col_map=ni, col_map8=oi)
    r["s_dyt"], r["q8_dyt"] = tj.NVFP4.empty(N, M, d), tj.MXFP8.empty(N, M, d)
    tj.quantize_nvfp4_mxfp8(dY, along_cols=True, mode=SR, rht=True, seed=seed, tag=tj.TAG_DY_COL,
                            rht_tag=tj.TAG_RHT_DW, out=r["s_dyt"], out8=r["q8_dyt"])
    r["s_x"] = tj.requantize_nvfp4(r["xq"], SR, True, seed, tj.TAG_XT, tj.TAG_RHT_DW)
    r["q8_x"] = tj.requantize_mxfp8(r["x8"])
    r["dW"] = torch.empty(N, K, dtype=torch.float32, device=d)
    tj.gemm_pair_f32(r["s_dyt"], r["s_x"], r["q8_dyt"], r["q8_x"], r["dW"], ni, oi, alpha=2.0 ** -7)
    torch.cuda.synchronize()
    tj.device_status()
    return r


def _run_api(tj, X, W, dY, seed):
    """The user-facing calls without outlier channels (tj_linear_fwd / bwd_dx / bwd_dw)."""
    M, K = X.shape
    N = W.shape[0]
    r = {"wq": tj.quantize_nvfp4(W), "w8": None, "x8": None, "q8_dy": None, "q8_w": None, "q8_dyt": None,
         "q8_x": None}
    y, r["xq"], _ = tj.linear_fwd(X, r["wq"], None, None, None)
    r["Y"] = y
    ws_dx = torch.empty(tj.workspace_size(tj.TJ_OP_BWD_DX, M, N, K, 0), dtype=torch.uint8, device=X.device)
    ws_dw = torch.empty(tj.workspace_size(tj.TJ_OP_BWD_DW, M, N, K, 0), dtype=torch.uint8, device=X.device)
    r["dX"] = tj.linear_bwd_dx(dY, r["wq"], None, None, None, seed=seed, workspace=ws_dx)
    r["dW"] = tj.linear_bwd_dw(dY, r["xq"], None, None, None, seed=seed, workspace=ws_dw)
    torch.cuda.synchronize()
    tj.device_status()
    r["s_dy"], r["s_w"] = carve_workspace(ws_dx, [("nv", M, N), ("nv", K, N)])
    r["s_dyt"], r["s_x"] = carve_workspace(ws_dw, [("nv", N, M), ("nv", K, M)])
    return r


def _check_sampled(r, Xf, Wf, dYf, outl, seed, rng):
    """Sampled bit-exact operand rows and sampled product entries of one linear."""
    M, K = Xf.shape
    N = Wf.shape[0]
    o = np.asarray(outl, dtype=np.int64)
    k = len(o)
    nc = OL.normal_channels(K, o)
    kn = len(nc)
    m_s, n_s, c_s = _samples(M, 10, rng), _samples(N, 10, rng), _channel_samples(kn, rng)
    j_s = _samples(k, 3, rng) if k else np.zeros(0, np.int64)

    for name in ("xq", "wq", "s_dy", "s_w", "s_dyt", "s_x"):
        assert nvfp4_padding_is_zero(r[name]), name

    # forward: X-hat and W-hat rows, Y entries
    fx = OL.quantize_forward_operand(Xf[m_s], o)
    fw = OL.quantize_forward_operand(Wf[n_s], o)
    _rows_equal(nvfp4_to_logical(r["xq"]), fx["q"], m_s, "X-hat rows")
    _rows_equal(nvfp4_to_logical(r["wq"]), fw["q"], n_s, "W-hat rows")
    y_ref = OL.gemm_fp4(fx["q"], fw["q"])
    y_abs = _abs_nv(fx["q"], fw["q"])
    if k:
        _rows_equal(mxfp8_to_logical(r["x8"]), fx["q8"], m_s, "X-hat FP8 slice rows")
        y_ref = y_ref + OL.gemm_fp8(fx["q8"], fw["q8"])
        y_abs = y_abs + _abs_mx(fx["q8"], fw["q8"])
    y = _f32(r["Y"])[np.ix_(m_s, n_s)]
    assert_gemm_close(y, y_ref, y_abs, bf16=r["Y"].dtype == torch.bfloat16, what="Y (sampled)")

    # dX: S_dY rows m, S_W rows c (= W-hat column c along N), FP8 slice
    s_dy = OL.sr_rht_rows(dYf[m_s], seed, OL.TAG_DY_ROW, OL.TAG_RHT_DX, row_ids=m_s)
    _rows_equal(nvfp4_to_logical(r["s_dy"]), s_dy, m_s, "S_dY rows")
    wcols = _nv_deq_cols(Wf, nc, c_s)                                      # [|c_s|, N]
    s_w = OL.sr_rht_rows(wcols, seed, OL.TAG_WT, OL.TAG_RHT_DX, row_ids=c_s)
    _rows_equal(nvfp4_to_logical(r["s_w"]), s_w, c_s, "S_W rows (re-aligned W-hat^T)")
    dx = _f32(r["dX"])
    assert_gemm_close(dx[np.ix_(m_s, nc[c_s])], OL.gemm_fp4(s_dy, s_w, OL.ALPHA_RHT)[:, : len(c_s)],
                      _abs_nv(s_dy, s_w, OL.ALPHA_RHT)[:, : len(c_s)], bf16=r["dX"].dtype == torch.bfloat16,
                      what="dX normal channels (sampled)")
    if k:
        q8_dy = Q.quantize_mxfp8(dYf[m_s])
        _rows_equal(mxfp8_to_logical(r["q8_dy"]), q8_dy, m_s, "Q8(dY) rows")
        wo = _mx_deq_cols(Wf, o, j_s)
        q8_w = Q.quantize_mxfp8(wo)
        _rows_equal(mxfp8_to_logical(r["q8_w"]), q8_w, j_s, "Q8(W-hat_O^T) rows")
        assert_gemm_close(dx[np.ix_(m_s, o[j_s])], OL.gemm_fp8(q8_dy, q8_w)[:, : len(j_s)],
                          _abs_mx(q8_dy, q8_w)[:, : len(j_s)], bf16=r["dX"].dtype == torch.bfloat16,
                          what="dX outlier channels (sampled)")

    # dW: S_dY^T rows n (= dY column n along the tokens), S_X rows c, FP8 slice
    dyt = np.ascontiguousarray(dYf[:, n_s].T)
    s_dyt = OL.sr_rht_rows(dyt, seed, OL.TAG_DY_COL, OL.TAG_RHT_DW, row_ids=n_s)
    _rows_equal(nvfp4_to_logical(r["s_dyt"]), s_dyt, n_s, "S_dY^T rows")
    xcols = _nv_deq_cols(Xf, nc, c_s)                                      # [|c_s|, M]
    s_x = OL.sr_rht_rows(xcols, seed, OL.TAG_XT, OL.TAG_RHT_DW, row_ids=c_s)
    _rows_equal(nvfp4_to_logical(r["s_x"]), s_x, c_s, "S_X rows (re-aligned X-hat^T)")
    dw = r["dW"].cpu().numpy()
    assert_gemm_close(dw[np.ix_(n_s, nc[c_s])], OL.gemm_fp4(s_dyt, s_x, OL.ALPHA_RHT)[:, : len(c_s)],
                      _abs_nv(s_dyt, s_x, OL.ALPHA_RHT)[:, : len(c_s)], what="dW normal channels (sampled)")
    if k:
        q8_dyt = Q.quantize_mxfp8(dyt)
        _rows_equal(mxfp8_to_logical(r["q8_dyt"]), q8_dyt, n_s, "Q8(dY^T) rows")
        xo = _mx_deq_cols(Xf, o, j_s)
        q8_x = Q.quantize_mxfp8(xo)
        _rows_equal(mxfp8_to_logical(r["q8_x"]), q8_x, j_s, "Q8(X-hat_O^T) rows")
        assert_gemm_close(dw[np.ix_(n_s, o[j_s])], OL.gemm_fp8(q8_dyt, q8_x)[:, : len(j_s)],
                          _abs_mx(q8_dyt, q8_x)[:, : len(j_s)], what="dW outlier channels (sampled)")
    for name in ("Y", "dX", "dW"):
        assert torch.isfinite(r[name]).all(), name


def _calibrate_both(tj, K, seed, stream_id, k, dev, heavy=20):
    """The layer's OutControl calibration (four batches of 16384 tokens) on the GPU and in the
    oracle; the two outlier sets must be identical.  Returns the oracle's set."""
    sumsq_gpu = torch.zeros(K, dtype=torch.float64, device=dev)
    sumsq = np.zeros(K, dtype=np.float64)
    for b in range(4):
        xb = wl.device_calibration_batch(K, TOKENS, heavy, b, seed, stream_id, dev)
        tj.outlier_calibrate(xb, sumsq_gpu)
        sumsq = OC.accumulate_sumsq(_f32(xb), sumsq)
        del xb
    oi, _ = tj.outlier_calibrate(None, sumsq_gpu, finalize=True, k=k)
    outl, _ = OC.top_k_channels(sumsq, k)
    assert np.array_equal(oi.cpu().numpy().astype(np.int64), outl), "calibrated outlier sets differ"
    return outl


@pytest.mark.parametrize("layer", [n for n, _, _ in wl.LAYER_SET])
def test_layer_set_linear_full_size_sampled(tj, layer):
    """One linear of the decoder-layer set at 16384 tokens, in the benchmark's calls."""
    _, N, K = next(t for t in wl.LAYER_SET if t[0] == layer)
    dev = "cuda"
    seed_in, step_seed = 3, 1000
    X, W, dY = wl.device_layer_set_linear(layer, N, K, seed=seed_in, M=TOKENS, device=dev)
    k = OC.outlier_count(K, 10)
    outl = _calibrate_both(tj, K, seed_in, 700 + K, k, dev)
    ni = torch.from_numpy(OL.normal_channels(K, outl).astype(np.int32)).to(dev)
    oi = torch.from_numpy(outl.astype(np.int32)).to(dev)
    r = _run_steps(tj, X, W, dY, ni, oi, k, step_seed)
    _check_sampled(r, _f32(X), _f32(W), _f32(dY), outl, step_seed, np.random.default_rng(len(layer) + N))


def test_forward_outcontrol_full_size_sampled(tj):
    """Forward NVFP4 linear with OutControl, 16384 x 1024 -> 4096: calibration on four batches
    with 20 heavy channels, top 10% in FP8; through tj_linear_fwd into a bf16 output."""
    batches, X, W, _heavy = wl.fwd_outctl(seed=1)
    K = X.shape[1]
    k = OC.outlier_count(K, 10)
    sumsq = np.zeros(K, dtype=np.float64)
    sumsq_gpu = torch.zeros(K, dtype=torch.float64, device="cuda")
    for xb in batches:
        tj.outlier_calibrate(xb.cuda(), sumsq_gpu)
        sumsq = OC.accumulate_sumsq(xb.float().numpy(), sumsq)
    oi, ni = tj.outlier_calibrate(None, sumsq_gpu, finalize=True, k=k)
    outl, normal = OC.top_k_channels(sumsq, k)
    assert np.array_equal(oi.cpu().numpy().astype(np.int64), outl)
    assert np.array_equal(ni.cpu().numpy().astype(np.int64), normal)
    wq = tj.quantize_nvfp4(W.cuda(), sel=ni)
    w8 = tj.quantize_mxfp8(W.cuda(), sel=oi)
    y, xq, x8 = tj.linear_fwd(X.cuda(), wq, w8, ni, oi)
    torch.cuda.synchronize()
    tj.device_status()
    assert y.dtype == torch.bfloat16 and torch.isfinite(y).all()
    rng = np.random.default_rng(5)
    Xf, Wf = X.float().numpy(), W.float().numpy()
    m_s, n_s = _samples(X.shape[0], 12, rng), _samples(W.shape[0], 12, rng)
    fx = OL.quantize_forward_operand(Xf[m_s], outl)
    fw = OL.quantize_forward_operand(Wf[n_s], outl)
    _rows_equal(nvfp4_to_logical(xq), fx["q"], m_s, "X-hat rows")
    _rows_equal(mxfp8_to_logical(x8), fx["q8"], m_s, "X-hat FP8 slice rows")
    _rows_equal(nvfp4_to_logical(wq), fw["q"], n_s, "W-hat rows")
    y_ref = OL.gemm_fp4(fx["q"], fw["q"]) + OL.gemm_fp8(fx["q8"], fw["q8"])
    y_abs = _abs_nv(fx["q"], fw["q"]) + _abs_mx(fx["q8"], fw["q8"])
    assert_gemm_close(_f32(y)[np.ix_(m_s, n_s)], y_ref, y_abs, bf16=True, what="Y (sampled)")


def test_backward_rht_sr_full_size_sampled(tj):
    """Backward NVFP4 linear with RHT and SR, dY 16384 x 4096 (Student-t rows), W 4096 x 1024,
    X 16384 x 1024, through tj_linear_fwd / bwd_dx / bwd_dw without outlier channels."""
    dY, W, X = wl.bwd_rht(seed=2)
    r = _run_api(tj, X.cuda(), W.cuda(), dY.cuda(), seed=2)
    _check_sampled(r, X.float().numpy(), W.float().numpy(), dY.float().numpy(), np.zeros(0, np.int64), 2,
                   np.random.default_rng(11))


@pytest.mark.parametrize("along", [False, True])
@pytest.mark.parametrize("mode", [0, 1])
def test_quantize_sweep_full_size_sampled(tj, along, mode):
    """The quantize-only sweep's largest tensor, 16384 x 4096 bf16 with 1% of the columns x30,
    in the benchmark's call: sampled rows (or columns) bit for bit."""
    rows, cols = 16384, 4096
    x = wl.device_heavy_columns((rows, cols), 1.0, 30.0, math.ceil(cols / 100), 0, 11, "cuda")
    q = tj.NVFP4.empty(cols if along else rows, rows if along else cols, "cuda")
    tj.quantize_nvfp4(x, along_cols=along, mode=mode, seed=1, tag=1, out=q)
    torch.cuda.synchronize()
    tj.device_status()
    assert nvfp4_padding_is_zero(q)
    xf = _f32(x)
    rng = np.random.default_rng(17 + 2 * mode + int(along))
    if along:
        s = _samples(cols, 14, rng)
        ref = Q.quantize_nvfp4(np.ascontiguousarray(xf[:, s].T), mode, seed=1, tag=1, row_ids=s)
    else:
        s = _samples(rows, 14, rng)
        ref = Q.quantize_nvfp4(xf[s], mode, seed=1, tag=1, row_ids=s)
    _rows_equal(nvfp4_to_logical(q), ref, s, "sampled %s" % ("columns" if along else "rows"))


def test_osci_reset_full_size_sampled(tj):
    """OsciReset over all 369,098,752 master weights of the benchmark (22 layers of the set, as
    [n / 1024, 1024] fp32), four passes with a synthetic update before each (a random step
    plus +-3e-4 on a fixed 5% of the weights, so that weights oscillate) and a learning rate
    that crosses the threshold.  Sampled rows of every piece of state, the reset mask and the
    emitted forward weight must equal the oracle's trajectory of those rows bit for bit."""
    from oracle import osci as OO

    lr_thr, risk_thr = 1e-4, 4.0
    w = wl.device_master_weights(wl.OSCI_PARAMS, seed=3, device="cuda")
    rows, cols = w.shape
    rng = np.random.default_rng(23)
    r_s = _samples(rows, 14, rng)
    w_prev = w.clone()
    dq = torch.zeros_like(w)
    dm = torch.zeros_like(w)
    q = [tj.quantize_nvfp4(w), tj.NVFP4.empty(rows, cols)]
    mask = torch.empty(rows * ((cols + 31) // 32), dtype=torch.int32, device="cuda")
    w_ref = _f32(w[r_s])
    state = OO.init_state(w_ref)
    g = torch.Generator(device="cuda")
    g.manual_seed(29)
    osc = torch.rand(w.shape, generator=g, device="cuda") < 0.05
    resets = 0
    for t, lr in enumerate((2e-4, 8e-5, 4e-5, 1e-5)):
        step = torch.randn(w.shape, generator=g, device="cuda") * lr
        step = torch.where(osc, torch.full_like(step, 3e-4 * (1 if t % 2 == 0 else -1)), step)
        w.add_(step)
        w_ref = (w_ref + _f32(step[r_s])).astype(np.float32)
        del step
        tj.osci_reset(w, w_prev, dq, dm, q[0], q[1], mask, lr, lr_thr, risk_thr)
        w_ref, state, m_ref, q_ref = OO.osci_reset_step(w_ref, state, lr, lr_thr, risk_thr)
        torch.cuda.synchronize()
        tj.device_status()
        assert np.array_equal(_f32(w[r_s]), w_ref), t
        assert np.array_equal(_f32(w_prev[r_s]), state["w_prev"]), t
        assert np.array_equal(_f32(dq[r_s]), state["dist_q"]), t
        assert np.array_equal(_f32(dm[r_s]), state["dist_m"]), t
        words = mask.view(rows, -1)[r_s].cpu().numpy().view(np.uint32)
        bits = ((words[:, :, None] >> np.arange(32, dtype=np.uint32)) & 1).reshape(len(r_s), -1)[:, :cols]
        assert np.array_equal(bits.astype(bool), m_ref), t
        _rows_equal(nvfp4_to_logical(q[1]), q_ref, r_s, "forward weight, pass %d" % t)
        resets += int(m_ref.sum())
        q.reverse()
    assert resets > 0


def test_adamw_osci_reset_full_size_sampled(tj):
    """The fused training-step pass (AdamW, OsciReset, forward-weight quantization) over all
    369,098,752 master weights, four steps with a synthetic gradient (5% of the weights get an
    alternating +-0.05, the rest N(0, 1e-2)) and a learning rate that crosses the threshold:
    sampled rows of w, m, v, the OsciReset state, the mask and the forward weight equal the
    oracle's AdamW step followed by its OsciReset step, bit for bit."""
    from oracle import osci as OO

    lr_thr, risk_thr, b1, b2, eps, wd = 1e-4, 0.5, 0.9, 0.95, 1e-8, 0.1
    w = wl.device_master_weights(wl.OSCI_PARAMS, seed=3, device="cuda")
    rows, cols = w.shape
    rng = np.random.default_rng(31)
    r_s = _samples(rows, 14, rng)
    m_dev, v_dev = torch.zeros_like(w), torch.zeros_like(w)
    w_prev = w.clone()
    dq = torch.zeros_like(w)
    dm = torch.zeros_like(w)
    q = [tj.quantize_nvfp4(w), tj.NVFP4.empty(rows, cols)]
    mask = torch.empty(rows * ((cols + 31) // 32), dtype=torch.int32, device="cuda")
    w_ref = _f32(w[r_s])
    m_ref = np.zeros_like(w_ref)
    v_ref = np.zeros_like(w_ref)
    state = OO.init_state(w_ref)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(37)
    osc = torch.rand(w.shape, generator=gen, device="cuda") < 0.05
    resets = 0
    for t, lr in enumerate((2e-4, 8e-5, 4e-5, 1e-5), start=1):
        g = torch.randn(w.shape, generator=gen, device="cuda") * 1e-2
        g = torch.where(osc, torch.full_like(g, 0.05 * (1 if t % 2 else -1)), g)
        tj.adamw_osci_reset(w, g, m_dev, v_dev, w_prev, dq, dm, q[0], q[1], mask, lr, b1, b2, eps, wd, t, lr_thr,
                            risk_thr)
        w_ref, m_ref, v_ref, state, mk_ref, q_ref = OO.adamw_osci_reset_step(
            w_ref, _f32(g[r_s]), m_ref, v_ref, state, lr, b1, b2, eps, wd, t, lr_thr, risk_thr)
        del g
        torch.cuda.synchronize()
        tj.device_status()
        for name, got, ref in (("w", w, w_ref), ("m", m_dev, m_ref), ("v", v_dev, v_ref),
                               ("w_prev", w_prev, state["w_prev"]), ("dist_Q", dq, state["dist_q"]),
                               ("dist_M", dm, state["dist_m"])):
            assert np.array_equal(_f32(got[r_s]), ref), (name, t)
        words = mask.view(rows, -1)[r_s].cpu().numpy().view(np.uint32)
        bits = ((words[:, :, None] >> np.arange(32, dtype=np.uint32)) & 1).reshape(len(r_s), -1)[:, :cols]
        assert np.array_equal(bits.astype(bool), mk_ref), t
        _rows_equal(nvfp4_to_logical(q[1]), q_ref, r_s, "forward weight, step %d" % t)
        resets += int(mk_ref.sum())
        q.reverse()
    assert resets > 0


def test_fp6_fp4_slice_full_size_sampled(tj):
    """The FP6 x FP4 outlier slice at the forward-with-OutControl shapes (16384 x 1024 -> 4096,
    103 outlier channels) in the calls the benchmark times: X's slice in E2M3, W's in E2M1;
    backward with dY 16384 x 4096 (Student-t rows), whose slices take the partner formats
    (dX: E2M3 x E2M1, dW: E2M1 x E2M3).  Sampled slice rows bit-exact; sampled Y and the
    outlier columns of dX and dW within tolerance."""
    from oracle import formats as F

    E2M3, E2M1 = F.MX_E2M3, F.MX_E2M1
    batches, X, W, _heavy = wl.fwd_outctl(seed=1)
    dY = wl.bwd_rht(seed=2)[0]
    K = X.shape[1]
    k = OC.outlier_count(K, 10)
    sumsq = np.zeros(K, dtype=np.float64)
    sumsq_gpu = torch.zeros(K, dtype=torch.float64, device="cuda")
    for xb in batches:
        tj.outlier_calibrate(xb.cuda(), sumsq_gpu)
        sumsq = OC.accumulate_sumsq(xb.float().numpy(), sumsq)
    oi, ni = tj.outlier_calibrate(None, sumsq_gpu, finalize=True, k=k)
    outl, _ = OC.top_k_channels(sumsq, k)
    assert np.array_equal(oi.cpu().numpy().astype(np.int64), outl)
    M, N = X.shape[0], W.shape[0]
    wq = tj.quantize_nvfp4(W.cuda(), sel=ni)
    w8 = tj.quantize_mxfp8(W.cuda(), sel=oi, fmt=E2M1)
    y, xq, x8 = tj.linear_fwd(X.cuda(), wq, w8, ni, oi, fmt_x8=E2M3)
    seed = 1001
    dx = tj.linear_bwd_dx(dY.cuda(), wq, w8, ni, oi, seed=seed, out_dtype=torch.float32)
    dw = tj.linear_bwd_dw(dY.cuda(), xq, x8, ni, oi, seed=seed)
    torch.cuda.synchronize()
    tj.device_status()

    rng = np.random.default_rng(9)
    Xf, Wf, dYf = X.float().numpy(), W.float().numpy(), dY.float().numpy()
    m_s, n_s = _samples(M, 10, rng), _samples(N, 10, rng)
    fx = OL.quantize_forward_operand(Xf[m_s], outl, E2M3)
    fw = OL.quantize_forward_operand(Wf[n_s], outl, E2M1)
    _rows_equal(mxfp8_to_logical(x8), fx["q8"], m_s, "X-hat E2M3 slice rows")
    _rows_equal(mxfp8_to_logical(w8), fw["q8"], n_s, "W E2M1 slice rows")
    _rows_equal(nvfp4_to_logical(xq), fx["q"], m_s, "X-hat rows")
    abs_mx = lambda qa, fa, qb, fb: np.abs(Q.dequantize_mx_f64(*qa, fa)) @ np.abs(Q.dequantize_mx_f64(*qb, fb)).T
    y_ref = OL.gemm_fp4(fx["q"], fw["q"]) + OL.gemm_mx(fx["q8"], E2M3, fw["q8"], E2M1)
    y_abs = _abs_nv(fx["q"], fw["q"]) + abs_mx(fx["q8"], E2M3, fw["q8"], E2M1)
    assert_gemm_close(_f32(y)[np.ix_(m_s, n_s)], y_ref, y_abs, bf16=True, what="Y (sampled)")

    # dX on the outlier channels: Q_E2M3(dY rows) x Q_E2M1(W-hat_O^T)^T
    w_slice = Q.quantize_mx(Wf[:, outl], E2M1)
    q8_w = Q.quantize_mx(np.ascontiguousarray(Q.dequantize_mx_f32(*w_slice, E2M1)[:, :k].T), E2M1)
    q8_dy = Q.quantize_mx(dYf[m_s], E2M3)
    dx_ref = OL.gemm_mx(q8_dy, E2M3, q8_w, E2M1)[:, :k]
    dx_abs = abs_mx(q8_dy, E2M3, q8_w, E2M1)[:, :k]
    assert_gemm_close(_f32(dx)[np.ix_(m_s, outl)], dx_ref, dx_abs, what="dX outlier columns (sampled rows)")

    # dW on the outlier channels: Q_E2M1(dY^T rows) x Q_E2M3(X-hat_O^T)^T
    x_slice = Q.quantize_mx(Xf[:, outl], E2M3)
    q8_x = Q.quantize_mx(np.ascontiguousarray(Q.dequantize_mx_f32(*x_slice, E2M3)[:, :k].T), E2M3)
    q8_dyt = Q.quantize_mx(np.ascontiguousarray(dYf[:, n_s].T), E2M1)
    dw_ref = OL.gemm_mx(q8_dyt, E2M1, q8_x, E2M3)[:, :k]
    dw_abs = abs_mx(q8_dyt, E2M1, q8_x, E2M3)[:, :k]
    assert_gemm_close(_f32(dw)[np.ix_(n_s, outl)], dw_ref, dw_abs, what="dW outlier columns (sampled rows)")
