"""GPU parity of the FP6 x FP4 outlier-slice variant (technical summary §5 names FP6 x FP4 as
a future direction; the slice rule is the FP8 slice's with each format's maximum).

  * the MX quantizers in E2M3 / E3M2 / E2M1, bit for bit against the oracle: rows,
    transposed, gathered columns, the one-read dual pass (with the RHT's sign-flipped rows),
    the OutControl split, the re-alignment from one format into another, dequantization;
  * the slice GEMMs with FP6 x FP4 (and other mixed) operands, alone, in one tile with an
    FP4 product, in pair launches: within 2e-3 sum|a||b| of the oracle;
  * the linear layer with an FP6 x FP4 slice: saved context and backward operands bit-exact
    (the dY slice in the partner format), Y / dX / dW within tolerance.
Inputs hold ties (grid midpoints at an exact block scale), negative zeros, values that round
to zero, all-zero blocks and ragged edges.
"""
import numpy as np
import pytest
import torch

from layouts import abs_product, assert_gemm_close, assert_mxfp8_equal, assert_nvfp4_equal, carve_workspace
from oracle import formats as F
from oracle import linear as OL
from oracle import quant as Q

pytestmark = pytest.mark.gpu

SUB = [F.MX_E2M3, F.MX_E3M2, F.MX_E2M1]
PAIRS = [(F.MX_E2M3, F.MX_E2M1), (F.MX_E3M2, F.MX_E2M1), (F.MX_E2M1, F.MX_E2M3), (F.MX_E4M3, F.MX_E2M1),
         (F.MX_E2M3, F.MX_E3M2)]


@pytest.fixture(scope="module")
def tj():
    from nvfp4_bit_fully_gb300 import tj as _tj

    _tj.load()
    return _tj


def _input(rows, cols, dtype, seed, fmt):
    """Gaussian rows with heavy columns; rows 0-3 carry exact ties of fmt (the block maximum
    fixes the scale 2^e, the other elements are grid midpoints times 2^e), negative zeros and
    values far below the smallest step; row 5's first block is zero."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g)
    x[:, torch.randperm(cols, generator=g)[: max(1, cols // 40)]] *= 25
    vals = F.mx_elem_decode(np.arange(0x7F if fmt == F.MX_E4M3 else (8 if fmt == F.MX_E2M1 else 32)), fmt)
    mids = (vals[1:] + vals[:-1]) / 2
    rng = np.random.default_rng(seed)
    for r in range(min(4, rows)):
        for b0 in range(0, cols - 31, 32):
            e = int(rng.integers(-6, 6))
            blk = rng.choice(mids, 32) * rng.choice([-1.0, 1.0], 32)
            blk[0] = F.MX_MAX[fmt]
            x[r, b0:b0 + 32] = torch.from_numpy(blk * 2.0 ** e)
    if rows > 4:
        x[4, :: 3] = -0.0
        x[4, 1:: 3] = -1e-30
    if rows > 5:
        x[5, : min(32, cols)] = 0.0
    return x.to(dtype)


@pytest.mark.parametrize("fmt", SUB)
@pytest.mark.parametrize("rows,cols,dtype", [(256, 512, torch.float32), (200, 300, torch.bfloat16),
                                             (64, 136, torch.float32)])
def test_quantize_rows_and_columns_bit_exact(tj, fmt, rows, cols, dtype):
    x = _input(rows, cols, dtype, rows + cols + fmt, fmt)
    xf = x.float().numpy()
    q = tj.quantize_mxfp8(x.cuda(), fmt=fmt)
    qt = tj.quantize_mxfp8(x.cuda(), along_cols=True, fmt=fmt)
    torch.cuda.synchronize()
    assert_mxfp8_equal(q, Q.quantize_mx(xf, fmt), "rows fmt %d" % fmt)
    assert_mxfp8_equal(qt, Q.quantize_mx(np.ascontiguousarray(xf.T), fmt), "columns fmt %d" % fmt)


@pytest.mark.parametrize("fmt", SUB)
def test_quantize_selected_columns(tj, fmt):
    x = _input(192, 400, torch.bfloat16, 7 + fmt, fmt)
    sel = np.sort(np.random.default_rng(fmt).choice(400, 71, replace=False)).astype(np.int32)
    q = tj.quantize_mxfp8(x.cuda(), sel=torch.from_numpy(sel).cuda(), fmt=fmt)
    torch.cuda.synchronize()
    assert_mxfp8_equal(q, Q.quantize_mx(x.float().numpy()[:, sel], fmt), "gathered")


@pytest.mark.parametrize("fmt", SUB)
@pytest.mark.parametrize("along_cols", [False, True])
def test_dual_pass_slice_with_rht(tj, fmt, along_cols):
    """The NVFP4 + slice pass of dY: the slice (no RHT) from the same read as the RHT + SR
    operand; in the transposed kernel the rows were loaded sign-flipped for the RHT."""
    x = _input(256, 384, torch.bfloat16, 30 + fmt, fmt)
    q, q8 = tj.quantize_nvfp4_mxfp8(x.cuda(), along_cols=along_cols, mode=tj.TJ_SR, rht=True, seed=9, tag=2,
                                    rht_tag=0x101, fmt8=fmt)
    torch.cuda.synchronize()
    xf = x.float().numpy()
    src = np.ascontiguousarray(xf.T) if along_cols else xf
    assert_mxfp8_equal(q8, Q.quantize_mx(src, fmt), "dual slice")
    assert_nvfp4_equal(q, OL.sr_rht_rows(src, 9, 2, 0x101), "dual NVFP4")


@pytest.mark.parametrize("fmt", SUB)
def test_outcontrol_split(tj, fmt):
    x = _input(300, 1024, torch.bfloat16, 40 + fmt, fmt)
    o = np.sort(np.random.default_rng(5).choice(1024, 103, replace=False))
    nc = OL.normal_channels(1024, o)
    q, q8 = tj.quantize_split(x.cuda(), torch.from_numpy(nc.astype(np.int32)).cuda(),
                              torch.from_numpy(o.astype(np.int32)).cuda(), fmt8=fmt)
    torch.cuda.synchronize()
    xf = x.float().numpy()
    assert_mxfp8_equal(q8, Q.quantize_mx(xf[:, o], fmt), "split slice")
    assert_nvfp4_equal(q, Q.quantize_nvfp4(xf[:, nc], Q.RTN), "split NVFP4")


@pytest.mark.parametrize("fin,fout", [(F.MX_E2M3, F.MX_E2M3), (F.MX_E2M1, F.MX_E2M1), (F.MX_E3M2, F.MX_E2M1),
                                      (F.MX_E4M3, F.MX_E2M3), (F.MX_E2M1, F.MX_E4M3)])
def test_realignment_between_formats_and_dequantize(tj, fin, fout):
    x = _input(200, 330, torch.float32, 50 + fin + 3 * fout, fin)
    q = tj.quantize_mxfp8(x.cuda(), fmt=fin)
    r = tj.requantize_mxfp8(q, fmt=fout)
    y = tj.dequantize_mxfp8(q)
    torch.cuda.synchronize()
    ref = Q.quantize_mx(x.float().numpy(), fin)
    deq = Q.dequantize_mx_f32(*ref, fin)[:, :330]
    assert np.array_equal(y.cpu().numpy(), deq)
    assert_mxfp8_equal(r, Q.quantize_mx(np.ascontiguousarray(deq.T), fout), "re-aligned")


def abs_product_mx(qa, fa, qb, fb):
    return np.abs(Q.dequantize_mx_f64(*qa, fa)) @ np.abs(Q.dequantize_mx_f64(*qb, fb)).T


def _slice_operands(tj, M, N, k, fa, fb, seed):
    g = torch.Generator().manual_seed(seed)
    A = (torch.randn(M, k, generator=g) * 30.0).to(torch.bfloat16)
    B = (torch.randn(N, k, generator=g) * 0.05).to(torch.bfloat16)
    a8 = tj.quantize_mxfp8(A.cuda(), fmt=fa)
    b8 = tj.quantize_mxfp8(B.cuda(), fmt=fb)
    ra, rb = Q.quantize_mx(A.float().numpy(), fa), Q.quantize_mx(B.float().numpy(), fb)
    torch.cuda.synchronize()
    assert_mxfp8_equal(a8, ra, "A slice")
    assert_mxfp8_equal(b8, rb, "B slice")
    return a8, b8, ra, rb


@pytest.mark.parametrize("fa,fb", PAIRS)
@pytest.mark.parametrize("M,N,k", [(128, 128, 128), (256, 103, 103), (300, 410, 700)])
def test_slice_gemm_mixed_formats(tj, fa, fb, M, N, k):
    a8, b8, ra, rb = _slice_operands(tj, M, N, k, fa, fb, seed=M + k + fa + fb)
    d = tj.gemm_mxfp8(a8, b8)
    torch.cuda.synchronize()
    tj.device_status()
    assert_gemm_close(d.cpu().numpy(), OL.gemm_mx(ra, fa, rb, fb), abs_product_mx(ra, fa, rb, fb),
                      what="slice %d x %d" % (fa, fb))


def _fp4_operands(tj, M, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16)
    qa, qb = tj.quantize_nvfp4(A.cuda()), tj.quantize_nvfp4(B.cuda())
    return qa, qb, Q.quantize_nvfp4(A.float().numpy(), Q.RTN), Q.quantize_nvfp4(B.float().numpy(), Q.RTN)


def test_fp4_product_with_fp6_fp4_slice_in_one_tile(tj):
    M, N, K, k = 256, 256, 384, 103
    qa, qb, ra, rb = _fp4_operands(tj, M, N, K, 3)
    a8, b8, ra8, rb8 = _slice_operands(tj, M, N, k, F.MX_E2M3, F.MX_E2M1, 4)
    d = tj.gemm_nvfp4(qa, qb, a8, b8)
    torch.cuda.synchronize()
    tj.device_status()
    ref = OL.gemm_fp4(ra, rb) + OL.gemm_mx(ra8, F.MX_E2M3, rb8, F.MX_E2M1)
    bound = abs_product(ra, rb) + abs_product_mx(ra8, F.MX_E2M3, rb8, F.MX_E2M1)
    assert_gemm_close(d.cpu().numpy(), ref, bound, what="fp4 + fp6 x fp4 slice")


def test_pair_launches_with_fp6_fp4_slice(tj):
    M, N, N8, K, k = 384, 300, 96, 2048, 1024
    qa, qb, ra, rb = _fp4_operands(tj, M, N, K, 5)
    a8, b8, ra8, rb8 = _slice_operands(tj, M, N8, k, F.MX_E2M1, F.MX_E2M3, 6)
    perm = torch.randperm(N + N8, generator=torch.Generator().manual_seed(9)).to(torch.int32)
    cm, cm8 = perm[:N].sort().values.cuda(), perm[N:].sort().values.cuda()
    out = torch.full((M, N + N8), -3.0, device="cuda")
    tj.gemm_pair(qa, qb, a8, b8, alpha=2.0 ** -7, out=out, out8=out, col_map=cm, col_map8=cm8)
    out32 = torch.full((M, N + N8), 5.0, device="cuda")
    tj.gemm_pair_f32(qa, qb, a8, b8, out32, cm, cm8, alpha=2.0 ** -7)     # K long enough to split
    torch.cuda.synchronize()
    tj.device_status()
    ref4, b4 = OL.gemm_fp4(ra, rb, 2.0 ** -7), abs_product(ra, rb, 2.0 ** -7)
    ref8, b8_ = OL.gemm_mx(ra8, F.MX_E2M1, rb8, F.MX_E2M3), abs_product_mx(ra8, F.MX_E2M1, rb8, F.MX_E2M3)
    for got, what in ((out, "pair"), (out32, "pair_f32")):
        g_ = got.cpu().numpy()
        assert_gemm_close(g_[:, cm.cpu().numpy()], ref4, b4, what=what + " fp4")
        assert_gemm_close(g_[:, cm8.cpu().numpy()], ref8, b8_, what=what + " fp4 x fp6 slice")


SLICE_PAIRS = [(F.MX_E2M3, F.MX_E2M1), (F.MX_E3M2, F.MX_E2M1), (F.MX_E2M1, F.MX_E2M3)]


def _slice_layer(rng, M, N, K, k):
    X = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32))
    outl = np.sort(rng.choice(K, k, replace=False))
    X[:, torch.from_numpy(outl)] *= 20
    X = X.to(torch.bfloat16)
    W = torch.from_numpy((rng.standard_normal((N, K)) * 0.05).astype(np.float32)).to(torch.bfloat16)
    dY = torch.from_numpy(rng.standard_normal((M, N)).astype(np.float32)).to(torch.bfloat16)
    return X, W, dY, outl


@pytest.mark.parametrize("fmt_x,fmt_w", SLICE_PAIRS)
def test_linear_with_fp6_fp4_slice(tj, fmt_x, fmt_w):
    rng = np.random.default_rng(fmt_x * 7 + fmt_w)
    X, W, dY, outl = _slice_layer(rng, 256, 320, 512, 40)
    _check_slice_linear(tj, X, W, dY, outl, fmt_x, fmt_w, 21)


@pytest.mark.parametrize("case", range(6))
def test_linear_with_fp6_fp4_slice_random_shapes(tj, case):
    """Six seeded random layers (M, N, K from one element to a few tiles, 1 to 80 outlier
    channels), each with a random FP6 x FP4 slice pairing, under the same checks."""
    rng = np.random.default_rng(5000 + case)
    M, N, K = int(rng.integers(1, 520)), int(rng.integers(1, 400)), int(rng.integers(2, 600))
    k = int(rng.integers(1, min(K, 80) + 1))
    fmt_x, fmt_w = SLICE_PAIRS[int(rng.integers(0, len(SLICE_PAIRS)))]
    X, W, dY, outl = _slice_layer(rng, M, N, K, k)
    _check_slice_linear(tj, X, W, dY, outl, fmt_x, fmt_w, 31 + case)


def _check_slice_linear(tj, X, W, dY, outl, fmt_x, fmt_w, seed):
    M, K = X.shape
    N = W.shape[0]
    k = len(outl)
    nc = OL.normal_channels(K, outl)
    ni, oi = torch.from_numpy(nc.astype(np.int32)).cuda(), torch.from_numpy(outl.astype(np.int32)).cuda()
    wq = tj.quantize_nvfp4(W.cuda(), sel=ni)
    w8 = tj.quantize_mxfp8(W.cuda(), sel=oi, fmt=fmt_w)
    y, xq, x8 = tj.linear_fwd(X.cuda(), wq, w8, ni, oi, out_dtype=torch.float32, fmt_x8=fmt_x)
    ws_dx = torch.empty(tj.workspace_size(tj.TJ_OP_BWD_DX, M, N, K, k), dtype=torch.uint8, device="cuda")
    ws_dw = torch.empty(tj.workspace_size(tj.TJ_OP_BWD_DW, M, N, K, k), dtype=torch.uint8, device="cuda")
    dx = tj.linear_bwd_dx(dY.cuda(), wq, w8, ni, oi, seed=seed, out_dtype=torch.float32, workspace=ws_dx)
    dw = tj.linear_bwd_dw(dY.cuda(), xq, x8, ni, oi, seed=seed, workspace=ws_dw)
    torch.cuda.synchronize()
    tj.device_status()

    Xf, Wf, dYf = X.float().numpy(), W.float().numpy(), dY.float().numpy()
    Y_ref, fx, fw = OL.forward(Xf, Wf, outl, fmt_x=fmt_x, fmt_w=fmt_w)
    assert_nvfp4_equal(xq, fx["q"], "X-hat")
    assert_mxfp8_equal(x8, fx["q8"], "X-hat slice")
    assert_gemm_close(y.cpu().numpy(), Y_ref, abs_product(fx["q"], fw["q"]) +
                      abs_product_mx(fx["q8"], fmt_x, fw["q8"], fmt_w), what="Y")

    K_N = K - k
    pdx = OL.SLICE_PARTNER[fmt_w]
    s_dy, s_w, q8_dy, q8_w = OL.bwd_dx_operands(dYf, fw, seed)
    views = carve_workspace(ws_dx, [("nv", M, N), ("nv", K_N, N), ("mx", M, N, pdx), ("mx", k, N, fmt_w)])
    assert_mxfp8_equal(views[2], q8_dy, "dY slice")
    assert_mxfp8_equal(views[3], q8_w, "W-hat_O^T slice")
    bx = np.zeros((M, K))
    bx[:, nc] = abs_product(s_dy, s_w, OL.ALPHA_RHT)[:, :K_N]
    bx[:, outl] = abs_product_mx(q8_dy, pdx, q8_w, fmt_w)[:, :k]
    assert_gemm_close(dx.cpu().numpy(), OL.bwd_dx(dYf, fw, outl, seed), bx, what="dX")

    pdw = OL.SLICE_PARTNER[fmt_x]
    s_dyt, s_x, q8_dyt, q8_x = OL.bwd_dw_operands(dYf, fx, seed)
    views = carve_workspace(ws_dw, [("nv", N, M), ("nv", K_N, M), ("mx", N, M, pdw), ("mx", k, M, fmt_x)])
    assert_mxfp8_equal(views[2], q8_dyt, "dY^T slice")
    assert_mxfp8_equal(views[3], q8_x, "X-hat_O^T slice")
    bw = np.zeros((N, K))
    bw[:, nc] = abs_product(s_dyt, s_x, OL.ALPHA_RHT)[:, :K_N]
    bw[:, outl] = abs_product_mx(q8_dyt, pdw, q8_x, fmt_x)[:, :k]
    assert_gemm_close(dw.cpu().numpy(), OL.bwd_dw(dYf, fx, outl, seed), bw, what="dW")


@pytest.mark.parametrize("fmt", [F.MX_E4M3] + SUB)
def test_extreme_magnitudes(tj, fmt):
    """Blocks near the top of fp32 (the scale exponent near +127), blocks of fp32-subnormal
    values (the exponent clamped at -127, elements far below a step), blocks mixing a huge
    maximum with tiny elements, and exact powers of two: codes and scales bit for bit, in
    both orientations."""
    rng = np.random.default_rng(77 + fmt)
    rows, cols = 64, 256
    x = rng.standard_normal((rows, cols)).astype(np.float32)
    x[0:8] *= np.float32(1e37)                                  # amax up to ~4e37
    x[8, :32] = np.float32(3.0e38)
    x[8, 32:64] = -np.float32(3.3e38)
    x[9:16] = (rng.standard_normal((7, cols)) * 1e-39).astype(np.float32)   # subnormal
    x[16:24, ::32] = np.float32(1e30)
    x[16:24, 1::32] = np.float32(1e-30)
    x[24:32] = np.exp2(rng.integers(-140, 120, (8, cols))).astype(np.float32) * rng.choice([-1, 1], (8, cols))
    t = torch.from_numpy(x).cuda()
    q = tj.quantize_mxfp8(t, fmt=fmt)
    qt = tj.quantize_mxfp8(t, along_cols=True, fmt=fmt)
    y = tj.dequantize_mxfp8(q)
    torch.cuda.synchronize()
    ref = Q.quantize_mx(x, fmt)
    assert_mxfp8_equal(q, ref, "rows, extreme magnitudes")
    assert_mxfp8_equal(qt, Q.quantize_mx(np.ascontiguousarray(x.T), fmt), "columns, extreme magnitudes")
    assert np.array_equal(y.cpu().numpy(), Q.dequantize_mx_f32(*ref, fmt)[:, :cols])
