"""GPU: empty and degenerate inputs through the C ABI.

An empty tensor (no rows or no columns) has no storage, so its pointers may be null (an
empty torch tensor hands over a null data pointer); a call whose outputs are empty does
nothing and succeeds; a product over an empty contraction is zero and is written as zeros
(dX with no output features, dW with no tokens, any GEMM with K = 0).  The degenerate
OutControl splits -- every channel an outlier, or none -- are checked against the oracle
in ``test_gpu_linear.py``.
"""
import numpy as np
import pytest
import torch

from layouts import assert_mxfp8_equal, assert_nvfp4_equal
from oracle import linear as OL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tj():
    from nvfp4_bit_fully_gb300 import tj as _tj

    _tj.load()
    return _tj


def _x(rows, cols, seed=0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(rows, cols, generator=g).to(torch.bfloat16).cuda()


@pytest.mark.parametrize("rows,cols", [(0, 300), (5, 0), (0, 0)])
@pytest.mark.parametrize("along", [False, True])
def test_quantize_empty(tj, rows, cols, along):
    x = _x(rows, cols)
    q = tj.quantize_nvfp4(x, along_cols=along, mode=tj.TJ_SR, rht=True, seed=1, tag=2, rht_tag=3)
    q8 = tj.quantize_mxfp8(x, along_cols=along)
    qd, qd8 = tj.quantize_nvfp4_mxfp8(x, along_cols=along, mode=tj.TJ_SR, rht=True, seed=1, tag=2, rht_tag=3)
    torch.cuda.synchronize()
    shape = (cols, rows) if along else (rows, cols)
    for t in (q, q8, qd, qd8):
        assert (t.rows, t.cols) == shape
    tj.device_status()


def test_quantize_no_selected_channels(tj):
    x = _x(64, 256)
    none = torch.empty(0, dtype=torch.int32, device="cuda")
    q = tj.quantize_nvfp4(x, sel=none)
    q8 = tj.quantize_mxfp8(x, sel=none)
    torch.cuda.synchronize()
    assert (q.rows, q.cols, q8.rows, q8.cols) == (64, 0, 64, 0)


def test_split_and_requantize_empty(tj):
    x = _x(0, 256)
    ni = torch.arange(0, 200, dtype=torch.int32, device="cuda")
    oi = torch.arange(200, 256, dtype=torch.int32, device="cuda")
    xq, x8 = tj.quantize_split(x, ni, oi)
    assert (xq.rows, xq.cols, x8.rows, x8.cols) == (0, 200, 0, 56)
    r = tj.requantize_nvfp4(xq, tj.TJ_SR, True, 1, 2, 3)
    r8 = tj.requantize_mxfp8(x8)
    p, p8 = tj.requantize_nvfp4_mxfp8(xq, x8, tj.TJ_SR, True, 1, 2, 3)
    torch.cuda.synchronize()
    for t in (r, p):
        assert (t.rows, t.cols) == (200, 0)
    for t in (r8, p8):
        assert (t.rows, t.cols) == (56, 0)
    assert tj.dequantize_nvfp4(xq).shape == (0, 200)
    assert tj.dequantize_mxfp8(x8).shape == (0, 56)
    assert tj.rht(torch.empty(0, 256, device="cuda"), 1, 2).shape == (0, 256)


def test_realignment_pair_with_one_empty_part(tj):
    """A pair launch whose NVFP4 part or slice is empty equals the other part's own call."""
    x = _x(300, 256, seed=4)
    all_ch = torch.arange(256, dtype=torch.int32, device="cuda")
    none = torch.empty(0, dtype=torch.int32, device="cuda")
    for ni, oi in ((none, all_ch), (all_ch, none)):
        xq, x8 = tj.quantize_split(x, ni, oi)
        x8 = x8 if x8 is not None else tj.MXFP8.empty(300, 0)        # no outlier: an empty slice
        a, a8 = tj.requantize_nvfp4_mxfp8(xq, x8, tj.TJ_SR, True, 7, 4, 0x101)
        b = tj.requantize_nvfp4(xq, tj.TJ_SR, True, 7, 4, 0x101)
        b8 = tj.requantize_mxfp8(x8)
        torch.cuda.synchronize()
        for u, v in ((a.codes, b.codes), (a.sf, b.sf), (a.outer, b.outer), (a8.codes, b8.codes), (a8.sf, b8.sf)):
            assert torch.equal(u, v)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_gemm_over_an_empty_contraction_writes_zeros(tj, out_dtype):
    a = tj.quantize_nvfp4(_x(200, 0))
    b = tj.quantize_nvfp4(_x(136, 0))
    d = torch.full((200, 136), 7.0, dtype=out_dtype, device="cuda")
    tj.gemm_nvfp4(a, b, out=d)
    a8, b8 = tj.quantize_mxfp8(_x(200, 0)), tj.quantize_mxfp8(_x(136, 0))
    d8 = torch.full((200, 136), 7.0, dtype=out_dtype, device="cuda")
    tj.gemm_mxfp8(a8, b8, out=d8)
    # scattered columns: the mapped columns become zero, the others are left alone
    cmap = torch.arange(0, 272, 2, dtype=torch.int32, device="cuda")
    ds = torch.full((200, 272), 7.0, dtype=out_dtype, device="cuda")
    tj.gemm_nvfp4(a, b, out=ds, col_map=cmap)
    torch.cuda.synchronize()
    assert torch.count_nonzero(d) == 0 and torch.count_nonzero(d8) == 0
    assert torch.count_nonzero(ds[:, ::2]) == 0 and bool((ds[:, 1::2] == 7.0).all())


def test_gemm_with_no_output_rows_or_columns(tj):
    a, b = tj.quantize_nvfp4(_x(0, 256)), tj.quantize_nvfp4(_x(136, 256))
    assert tj.gemm_nvfp4(a, b).shape == (0, 136)
    assert tj.gemm_nvfp4(b, a).shape == (136, 0)
    torch.cuda.synchronize()


def test_gemm_pairs_over_an_empty_contraction(tj):
    M, N, k = 200, 136, 40
    a, b = tj.quantize_nvfp4(_x(M, 0)), tj.quantize_nvfp4(_x(N, 0))
    a8, b8 = tj.quantize_mxfp8(_x(M, 0)), tj.quantize_mxfp8(_x(k, 0))
    nm = torch.arange(N, dtype=torch.int32, device="cuda")
    om = torch.arange(N, N + k, dtype=torch.int32, device="cuda")
    d = torch.full((M, N + k), 5.0, device="cuda")
    tj.gemm_pair(a, b, a8, b8, out=d, out8=d, col_map=nm, col_map8=om)
    f = torch.full((M, N + k), 5.0, device="cuda")
    tj.gemm_pair_f32(a, b, a8, b8, f, nm, om)
    torch.cuda.synchronize()
    assert torch.count_nonzero(d) == 0 and torch.count_nonzero(f) == 0


def _linear_operands(tj, M, N, K, outl):
    x = _x(M, K, seed=1)
    w = (_x(N, K, seed=2).float() * 0.05).to(torch.bfloat16)
    dy = (_x(M, N, seed=3).float() * 1e-3).to(torch.bfloat16)
    normal = OL.normal_channels(K, outl)
    ni = torch.from_numpy(normal.astype(np.int32)).cuda()
    oi = torch.from_numpy(np.asarray(outl, np.int32)).cuda()
    wq, w8 = tj.quantize_nvfp4(w, sel=ni), tj.quantize_mxfp8(w, sel=oi)
    return x, w, dy, ni, oi, wq, w8


def test_linear_with_no_tokens(tj):
    """M = 0: Y, X-hat and dX are empty; dW, a sum over no tokens, is zero."""
    N, K, outl = 136, 256, np.array([3, 40, 41, 200])
    x, w, dy, ni, oi, wq, w8 = _linear_operands(tj, 0, N, K, outl)
    y, xq, x8 = tj.linear_fwd(x, wq, w8, ni, oi)
    assert y.shape == (0, N) and (xq.rows, xq.cols, x8.rows, x8.cols) == (0, K - 4, 0, 4)
    dx = tj.linear_bwd_dx(dy, wq, w8, ni, oi, seed=3)
    dw = tj.linear_bwd_dw(dy, xq, x8, ni, oi, seed=3, out=torch.full((N, K), 9.0, device="cuda"))
    torch.cuda.synchronize()
    assert dx.shape == (0, K) and torch.count_nonzero(dw) == 0
    tj.device_status()


def test_linear_with_no_output_features(tj):
    """N = 0: Y and dW are empty; X-hat is still saved (bit-exact); dX, a sum over no
    output features, is zero."""
    M, K, outl = 200, 256, np.array([3, 40, 41, 200])
    x, w, dy, ni, oi, wq, w8 = _linear_operands(tj, M, 0, K, outl)
    y, xq, x8 = tj.linear_fwd(x, wq, w8, ni, oi)
    dx = tj.linear_bwd_dx(dy, wq, w8, ni, oi, seed=3, out_dtype=torch.float32,
                          out=torch.full((M, K), 9.0, device="cuda"))
    dw = tj.linear_bwd_dw(dy, xq, x8, ni, oi, seed=3)
    torch.cuda.synchronize()
    assert y.shape == (M, 0) and dw.shape == (0, K) and torch.count_nonzero(dx) == 0
    _, fx, _ = OL.forward(x.float().cpu().numpy(), w.float().cpu().numpy(), outl)
    assert_nvfp4_equal(xq, fx["q"], "X-hat with N = 0")
    assert_mxfp8_equal(x8, fx["q8"], "X-hat slice with N = 0")


def test_fp8_baseline_with_no_tokens(tj):
    N, K = 136, 256
    w8 = tj.quantize_mxfp8(_x(N, K, seed=2))
    x = _x(0, K)
    y, x8, xt8 = tj.fp8_linear_fwd(x, w8)
    wt8 = tj.quantize_mxfp8(_x(N, K, seed=2), along_cols=True)
    dy = _x(0, N)
    dx = tj.fp8_linear_bwd_dx(dy, wt8)
    dw = tj.fp8_linear_bwd_dw(dy, xt8, out=torch.full((N, K), 9.0, device="cuda"))
    torch.cuda.synchronize()
    assert y.shape == (0, N) and dx.shape == (0, K) and torch.count_nonzero(dw) == 0


def test_osci_and_calibration_with_nothing_to_do(tj):
    w = torch.empty(0, 256, device="cuda")
    q = [tj.NVFP4.empty(0, 256), tj.NVFP4.empty(0, 256)]
    mask = torch.empty(0, dtype=torch.int32, device="cuda")
    tj.osci_reset(w, w.clone(), w.clone(), w.clone(), q[0], q[1], mask, 1e-5, 1e-4, 4.0)
    sumsq = torch.zeros(256, dtype=torch.float64, device="cuda")
    tj.outlier_calibrate(_x(0, 256), sumsq)
    torch.cuda.synchronize()
    assert torch.count_nonzero(sumsq) == 0
    tj.device_status()
