"""GPU parity: the FP8 linear baseline (technical summary §4's comparison with FP8
training) through its C-ABI calls tj_fp8_linear_fwd / _bwd_dx / _bwd_dw.

Every operand is MXFP8 along the contraction axis of its GEMM: the saved X along K
and X^T along M must equal the oracle's quantization bit for bit; Y, dX and dW must
lie within 2e-3 * sum|a||b| of the oracle's fp64 product of the same quantized
operands (plus half a bf16 ulp for bf16 outputs).  Cases span several tiles, ragged
sizes and a long token axis whose weight gradient is split in two.
"""
import numpy as np
import pytest
import torch

from layouts import abs_product_fp8, assert_gemm_close, mxfp8_to_logical
from nvfp4_bit_fully_gb300 import workloads
from oracle import linear as OL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tj():
    from nvfp4_bit_fully_gb300 import tj as _tj

    _tj.load()
    return _tj


@pytest.mark.parametrize("M,N,K,out_dtype", [(256, 512, 512, torch.float32), (200, 328, 300, torch.bfloat16),
                                             (4096, 256, 384, torch.float32)])
def test_fp8_baseline_matches_oracle(tj, M, N, K, out_dtype):
    X = workloads.with_heavy_columns((M, K), 1.0, 30.0, 5, M + K, 1)
    W = workloads.normal((N, K), 0.02, M + K, 2)
    dY = workloads.student_t_rows(M, N, 1e-3, 3, M + K, 3)
    Xd, Wd, dYd = X.cuda(), W.cuda(), dY.cuda()
    w8 = tj.quantize_mxfp8(Wd)
    wt8 = tj.quantize_mxfp8(Wd, along_cols=True)
    y, x8, xt8 = tj.fp8_linear_fwd(Xd, w8, out_dtype=out_dtype)
    dx = tj.fp8_linear_bwd_dx(dYd, wt8, out_dtype=out_dtype)
    dw = tj.fp8_linear_bwd_dw(dYd, xt8)
    torch.cuda.synchronize()
    tj.device_status()
    Xf, Wf, dYf = (t.float().numpy() for t in (X, W, dY))
    Y_ref, q8x, q8w = OL.fp8_forward(Xf, Wf)
    dX_ref, q8dy, q8wt = OL.fp8_bwd_dx(dYf, Wf)
    dW_ref, q8dyt, q8xt = OL.fp8_bwd_dw(dYf, Xf)
    for got, ref, what in ((mxfp8_to_logical(x8), q8x, "X along K"), (mxfp8_to_logical(xt8), q8xt, "X^T along M"),
                           (mxfp8_to_logical(wt8), q8wt, "W^T along N")):
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1]), what
    bf = out_dtype == torch.bfloat16
    assert_gemm_close(y.float().cpu().numpy(), Y_ref, abs_product_fp8(q8x, q8w), bf16=bf, what="Y")
    assert_gemm_close(dx.float().cpu().numpy(), dX_ref, abs_product_fp8(q8dy, q8wt), bf16=bf, what="dX")
    assert_gemm_close(dw.cpu().numpy(), dW_ref, abs_product_fp8(q8dyt, q8xt), what="dW")


def test_fp8_baseline_argument_errors(tj):
    x = torch.randn(128, 256, device="cuda").to(torch.bfloat16)
    w8 = tj.quantize_mxfp8(torch.randn(64, 128, device="cuda").to(torch.bfloat16))     # K mismatch
    with pytest.raises(tj.TjError):
        tj.fp8_linear_fwd(x, w8)
    wt8 = tj.quantize_mxfp8(torch.randn(64, 256, device="cuda").to(torch.bfloat16), along_cols=True)
    with pytest.raises(tj.TjError):                                                   # workspace too small
        tj.fp8_linear_bwd_dx(x, wt8, workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
