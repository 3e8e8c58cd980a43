"""NVFP4 linear layer: forward Y = X W^T, backward dX = dY W, dW = dY^T X.

Test infrastructure only (see the package docstring).

TetraJet-v2 technical summary §2 (all linear layers take NVFP4 activations,
weights and gradients), §2.A (backward "aligned": it estimates with X-hat, the
dequantized forward operand, not X; SR in the backward; 1x16 weight groups, so
the transposed weight is re-grouped along the new contraction axis) and §2.C
(RHT on the backward contractions; a static top-p% set of outlier channels kept
in FP8 in forward and backward).

Notation: X [M, K], W [N, K], dY [M, N].  O = outlier channels (sorted), k = |O|;
NC = the other channels, ascending, K_N = K - k.  Readings:
  * channels are the input features K; normal channels are compacted in
    ascending order before blocking;
  * both operands of an outlier-slice product are MXFP8 (RTN, no RHT);
  * the mixed FP6 x FP4 variant of the slice (technical summary §5 names FP6 x FP4 as
    a future direction, no recipe): the slice operands take other MX element formats.
    The forward operands choose theirs (e.g. X in E2M3, W in E2M1); in the backward the
    re-aligned operand keeps its forward format and dY's slice takes the partner format
    (SLICE_PARTNER), so that every slice product is FP6 x FP4 (or FP8 x FP8);
  * the backward re-quantizes the fp32 dequantized forward operands;
  * SR tags: 1 = dY rows (dX), 2 = dY^T rows (dW), 3 = W-hat^T, 4 = X-hat^T;
    RHT sign tags 0x100 (dX) and 0x101 (dW); alpha = 2^-7 undoes H^T H = 128 I.
All products are accumulated in fp64 on exactly dequantized operands.
"""
import numpy as np

from . import quant as Q
from .formats import MX_E2M1, MX_E2M3, MX_E3M2, MX_E4M3
from .philox import rht_signs
from .rht import rht_f32

F32 = np.float32
TAG_DY_ROW, TAG_DY_COL, TAG_WT, TAG_XT = 1, 2, 3, 4
TAG_RHT_DX, TAG_RHT_DW = 0x100, 0x101
ALPHA_RHT = 2.0 ** -7
# format of dY's slice in a backward product whose other slice operand has format f
SLICE_PARTNER = {MX_E4M3: MX_E4M3, MX_E2M1: MX_E2M3, MX_E2M3: MX_E2M1, MX_E3M2: MX_E2M1}


def normal_channels(K, outlier_idx):
    """Ascending complement of the outlier set in 0..K-1."""
    mask = np.ones(K, dtype=bool)
    mask[np.asarray(outlier_idx, dtype=np.int64)] = False
    return np.nonzero(mask)[0].astype(np.int64)


def quantize_forward_operand(A, outlier_idx, fmt8=MX_E4M3):
    """Forward quantization of an operand [rows, K] along K (X or W).

    Returns dict(q=(codes, sf, outer) of the normal channels, RTN double-block,
                 q8=(codes, scales) MX slice of the outlier channels in element format
                 fmt8 (E4M3 = the FP8 slice) or None, fmt8).
    """
    A = np.asarray(A, dtype=F32)
    K = A.shape[1]
    o = np.asarray(outlier_idx, dtype=np.int64)
    nc = normal_channels(K, o)
    q = Q.quantize_nvfp4(A[:, nc], Q.RTN)
    q8 = Q.quantize_mx(A[:, o], fmt8) if len(o) else None
    return {"q": q, "q8": q8, "fmt8": fmt8, "K_N": len(nc), "k": len(o)}


def gemm_fp4(qa, qb, alpha=1.0):
    """alpha * deq(A) deq(B)^T in fp64 for two double-block operands (same Lp)."""
    a = Q.dequantize_nvfp4_f64(*qa)
    b = Q.dequantize_nvfp4_f64(*qb)
    return alpha * (a @ b.T)


def gemm_fp8(qa, qb):
    """deq(A) deq(B)^T in fp64 for two MXFP8 operands."""
    return Q.dequantize_mxfp8_f64(*qa) @ Q.dequantize_mxfp8_f64(*qb).T


def gemm_mx(qa, fmt_a, qb, fmt_b):
    """deq(A) deq(B)^T in fp64 for two MX slice operands of element formats fmt_a, fmt_b."""
    return Q.dequantize_mx_f64(*qa, fmt_a) @ Q.dequantize_mx_f64(*qb, fmt_b).T


def _fmt8(fq):
    return fq.get("fmt8", MX_E4M3)


def forward(X, W, outlier_idx, fmt_x=MX_E4M3, fmt_w=MX_E4M3):
    """Y = X-hat W-hat^T (fp64), plus the saved quantized forward operands.  fmt_x / fmt_w:
    the element formats of the two outlier slices (E4M3: the FP8 slice)."""
    fx = quantize_forward_operand(X, outlier_idx, fmt_x)
    fw = quantize_forward_operand(W, outlier_idx, fmt_w)
    Y = gemm_fp4(fx["q"], fw["q"])
    if fx["q8"] is not None:
        Y = Y + gemm_mx(fx["q8"], fmt_x, fw["q8"], fmt_w)
    return Y, fx, fw


def sr_rht_rows(A, seed, sr_tag, rht_tag, row_ids=None):
    """SR double-block quantization of RHT(rows of A) along the row (zero-padded to 128)."""
    Ap = Q.pad_cols(A, Q.OUTER)
    d = rht_signs(seed, rht_tag)
    return Q.quantize_nvfp4(rht_f32(Ap, d), Q.SR, seed=seed, tag=sr_tag, row_ids=row_ids)


def deq_normal_f32(fq):
    """fp32 X-hat / W-hat of the normal channels, [rows, K_N] (padding dropped)."""
    return Q.dequantize_nvfp4_f32(*fq["q"])[:, : fq["K_N"]]


def deq_outlier_f32(fq):
    """fp32 dequantized outlier slice, [rows, k]."""
    return Q.dequantize_mx_f32(*fq["q8"], _fmt8(fq))[:, : fq["k"]]


def bwd_dx_operands(dY, fw, seed):
    """Quantized operands of dX: (S_dY, S_W, Q8(dY), Q8(W-hat_O^T)); the slices in
    SLICE_PARTNER[f] and f, f the format of W's forward slice."""
    s_dy = sr_rht_rows(dY, seed, TAG_DY_ROW, TAG_RHT_DX)
    s_w = sr_rht_rows(deq_normal_f32(fw).T, seed, TAG_WT, TAG_RHT_DX)
    if fw["k"]:
        f = _fmt8(fw)
        q8_dy = Q.quantize_mx(dY, SLICE_PARTNER[f])
        q8_w = Q.quantize_mx(deq_outlier_f32(fw).T, f)
    else:
        q8_dy = q8_w = None
    return s_dy, s_w, q8_dy, q8_w


def bwd_dx(dY, fw, outlier_idx, seed):
    """dX [M, K] = 2^-7 S_dY S_W^T on the normal channels, FP8 slice on the outliers."""
    dY = np.asarray(dY, dtype=F32)
    M = dY.shape[0]
    o = np.asarray(outlier_idx, dtype=np.int64)
    K = fw["K_N"] + fw["k"]
    nc = normal_channels(K, o)
    s_dy, s_w, q8_dy, q8_w = bwd_dx_operands(dY, fw, seed)
    dX = np.zeros((M, K), dtype=np.float64)
    dX[:, nc] = gemm_fp4(s_dy, s_w, ALPHA_RHT)[:, : len(nc)]
    if len(o):
        f = _fmt8(fw)
        dX[:, o] = gemm_mx(q8_dy, SLICE_PARTNER[f], q8_w, f)[:, : len(o)]
    return dX


def bwd_dw_operands(dY, fx, seed):
    """Quantized operands of dW: (S_dY^T, S_X, Q8(dY^T), Q8(X-hat_O^T)); the slices in
    SLICE_PARTNER[f] and f, f the format of X's forward slice."""
    dYt = np.ascontiguousarray(np.asarray(dY, dtype=F32).T)
    s_dy = sr_rht_rows(dYt, seed, TAG_DY_COL, TAG_RHT_DW)
    s_x = sr_rht_rows(deq_normal_f32(fx).T, seed, TAG_XT, TAG_RHT_DW)
    if fx["k"]:
        f = _fmt8(fx)
        q8_dy = Q.quantize_mx(dYt, SLICE_PARTNER[f])
        q8_x = Q.quantize_mx(deq_outlier_f32(fx).T, f)
    else:
        q8_dy = q8_x = None
    return s_dy, s_x, q8_dy, q8_x


def bwd_dw(dY, fx, outlier_idx, seed):
    """dW [N, K] = 2^-7 S_dY^T S_X^T on the normal channels, FP8 slice on the outliers."""
    dY = np.asarray(dY, dtype=F32)
    N = dY.shape[1]
    o = np.asarray(outlier_idx, dtype=np.int64)
    K = fx["K_N"] + fx["k"]
    nc = normal_channels(K, o)
    s_dy, s_x, q8_dy, q8_x = bwd_dw_operands(dY, fx, seed)
    dW = np.zeros((N, K), dtype=np.float64)
    dW[:, nc] = gemm_fp4(s_dy, s_x, ALPHA_RHT)[:, : len(nc)]
    if len(o):
        f = _fmt8(fx)
        dW[:, o] = gemm_mx(q8_dy, SLICE_PARTNER[f], q8_x, f)[:, : len(o)]
    return dW


# ---------------------------------------------------------------------------
# The FP8 linear baseline the pages compare against (technical summary §4: training
# speed vs FP8 with TransformerEngine).  Reading: every GEMM operand in MXFP8 (E4M3
# with a UE8M0 scale per 1x32 along the GEMM's contraction axis, round to nearest),
# quantized from its unquantized source; no RHT, SR, outlier split or double-block
# scale.  fp64 products of the exactly dequantized operands.
# ---------------------------------------------------------------------------
def fp8_forward(X, W):
    """Y [M, N] = Q8(X) Q8(W)^T, both along K.  Returns (Y, Q8(X), Q8(W))."""
    q8x = Q.quantize_mxfp8(np.asarray(X, dtype=F32))
    q8w = Q.quantize_mxfp8(np.asarray(W, dtype=F32))
    return gemm_fp8(q8x, q8w), q8x, q8w


def fp8_bwd_dx(dY, W):
    """dX [M, K] = Q8(dY) Q8(W^T)^T, both along N."""
    q8dy = Q.quantize_mxfp8(np.asarray(dY, dtype=F32))
    q8wt = Q.quantize_mxfp8(np.ascontiguousarray(np.asarray(W, dtype=F32).T))
    return gemm_fp8(q8dy, q8wt), q8dy, q8wt


def fp8_bwd_dw(dY, X):
    """dW [N, K] = Q8(dY^T) Q8(X^T)^T, both along M."""
    q8dyt = Q.quantize_mxfp8(np.ascontiguousarray(np.asarray(dY, dtype=F32).T))
    q8xt = Q.quantize_mxfp8(np.ascontiguousarray(np.asarray(X, dtype=F32).T))
    return gemm_fp8(q8dyt, q8xt), q8dyt, q8xt
