"""Double-block NVFP4 quantization (RTN / SR) and the MXFP8 outlier slice.

Test infrastructure only (see the package docstring).

TetraJet-v2 technical summary §2.A: an outer block of 128 elements carries a
global (FP32) scale, and inner blocks of 16 elements inside it carry a local
8-bit scale; no whole-tensor amax is needed.  Forward operands are rounded to
nearest; backward operands use stochastic rounding so that E[round(x)] = x.
Weight groups are 1x16, i.e. both block levels lie along one row, along the
contraction dimension of the GEMM that consumes the operand.

Readings taken where the pages are silent:
  * outer scale s_o = amax_128 / (6 * 448) in fp32 (so the largest inner block
    gets the largest inner scale); 2^-149 if that underflows to 0;
  * inner scale s_i = the smallest normal E4M3 value whose dequantized top
    value fl(fl(6 * s_i) * s_o) covers amax_16, 448 if none does (rounded up,
    so scaled elements never exceed the E2M1 maximum 6, decided on the
    dequantized values so that re-quantizing a dequantized tensor gives it
    back; see formats.e4m3_inner_scale_byte);
  * element step: r = 1 / (s_i * s_o) in fp32, v = x * r, a = min(|v|, 6);
  * RTN picks the nearest grid magnitude, ties to the even code;
  * SR rounds up from the grid point below a with probability
    (a - lo) / (hi - lo), decided as  float(u16) < p * 65536;
  * a zero element gives code 0; otherwise bit 3 = (x < 0);
  * rows are zero-padded to a multiple of 128 along the quantized axis.

Outputs use a LOGICAL layout: codes uint8 [R, Lp] (one code per element, low
nibble), inner scale bytes uint8 [R, Lp/16], outer scales float32 [R, Lp/128].
"""
import numpy as np

from .formats import E2M1_GRID, e2m1_decode, e4m3_decode, e4m3_inner_scale_byte
from .formats import e4m3_rne_satfinite_byte, ue8m0_decode
from .formats import MX_E4M3, MX_MAX, mx_elem_decode, mx_rne_code
from .philox import sr_uniform16

F32 = np.float32
OUTER = 128
INNER = 16
RTN = 0
SR = 1


def pad_cols(x, multiple):
    """Zero-pad the last axis of a 2-D fp32 array to a multiple of `multiple`."""
    x = np.asarray(x, dtype=F32)
    r, l = x.shape
    lp = ((l + multiple - 1) // multiple) * multiple
    out = np.zeros((r, lp), dtype=F32)
    out[:, :l] = x
    return out


def rtn_index(a):
    """Grid index nearest to a in [0, 6]; ties go to the even index."""
    a = np.asarray(a, dtype=F32)
    # candidates: the grid index just below (lo) and just above (hi)
    hi = np.searchsorted(E2M1_GRID, a, side="left")            # GRID[hi] >= a
    hi = np.minimum(hi, 7)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - E2M1_GRID[lo]
    d_hi = E2M1_GRID[hi] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    return np.where(take_hi, hi, lo).astype(np.uint8)


def sr_index(a, u16):
    """Stochastic rounding of a in [0, 6] between its two neighbouring grid points."""
    a = np.asarray(a, dtype=F32)
    hi = np.searchsorted(E2M1_GRID, a, side="left")
    hi = np.minimum(hi, 7)
    exact = E2M1_GRID[hi] == a
    lo = np.maximum(hi - 1, 0)
    g_lo = E2M1_GRID[lo]
    g_hi = E2M1_GRID[hi]
    gap = np.where(exact, F32(1.0), g_hi - g_lo)                # a power of two
    p = ((a - g_lo) / gap).astype(F32)                          # exact
    up = u16.astype(F32) < (p * F32(65536.0))
    return np.where(exact, hi, np.where(up, hi, lo)).astype(np.uint8)


def quantize_nvfp4(x, mode=RTN, seed=0, tag=0, row_ids=None):
    """Double-block quantize each row of x [R, L] along its length.

    row_ids: the row index of each given row in the full operand (for the SR
    element index e = row * Lp + col); defaults to 0..R-1.
    Returns (codes [R, Lp] uint8, sf [R, Lp/16] uint8, outer [R, Lp/128] f32).
    """
    xp = pad_cols(x, OUTER)
    R, Lp = xp.shape
    nb = Lp // OUTER
    xb = xp.reshape(R, nb, OUTER // INNER, INNER)
    ax = np.abs(xb)

    # outer block: FP32 scale from its amax
    a_o = ax.max(axis=(2, 3))                                   # [R, nb]
    s_o = (a_o / F32(6.0 * 448.0)).astype(F32)
    s_o = np.where((a_o > 0) & (s_o == 0), F32(2.0 ** -149), s_o).astype(F32)

    # inner blocks: E4M3 scale, rounded up on the dequantized side
    a_i = ax.max(axis=3)                                        # [R, nb, 8]
    sf = e4m3_inner_scale_byte(a_i, s_o[:, :, None])
    s_i = e4m3_decode(sf).astype(F32)

    # element step
    s = (s_i * s_o[:, :, None]).astype(F32)                     # [R, nb, 8]
    with np.errstate(divide="ignore", over="ignore"):
        r = np.where(s > 0, F32(1.0) / np.where(s > 0, s, F32(1.0)), F32(0.0)).astype(F32)
    with np.errstate(over="ignore", invalid="ignore"):
        v = (xb * r[:, :, :, None]).astype(F32)
    a = np.minimum(np.abs(v), F32(6.0)).astype(F32)

    if mode == RTN:
        idx = rtn_index(a)
    else:
        rows = np.arange(R, dtype=np.int64) if row_ids is None else np.asarray(row_ids, np.int64)
        e = rows[:, None] * Lp + np.arange(Lp, dtype=np.int64)[None, :]
        u = sr_uniform16(e.astype(np.uint64), seed, tag).reshape(R, nb, OUTER // INNER, INNER)
        idx = sr_index(a, u)

    nonzero = (xb != 0) & (s[:, :, :, None] > 0)
    sign = np.where(xb < 0, 8, 0).astype(np.uint8)
    codes = np.where(nonzero, idx | sign, 0).astype(np.uint8)
    return codes.reshape(R, Lp), sf.reshape(R, nb * 8), s_o


def dequantize_nvfp4_f32(codes, sf, outer):
    """fp32 dequantization (G * s_i) * s_o, the value the backward re-quantizes."""
    R, Lp = codes.shape
    g = e2m1_decode(codes).astype(F32)                          # exact
    s_i = np.repeat(e4m3_decode(sf).astype(F32), INNER, axis=1)
    s_o = np.repeat(np.asarray(outer, F32), OUTER, axis=1)
    return ((g * s_i).astype(F32) * s_o).astype(F32)


def dequantize_nvfp4_f64(codes, sf, outer):
    """Exact dequantized values in fp64 (the GEMM operands of the oracle)."""
    g = e2m1_decode(codes)
    s_i = np.repeat(e4m3_decode(sf), INNER, axis=1)
    s_o = np.repeat(np.asarray(outer, np.float64), OUTER, axis=1)
    return g * s_i * s_o


# ---------------------------------------------------------------------------
# MXFP8 outlier slice (technical summary §2.C, "kept in higher precision,
# e.g. FP8, in the forward and backward passes").
# Reading: E4M3 values with one power-of-two UE8M0 scale 2^E per 1x32 block
# along the contraction dimension; E is the smallest integer with
# 448 * 2^E >= amax_32, clamped to [-127, 127]; elements are x * 2^-E rounded
# to nearest-even and saturated to +-448; an all-zero block gets E = 0.
# ---------------------------------------------------------------------------
MX = 32


def mx_exponent(amax):
    """Smallest integer E with 448 * 2^E >= amax (amax > 0), clamped to [-127, 127]."""
    amax = np.asarray(amax, dtype=np.float64)
    mant, ex = np.frexp(amax)                 # amax = mant * 2^ex, mant in [0.5, 1)
    # 448 = 0.875 * 2^9, so 448 * 2^E >= mant * 2^ex  <=>  2^(9+E-ex) >= mant / 0.875
    E = np.where(mant <= 0.875, ex - 9, ex - 8)
    E = np.where(amax > 0, E, 0)
    return np.clip(E, -127, 127).astype(np.int64)


def quantize_mxfp8(x, pad_to=128):
    """MXFP8 quantize rows of x [R, L] along L (zero-padded to `pad_to`).

    Returns (codes uint8 [R, Lp] E4M3 bytes, scale bytes uint8 [R, Lp/32] UE8M0).
    """
    xp = pad_cols(x, pad_to)
    R, Lp = xp.shape
    xb = xp.reshape(R, Lp // MX, MX)
    amax = np.abs(xb).max(axis=2)
    E = mx_exponent(amax)
    scale_inv = np.exp2(-E.astype(np.float64)).astype(F32)      # exact power of two
    with np.errstate(over="ignore"):
        y = (xb * scale_inv[:, :, None]).astype(F32)
    codes = e4m3_rne_satfinite_byte(y)
    return codes.reshape(R, Lp), (E + 127).astype(np.uint8)


def dequantize_mxfp8_f64(codes, sbytes):
    """Exact fp64 values of an MXFP8 slice."""
    v = e4m3_decode(codes)
    s = np.repeat(ue8m0_decode(sbytes), MX, axis=1)
    return v * s


def dequantize_mxfp8_f32(codes, sbytes):
    """fp32 values of an MXFP8 slice (exact: an E4M3 value times a power of two)."""
    return dequantize_mxfp8_f64(codes, sbytes).astype(F32)


# ---------------------------------------------------------------------------
# The outlier slice in any MX element format (E4M3, or the FP6 / FP4 formats of the mixed
# FP6 x FP4 variant, technical summary §5).  Reading: the FP8 slice's rule with the
# format's own maximum: E = the smallest integer with max_fmt * 2^E >= amax_32, clamped
# to [-127, 127] (0 for an all-zero block); elements x * 2^-E rounded to the nearest
# value of the format, ties to even, saturating.  With E4M3 this is quantize_mxfp8.
# ---------------------------------------------------------------------------
def mx_exponent_fmt(amax, fmt):
    """Smallest integer E with MX_MAX[fmt] * 2^E >= amax (amax > 0), clamped to [-127, 127]."""
    amax = np.asarray(amax, dtype=np.float64)
    mant, ex = np.frexp(amax)                       # amax = mant * 2^ex, mant in [0.5, 1)
    mf, exf = np.frexp(MX_MAX[fmt])                 # the format's maximum, the same way
    # max * 2^E >= amax  <=>  2^(exf + E - ex) >= mant / mf, and 1/2 < mant / mf < 2
    E = np.where(mant <= mf, ex - exf, ex - exf + 1)
    E = np.where(amax > 0, E, 0)
    return np.clip(E, -127, 127).astype(np.int64)


def quantize_mx(x, fmt, pad_to=128):
    """MX quantize rows of x [R, L] along L (zero-padded to `pad_to`) in element format fmt.

    Returns (codes uint8 [R, Lp], one code per element; scale bytes uint8 [R, Lp/32] UE8M0).
    """
    xp = pad_cols(x, pad_to)
    R, Lp = xp.shape
    xb = xp.reshape(R, Lp // MX, MX)
    amax = np.abs(xb).max(axis=2)
    E = mx_exponent_fmt(amax, fmt)
    scale_inv = np.exp2(-E.astype(np.float64))
    y = xb.astype(np.float64) * scale_inv[:, :, None]          # exact: a power of two
    codes = mx_rne_code(y, fmt)
    return codes.reshape(R, Lp), (E + 127).astype(np.uint8)


def dequantize_mx_f64(codes, sbytes, fmt):
    """Exact fp64 values of an MX slice of element format fmt."""
    v = mx_elem_decode(codes, fmt)
    s = np.repeat(ue8m0_decode(sbytes), MX, axis=1)
    return v * s


def dequantize_mx_f32(codes, sbytes, fmt):
    """fp32 values of an MX slice (exact: a short-mantissa value times a power of two).  An
    element of a block scaled near the top of the fp32 range can round up to a grid value
    beyond it (E2M1 6 x 2^126 = 5.1e38); its fp32 value is then infinite, as on the GPU."""
    with np.errstate(over="ignore"):
        return dequantize_mx_f64(codes, sbytes, fmt).astype(F32)
