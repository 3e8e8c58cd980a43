"""Number formats: E2M1 elements, E4M3 inner scales, UE8M0 FP8-slice scales.

Test infrastructure only (see the package docstring).

TetraJet-v2 technical summary §2.A: NVFP4 stores 4-bit values in groups of 16
with an 8-bit scale.  The 4-bit value format is E2M1 (sign, 2 exponent bits,
1 mantissa bit); its magnitudes are the grid below, which is the format's own
definition (the lay explainer's "only 0 or 0.5" example is its first step).
The 8-bit group scale is E4M3 (bias 7, no infinities, max 448, the all-ones
mantissa at exponent 15 is NaN).  The FP8 outlier slice of §2.C uses E4M3
values with a power-of-two UE8M0 scale per 32 elements (reading: the pages
only say "e.g. FP8").
"""
import numpy as np

# E2M1 magnitudes, indexed by the 3 low bits of a code; bit 3 is the sign.
E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float32)
E2M1_MAX = np.float32(6.0)
E4M3_MAX = np.float32(448.0)


def e4m3_decode(byte):
    """Value of an E4M3 byte (array of uint8) as float64; NaN for 0x7F/0xFF."""
    b = np.asarray(byte, dtype=np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 0x7
    sub = m.astype(np.float64) * 2.0 ** -9           # e == 0: m/8 * 2^(1-7)
    nor = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    val = np.where(e == 0, sub, nor)
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


# All non-negative finite E4M3 values with their byte, in increasing order.
_E4M3_POS_BYTES = np.arange(0, 0x7F, dtype=np.uint8)          # 0x00 .. 0x7E
_E4M3_POS_VALS = e4m3_decode(_E4M3_POS_BYTES)                  # strictly increasing


# The inner scales a group may take: the normal E4M3 values 2^-6 .. 448 (bytes 0x08 .. 0x7E).
_INNER_BYTES = np.arange(0x08, 0x7F, dtype=np.uint8)
_INNER_VALS = e4m3_decode(_INNER_BYTES).astype(np.float32)


def e4m3_inner_scale_byte(a_i, s_o):
    """Inner-scale byte of 16-element groups with amax a_i inside outer blocks of scale s_o.

    Reading (inner-scale rounding, technical summary §2.A): the scale is the
    smallest normal E4M3 value sigma whose largest representable magnitude, the
    E2M1 maximum 6 dequantized the way every consumer dequantizes it,
    fl(fl(6 * sigma) * s_o) in fp32, is at least a_i; 448 if none is.  So:
      * no element of the group exceeds the E2M1 range: stochastic rounding
        never clips and stays unbiased (§2.A's E[round(x)] = x);
      * the rule is decided on the dequantized values themselves, so a weight
        moved onto its own dequantized value (OsciReset's reset to the bin
        centre, §2.B) quantizes to the same scale and code again;
      * it starts at the smallest normal E4M3 value 2^-6: with the coarser
        subnormal steps a group maximum can round down onto the previous
        scale's top value, and a reset would then change the group's scale.
    a_i == 0 gives byte 0.  Brute force over all 119 candidate scales.
    """
    a_i = np.asarray(a_i, dtype=np.float32)
    s_o = np.broadcast_to(np.asarray(s_o, dtype=np.float32), a_i.shape)
    flat_a, flat_s = a_i.reshape(-1), s_o.reshape(-1)
    out = np.empty(flat_a.shape, dtype=np.uint8)
    six_sigma = (np.float32(6.0) * _INNER_VALS).astype(np.float32)          # exact
    step = 1 << 16
    for i in range(0, flat_a.size, step):
        a = flat_a[i:i + step]
        with np.errstate(over="ignore"):
            top = (six_sigma[None, :] * flat_s[i:i + step, None]).astype(np.float32)
        ok = top >= a[:, None]
        first = np.where(ok.any(axis=1), ok.argmax(axis=1), len(_INNER_BYTES) - 1)
        out[i:i + step] = np.where(a > 0, _INNER_BYTES[first], 0)
    return out.reshape(a_i.shape)


def e4m3_rne_satfinite_byte(x):
    """Nearest finite E4M3 value to fp32 x, ties to even mantissa, |x|>448 -> 448.

    Used for the FP8 outlier slice (§2.C).  Returns the byte (sign in bit 7).
    Zero and values that round to zero give +0 / -0 by the sign of x.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    vals = _E4M3_POS_VALS
    hi = np.searchsorted(vals, a, side="left")                   # vals[hi] >= a
    hi = np.minimum(hi, len(vals) - 1)
    lo = np.maximum(hi - 1, 0)
    v_hi = vals[hi]
    v_lo = vals[lo]
    exact = v_hi == a
    d_lo = a - v_lo
    d_hi = v_hi - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((_E4M3_POS_BYTES[hi] & 1) == 0))
    byte = np.where(exact | pick_hi, _E4M3_POS_BYTES[hi], _E4M3_POS_BYTES[lo])
    byte = np.where(a >= 448.0, np.uint8(0x7E), byte)               # satfinite
    sign = np.where(np.signbit(x), 0x80, 0x00).astype(np.uint8)
    return (byte.astype(np.uint8) | sign).astype(np.uint8)


def ue8m0_decode(byte):
    """UE8M0 scale byte -> 2^(byte-127) as float64."""
    return np.exp2(np.asarray(byte, dtype=np.float64) - 127.0)


def e2m1_decode(code):
    """Signed E2M1 value of a code (low 4 bits), as float64."""
    c = np.asarray(code, dtype=np.int64)
    mag = E2M1_GRID[c & 7].astype(np.float64)
    return np.where(c & 8, -mag, mag)


# ---------------------------------------------------------------------------
# Element formats of an MX outlier slice.  The FP8 slice uses E4M3.  The mixed FP6 x FP4
# variant of the slice (technical summary §5: the authors name FP6 x FP4 mixed precision
# as a future direction, without a recipe) uses the FP6 formats E2M3 / E3M2 and the FP4
# format E2M1.  Their definitions are those of the OCP Microscaling (MX) specification
# v1.0, §5.3: no infinities or NaN, subnormals at the zero exponent,
#   E2M3: bias 1, values m/8 (e = 0) and (1 + m/8) 2^(e-1), max 7.5;
#   E3M2: bias 3, values m/4 2^-2 (e = 0) and (1 + m/4) 2^(e-3), max 28;
#   E2M1: the grid above, max 6.
# A code holds the sign in its top bit (bit 5 of a 6-bit code, bit 3 of a 4-bit code, bit 7
# of an E4M3 byte).  The format numbers are the ones the tensor core uses.
# ---------------------------------------------------------------------------
MX_E4M3, MX_E2M3, MX_E3M2, MX_E2M1 = 0, 3, 4, 5
MX_FORMATS = (MX_E4M3, MX_E2M3, MX_E3M2, MX_E2M1)
MX_BITS = {MX_E4M3: 8, MX_E2M3: 6, MX_E3M2: 6, MX_E2M1: 4}
MX_MAX = {MX_E4M3: 448.0, MX_E2M3: 7.5, MX_E3M2: 28.0, MX_E2M1: 6.0}


def e2m3_decode(code):
    """Signed E2M3 value of a 6-bit code, as float64."""
    c = np.asarray(code, dtype=np.int64)
    e = (c >> 3) & 3
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 1.0))
    return np.where(c & 0x20, -mag, mag)


def e3m2_decode(code):
    """Signed E3M2 value of a 6-bit code, as float64."""
    c = np.asarray(code, dtype=np.int64)
    e = (c >> 2) & 7
    m = (c & 3).astype(np.float64)
    mag = np.where(e == 0, m / 4.0 * 0.25, (1.0 + m / 4.0) * np.exp2(e.astype(np.float64) - 3.0))
    return np.where(c & 0x20, -mag, mag)


def mx_elem_decode(code, fmt):
    """Value (float64) of an MX element code of format fmt."""
    if fmt == MX_E4M3:
        return e4m3_decode(np.asarray(code, dtype=np.uint8))
    if fmt == MX_E2M3:
        return e2m3_decode(code)
    if fmt == MX_E3M2:
        return e3m2_decode(code)
    if fmt == MX_E2M1:
        return e2m1_decode(code)
    raise ValueError("unknown MX element format %r" % (fmt,))


def _mx_positive_codes(fmt):
    """The non-negative finite codes of fmt in increasing order of value, and the values."""
    n = {MX_E4M3: 0x7F, MX_E2M3: 32, MX_E3M2: 32, MX_E2M1: 8}[fmt]
    codes = np.arange(n, dtype=np.int64)
    return codes, mx_elem_decode(codes, fmt)


def mx_rne_code(x, fmt):
    """Code of the value of fmt nearest to x, ties to the even code, |x| beyond the maximum
    -> the maximum (saturating).  Sign from the sign bit of x (so -0 and negative values
    that round to zero give the negative zero code), as for the FP8 slice.

    Brute force: the positive codes of every format here are ordered by value, and between
    two neighbours the one with an even code has the even mantissa.
    """
    x = np.asarray(x, dtype=np.float64)
    codes, vals = _mx_positive_codes(fmt)
    a = np.abs(x)
    hi = np.minimum(np.searchsorted(vals, a, side="left"), len(vals) - 1)     # vals[hi] >= a
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - vals[lo], vals[hi] - a
    pick_hi = (vals[hi] == a) | (d_hi < d_lo) | ((d_hi == d_lo) & ((codes[hi] & 1) == 0))
    mag = np.where(pick_hi, codes[hi], codes[lo])
    mag = np.where(a >= MX_MAX[fmt], codes[-1], mag)
    sign = {MX_E4M3: 0x80, MX_E2M3: 0x20, MX_E3M2: 0x20, MX_E2M1: 0x8}[fmt]
    return (mag | np.where(np.signbit(x), sign, 0)).astype(np.uint8)
