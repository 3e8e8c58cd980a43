"""Pins of the oracle's MX element formats and the generic MX slice quantizer (the FP6 x FP4
variant of the outlier slice; technical summary §5 names FP6 x FP4 as a future direction).

Independent of the oracle's own arithmetic:
  * the value tables of E2M3 and E3M2 are typed in by hand from the format definitions
    (OCP Microscaling Formats v1.0, §5.3: E2M3 max 7.5, smallest subnormal 1/8; E3M2 max
    28, smallest subnormal 1/16);
  * round-to-nearest-even is checked by brute force with exact fractions over those tables;
  * the block exponent is checked for minimality (max * 2^E >= amax > max * 2^(E-1));
  * quantized elements obey the format's error bound, grid-valued inputs quantize exactly,
    and the slice product then reduces to a plain matmul;
  * in E4M3 the generic quantizer equals the FP8 slice's, pinned elsewhere.
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle import formats as F
from oracle import linear as OL
from oracle import quant as Q

E2M3_POS = [0, 0.125, 0.25, 0.375, 0.5, 0.625, 0.75, 0.875,
            1, 1.125, 1.25, 1.375, 1.5, 1.625, 1.75, 1.875,
            2, 2.25, 2.5, 2.75, 3, 3.25, 3.5, 3.75,
            4, 4.5, 5, 5.5, 6, 6.5, 7, 7.5]
E3M2_POS = [0, 0.0625, 0.125, 0.1875,
            0.25, 0.3125, 0.375, 0.4375,
            0.5, 0.625, 0.75, 0.875,
            1, 1.25, 1.5, 1.75,
            2, 2.5, 3, 3.5,
            4, 5, 6, 7,
            8, 10, 12, 14,
            16, 20, 24, 28]
E2M1_POS = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
TABLES = {F.MX_E2M3: (E2M3_POS, 0x20), F.MX_E3M2: (E3M2_POS, 0x20), F.MX_E2M1: (E2M1_POS, 0x8)}
SUB_FORMATS = (F.MX_E2M3, F.MX_E3M2, F.MX_E2M1)


@pytest.mark.parametrize("fmt", SUB_FORMATS)
def test_decode_matches_the_hand_tables(fmt):
    table, sign = TABLES[fmt]
    codes = np.arange(len(table))
    assert np.array_equal(F.mx_elem_decode(codes, fmt), np.array(table, dtype=np.float64))
    neg = F.mx_elem_decode(codes | sign, fmt)
    assert np.array_equal(neg, -np.array(table, dtype=np.float64))
    assert np.signbit(F.mx_elem_decode(sign, fmt))                  # the negative zero code
    assert F.MX_MAX[fmt] == table[-1]


def _brute_rne(x, table):
    """Nearest table value to x (exact), ties to the even index, saturating; returns index."""
    a = abs(Fraction(x))
    if a >= Fraction(table[-1]):
        return len(table) - 1
    best = None
    for i, v in enumerate(table):
        d = abs(a - Fraction(v))
        if best is None or d < best[0] or (d == best[0] and i % 2 == 0):
            best = (d, i)
    return best[1]


@pytest.mark.parametrize("fmt", SUB_FORMATS)
def test_rne_by_brute_force(fmt):
    table, sign = TABLES[fmt]
    rng = np.random.default_rng(11 + fmt)
    vals = np.array(table, dtype=np.float64)
    mids = (vals[1:] + vals[:-1]) / 2                                # every tie
    xs = np.concatenate([vals, mids, mids + 1e-9, mids - 1e-9,
                         rng.uniform(0, table[-1] * 1.3, 400), rng.uniform(0, table[1] * 3, 100),
                         [table[-1] * 4, 1e30, 1e-30]])
    xs = np.concatenate([xs, -xs])
    got = F.mx_rne_code(xs, fmt)
    for x, c in zip(xs, got):
        want = _brute_rne(x, table) | (sign if np.signbit(x) else 0)
        assert c == want, (fmt, x, c, want)


@pytest.mark.parametrize("fmt", SUB_FORMATS)
def test_negative_zero_and_tiny_negatives_keep_the_sign(fmt):
    _, sign = TABLES[fmt]
    assert list(F.mx_rne_code([-0.0, 0.0, -1e-12], fmt)) == [sign, 0, sign]


@pytest.mark.parametrize("fmt", F.MX_FORMATS)
def test_block_exponent_is_minimal(fmt):
    rng = np.random.default_rng(3 + fmt)
    amax = np.concatenate([np.exp2(rng.uniform(-100, 100, 2000)),
                           F.MX_MAX[fmt] * np.exp2(np.arange(-60, 60, dtype=np.float64)),    # exact fits
                           F.MX_MAX[fmt] * np.exp2(np.arange(-60, 60, dtype=np.float64)) * (1 + 2.0 ** -20)])
    E = Q.mx_exponent_fmt(amax, fmt)
    m = F.MX_MAX[fmt]
    assert np.all(m * np.exp2(E.astype(np.float64)) >= amax)
    assert np.all(m * np.exp2(E.astype(np.float64) - 1) < amax)
    assert Q.mx_exponent_fmt(0.0, fmt) == 0
    assert Q.mx_exponent_fmt(1e-300, fmt) == -127 and Q.mx_exponent_fmt(1e300, fmt) == 127


@pytest.mark.parametrize("fmt", SUB_FORMATS)
def test_quantized_elements_obey_the_format_error_bound(fmt):
    """Normal range: |q - x| <= 2^-(m+1) |x| (m mantissa bits); subnormal range: half the
    subnormal step; both times the block scale 2^E.  No element clips."""
    table, _ = TABLES[fmt]
    mbits = {F.MX_E2M3: 3, F.MX_E3M2: 2, F.MX_E2M1: 1}[fmt]
    rng = np.random.default_rng(21 + fmt)
    x = (rng.standard_normal((64, 256)) * np.exp2(rng.integers(-20, 20, (64, 1)))).astype(np.float32)
    x[::7, 5] *= 50.0                                               # outliers inside blocks
    codes, sb = Q.quantize_mx(x, fmt)
    q = Q.dequantize_mx_f64(codes, sb, fmt)
    s = np.repeat(np.exp2(sb.astype(np.float64) - 127), 32, axis=1)
    bound = np.maximum(np.abs(x) * 2.0 ** -(mbits + 1), s * table[1] / 2)
    assert np.all(np.abs(q - x) <= bound * (1 + 1e-12))
    blk = np.abs(x).reshape(64, -1, 32).max(axis=2)
    assert np.all(blk <= F.MX_MAX[fmt] * np.exp2(sb.astype(np.float64) - 127))


@pytest.mark.parametrize("fmt", F.MX_FORMATS)
def test_grid_inputs_quantize_exactly_and_the_product_is_a_matmul(fmt):
    """Grid values times a power of two per 32-block, with the format maximum in each block,
    quantize exactly; the slice product of two such operands is then A B^T."""
    rng = np.random.default_rng(31 + fmt)

    def grid_operand(rows, cols, f):
        codes = np.arange(0x7F if f == F.MX_E4M3 else len(TABLES[f][0]))
        vals = F.mx_elem_decode(codes, f)
        v = rng.choice(vals, size=(rows, cols)) * rng.choice([-1.0, 1.0], size=(rows, cols))
        v[:, ::32] = F.MX_MAX[f]
        e = rng.integers(-30, 30, (rows, cols // 32))
        return (v * np.exp2(np.repeat(e, 32, axis=1))).astype(np.float32)

    partner = OL.SLICE_PARTNER[fmt]
    a = grid_operand(48, 128, fmt)
    b = grid_operand(40, 128, partner)
    qa, qb = Q.quantize_mx(a, fmt), Q.quantize_mx(b, partner)
    assert np.array_equal(Q.dequantize_mx_f64(*qa, fmt), a.astype(np.float64))
    assert np.array_equal(Q.dequantize_mx_f64(*qb, partner), b.astype(np.float64))
    assert np.array_equal(OL.gemm_mx(qa, fmt, qb, partner), a.astype(np.float64) @ b.astype(np.float64).T)


def test_e4m3_generic_equals_the_fp8_slice():
    rng = np.random.default_rng(41)
    x = (rng.standard_normal((33, 300)) * np.exp2(rng.integers(-30, 30, (33, 1)))).astype(np.float32)
    x[0, :40] = 0.0
    x[1, 3] = -0.0
    c8, s8 = Q.quantize_mxfp8(x)
    c, s = Q.quantize_mx(x, F.MX_E4M3)
    assert np.array_equal(c8, c) and np.array_equal(s8, s)


def test_slice_partner_pairs_fp6_with_fp4():
    for f in SUB_FORMATS:
        pair = {F.MX_BITS[f], F.MX_BITS[OL.SLICE_PARTNER[f]]}
        assert pair == {6, 4}
    assert OL.SLICE_PARTNER[F.MX_E4M3] == F.MX_E4M3


def test_fp6_fp4_linear_slice_formats_flow_through_the_backward():
    """Forward X in E2M3 and W in E2M1: the dX slice is dY(E2M3) x W-hat^T(E2M1) and the dW
    slice dY^T(E2M1) x X-hat^T(E2M3); with the FP8 slice the results are those of the
    FP8 composition."""
    rng = np.random.default_rng(51)
    M, N, K = 64, 96, 256
    X = rng.standard_normal((M, K)).astype(np.float32)
    W = (rng.standard_normal((N, K)) * 0.1).astype(np.float32)
    dY = rng.standard_normal((M, N)).astype(np.float32)
    o = np.array([3, 40, 41, 100, 200], dtype=np.int64)
    Y, fx, fw = OL.forward(X, W, o, fmt_x=F.MX_E2M3, fmt_w=F.MX_E2M1)
    assert fx["fmt8"] == F.MX_E2M3 and fw["fmt8"] == F.MX_E2M1
    assert fx["q8"][0].max() < 64 and fw["q8"][0].max() < 16
    _, _, q8_dy, q8_w = OL.bwd_dx_operands(dY, fw, seed=5)
    assert np.array_equal(q8_dy[0], Q.quantize_mx(dY, F.MX_E2M3)[0])
    assert q8_w[0].max() < 16
    _, _, q8_dyt, q8_x = OL.bwd_dw_operands(dY, fx, seed=5)
    assert q8_dyt[0].max() < 16 and q8_x[0].max() < 64
    # the slice columns of dX / dW are the products of those operands
    dX = OL.bwd_dx(dY, fw, o, seed=5)
    assert np.array_equal(dX[:, o], OL.gemm_mx(q8_dy, F.MX_E2M3, q8_w, F.MX_E2M1)[:, : len(o)])
    dW = OL.bwd_dw(dY, fx, o, seed=5)
    assert np.array_equal(dW[:, o], OL.gemm_mx(q8_dyt, F.MX_E2M1, q8_x, F.MX_E2M3)[:, : len(o)])
    # the FP8 default is unchanged
    Y8, fx8, fw8 = OL.forward(X, W, o)
    assert np.array_equal(Y8, OL.gemm_fp4(fx8["q"], fw8["q"]) + OL.gemm_fp8(fx8["q8"], fw8["q8"]))
