"""Pins for the oracle's double-block NVFP4 quantizer and MXFP8 slice.

Each test checks a property fixed by the pages or by mathematics, chosen so a
plausible slip (wrong tie rule, dropped scale level, transposed block, biased
SR, wrong padding) fails at least one of them:
  * RTN picks the nearest E2M1 grid point (argmin brute force), ties even;
  * SR is exactly unbiased up to its 16-bit resolution (enumeration of all
    65536 uniforms) and only ever returns the two neighbouring grid points;
  * per-element error bounds; the block maximum takes inner scale 448 and
    code 6; zero blocks give zeros; scale invariance under powers of two;
  * tensors built from grid values quantize exactly (the special case that
    reduces the method to a plain matmul);
  * MXFP8: values representable in the slice's format round-trip exactly.
"""
import numpy as np
import pytest

from oracle import formats as F
from oracle import quant as Q

F32 = np.float32


def _dense_a_values():
    """All fp32 values near every grid point and midpoint in [0, 6], plus a dense sweep."""
    pts = np.concatenate([F.E2M1_GRID, (F.E2M1_GRID[1:] + F.E2M1_GRID[:-1]) / 2]).astype(F32)
    near = [pts]
    x = pts.copy()
    y = pts.copy()
    for _ in range(64):
        x = np.nextafter(x, F32(np.inf))
        y = np.nextafter(y, F32(0))
        near += [x.copy(), y.copy()]
    sweep = np.linspace(0, 6, 200001, dtype=np.float64).astype(F32)
    a = np.concatenate(near + [sweep])
    return np.unique(a[(a >= 0) & (a <= 6)])


def test_rtn_is_nearest_grid_point_ties_even():
    a = _dense_a_values()
    idx = Q.rtn_index(a)
    d = np.abs(a.astype(np.float64)[:, None] - F.E2M1_GRID.astype(np.float64)[None, :])
    best = d.min(axis=1)
    assert np.all(d[np.arange(len(a)), idx] == best)
    ties = (d == best[:, None]).sum(axis=1) > 1
    assert ties.sum() == 7                                  # the 7 midpoints
    assert np.all(idx[ties] % 2 == 0)


def test_sr_enumeration_is_unbiased():
    a = _dense_a_values()[::37]
    u = np.arange(65536, dtype=np.uint32)
    for ai in a:
        idx = Q.sr_index(np.full(65536, ai, dtype=F32), u)
        vals = F.E2M1_GRID[idx].astype(np.float64)
        lo = F.E2M1_GRID[F.E2M1_GRID <= ai].max()
        hi = F.E2M1_GRID[F.E2M1_GRID >= ai].min()
        assert set(np.unique(vals)) <= {lo, hi}
        gap = max(hi - lo, 1e-30)
        assert abs(vals.mean() - float(ai)) <= gap * 2.0 ** -16 + 1e-12


def test_sr_sampled_mean_converges():
    # 10^5 draws of SR(x) through the full quantizer: mean -> x within 5 sigma
    rng = np.random.default_rng(3)
    row = (rng.standard_normal(128) * 0.7).astype(F32)
    row[0] = 3.0
    reps = 100000 // 128 + 1
    x = np.tile(row, (reps, 1))
    c, s, o = Q.quantize_nvfp4(x, Q.SR, seed=9, tag=1)
    xh = Q.dequantize_nvfp4_f64(c, s, o)
    mean = xh.mean(axis=0)
    std = xh.std(axis=0) + 1e-12
    # plus the fp32 rounding of the scaled value v = x * r (relative 2^-22 at most)
    assert np.all(np.abs(mean - row) <= 5 * std / np.sqrt(reps) + np.abs(row) * 2.0 ** -21)


def _random_rows(seed, R=64, L=512):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((R, L)).astype(F32)
    x[:, rng.choice(L, 5, replace=False)] *= 30
    x[3, 128:256] = 0                                   # an all-zero outer block
    x[4, 16:32] = 0                                     # an all-zero inner block
    x[5] *= F32(2.0 ** -20)                             # small magnitudes
    return x


@pytest.mark.parametrize("mode", [Q.RTN, Q.SR])
def test_codes_scales_and_error_bound(mode):
    x = _random_rows(4)
    c, s, o = Q.quantize_nvfp4(x, mode, seed=5, tag=3)
    assert c.shape == (64, 512) and s.shape == (64, 32) and o.shape == (64, 4)
    assert c.max() <= 15 and s.max() <= 0x7E
    xh = Q.dequantize_nvfp4_f64(c, s, o)
    s_elem = np.repeat(F.e4m3_decode(s), 16, axis=1) * np.repeat(o.astype(np.float64), 128, axis=1)
    err = np.abs(xh - x)
    # grid gap around |x|/s is at most 2 (between 4 and 6); RTN error <= gap/2, SR < gap
    v = np.abs(x) / np.where(s_elem > 0, s_elem, 1)
    gap = np.select([v <= 2, v <= 4], [0.5, 1.0], 2.0)
    bound = (0.5 if mode == Q.RTN else 1.0) * gap * s_elem * (1 + 1e-6)
    assert np.all(err <= bound + 1e-30)
    # zero blocks give zero codes, zero inner scale bytes, zero outer scale
    assert np.all(c[3, 128:256] == 0) and np.all(s[3, 8:16] == 0) and o[3, 1] == 0
    assert np.all(c[4, 16:32] == 0) and s[4, 1] == 0


def test_block_maximum_takes_top_scale_and_code():
    x = _random_rows(5)
    c, s, o = Q.quantize_nvfp4(x, Q.RTN)
    R, L = x.shape
    for r in range(R):
        for b in range(L // 128):
            blk = x[r, b * 128:(b + 1) * 128]
            if np.all(blk == 0):
                continue
            sb = s[r, b * 8:(b + 1) * 8]
            assert sb.max() == 0x7E                     # inner scale 448 at the block max
            for j in range(8):
                inner = blk[j * 16:(j + 1) * 16]
                if F.e4m3_decode(sb[j]) >= 2.0 ** -6:  # normal inner scale
                    assert (c[r, b * 128 + j * 16: b * 128 + (j + 1) * 16] & 7).max() == 7, (r, b, j)


def test_scale_invariance_power_of_two():
    x = _random_rows(6)
    x[5] = 1                                            # keep away from subnormals
    c, s, o = Q.quantize_nvfp4(x, Q.SR, seed=1, tag=1)
    for k in (-7, 3, 11):
        c2, s2, o2 = Q.quantize_nvfp4(x * F32(2.0 ** k), Q.SR, seed=1, tag=1)
        assert np.array_equal(c, c2) and np.array_equal(s, s2)
        assert np.array_equal(o2, (o * F32(2.0 ** k)).astype(F32))


def grid_tensor(rng, R, L, so_exp_range=(-12, -4)):
    """A tensor every 16-block of which holds a +-6 and grid values only, with an
    E4M3 inner scale (448 in the first block of each 128) and a power-of-two
    outer scale: it quantizes exactly under the method's scale rules."""
    x = np.zeros((R, L), dtype=np.float64)
    normal_scales = [F.e4m3_decode(np.uint8(b)) for b in range(0x30, 0x7F)]   # >= 2^-6 *...
    for r in range(R):
        for b in range(L // 128):
            so = 2.0 ** rng.integers(*so_exp_range)
            for j in range(8):
                si = 448.0 if j == 0 else float(rng.choice(normal_scales))
                g = F.E2M1_GRID[rng.integers(0, 8, 16)].astype(np.float64)
                g[rng.integers(0, 16)] = 6.0
                g *= rng.choice([-1.0, 1.0], 16)
                x[r, b * 128 + j * 16: b * 128 + (j + 1) * 16] = g * si * so
    return x.astype(F32)


def test_grid_tensors_quantize_exactly():
    rng = np.random.default_rng(7)
    x = grid_tensor(rng, 16, 384)
    for mode in (Q.RTN, Q.SR):
        c, s, o = Q.quantize_nvfp4(x, mode, seed=3, tag=2)
        assert np.array_equal(Q.dequantize_nvfp4_f64(c, s, o), x.astype(np.float64))
        assert np.array_equal(Q.dequantize_nvfp4_f32(c, s, o), x)


def test_padding_and_row_ids():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((6, 200)).astype(F32)
    c, s, o = Q.quantize_nvfp4(x, Q.SR, seed=2, tag=4)
    assert c.shape == (6, 256) and np.all(c[:, 200:] == 0)
    # quantizing a subset of rows with their row ids reproduces those rows
    c2, s2, o2 = Q.quantize_nvfp4(x[[1, 4]], Q.SR, seed=2, tag=4, row_ids=[1, 4])
    assert np.array_equal(c2, c[[1, 4]]) and np.array_equal(s2, s[[1, 4]])


def test_mxfp8_roundtrip_and_bound():
    rng = np.random.default_rng(9)
    # values exactly representable: E4M3 values times a per-block power of two
    R, L = 8, 256
    bytes_ = rng.integers(0, 0x7F, (R, L)).astype(np.uint8)
    bytes_[:, ::32] = 0x7E                               # each 32-block reaches 448
    sign = rng.choice([0, 0x80], (R, L)).astype(np.uint8)
    E = rng.integers(-20, 10, (R, L // 32))
    x = (F.e4m3_decode(bytes_ | sign) * np.repeat(np.exp2(E), 32, axis=1)).astype(F32)
    codes, sb = Q.quantize_mxfp8(x)
    assert np.array_equal(Q.dequantize_mxfp8_f64(codes, sb), x.astype(np.float64))
    assert np.array_equal(sb.astype(np.int64) - 127, E)
    # random input: relative error of an E4M3 value is at most 2^-4, scale never clips
    y = (rng.standard_normal((R, 300)) * 40).astype(F32)
    cq, sq = Q.quantize_mxfp8(y)
    yh = Q.dequantize_mxfp8_f64(cq, sq)[:, :300]
    blk_scale = np.repeat(np.exp2(sq.astype(np.float64) - 127), 32, axis=1)[:, :300]
    assert np.all(np.abs(yh - y) <= np.maximum(np.abs(y) * 2.0 ** -4, blk_scale * 2.0 ** -10) + 1e-30)
    assert np.all(np.abs(yh) <= 448 * blk_scale)
