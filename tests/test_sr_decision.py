"""The stochastic-rounding decision the quantize kernels take, restated on the CPU.

The kernels decide SR two elements at a time without comparisons: with a = min(|v|, 6) and
the element's 16-bit uniform U,
    S = max(bits of RP(0.5 + a / 2), bits of a)       (RP: fp32 rounded towards +infinity)
    T = S * 64 + ((U << 12) xor 0x4FFFFFC0)           (mod 2^32)
and the E2M1 grid index is T >> 28.  This file restates that integer recipe in numpy and
checks it against the oracle's definition of SR (`oracle.quant.sr_index`: round up from the
grid point below iff float(U) < p * 65536), so the recipe's exactness is pinned on the CPU:
- every fp32 value within 24 ulps of each grid point and each midpoint, with all 65536 uniforms;
- a dense stride through [0, 6], with uniforms on a stride plus the ends 0 and 65535;
- every uniform near the decision threshold of random values.
The GPU tests then compare the kernels' codes with the oracle bit for bit.
"""
import numpy as np

from oracle import quant as Q

GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float32)


def _half_plus_half_rp(a):
    """0.5 + a / 2 rounded to fp32 towards +infinity, for fp32 a in [0, 6].  The fp64 sum can
    itself round (a tiny a), so the comparison uses the exact parts: f - 0.5 and a / 2 are
    both exact in fp64."""
    half_a = a.astype(np.float64) * 0.5
    f = (half_a + 0.5).astype(np.float32)
    low = (f.astype(np.float64) - 0.5) < half_a
    f[low] = np.nextafter(f[low], np.float32(np.inf))
    return f


def _recipe_index(a, u):
    """Grid index by the kernels' integer recipe; a fp32 in [0, 6], u uint in [0, 65535]."""
    a = np.asarray(a, dtype=np.float32)
    f = _half_plus_half_rp(a)
    s = np.maximum(f.view(np.uint32), a.view(np.uint32)).astype(np.uint64)
    uc = ((np.asarray(u, dtype=np.uint64) << np.uint64(12)) ^ np.uint64(0x4FFFFFC0))
    t = (s * np.uint64(64) + uc) & np.uint64(0xFFFFFFFF)
    return (t >> np.uint64(28)).astype(np.uint8)


def _check(a, u):
    a = np.asarray(a, dtype=np.float32)
    u = np.asarray(u, dtype=np.uint32)
    got = _recipe_index(a, u)
    ref = Q.sr_index(a, u)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, ("recipe differs from the oracle", float(a[bad[0]]), int(u[bad[0]]), int(got[bad[0]]),
                           int(ref[bad[0]]))


def _neighbours(v, n):
    """n fp32 values on each side of v (inside [0, 6]), v included."""
    b = np.float32(v).view(np.int32)
    out = (b + np.arange(-n, n + 1, dtype=np.int32)).view(np.float32)
    return out[(out >= 0) & (out <= 6) & np.isfinite(out)]


def test_recipe_near_grid_points_and_midpoints_all_uniforms():
    points = list(GRID) + [(GRID[i] + GRID[i + 1]) / 2 for i in range(7)]
    a = np.unique(np.concatenate([_neighbours(p, 24) for p in points] + [np.array([0.0], np.float32)]))
    u = np.arange(65536, dtype=np.uint32)
    for chunk in np.array_split(a, 8):
        aa = np.repeat(chunk, u.size)
        uu = np.tile(u, chunk.size)
        _check(aa, uu)


def test_recipe_dense_stride_through_the_range():
    # every 389th fp32 value in [0, 6] (about 2.8 million), each with a spread of uniforms
    top = np.float32(6.0).view(np.int32)
    a = np.arange(0, top + 1, 389, dtype=np.int32).view(np.float32)
    u_set = np.array([0, 1, 2, 255, 256, 4095, 4096, 32767, 32768, 40000, 65534, 65535], dtype=np.uint32)
    for i, uv in enumerate(u_set):
        sub = a[i::4]                      # a quarter of the values per uniform keeps it quick
        _check(sub, np.full(sub.size, uv, dtype=np.uint32))


def test_recipe_at_the_decision_threshold():
    # for random a, the uniforms on either side of p * 65536, where the decision flips
    rng = np.random.default_rng(0)
    a = (rng.random(200000) * 6.0).astype(np.float32)
    hi = np.minimum(np.searchsorted(GRID, a, side="left"), 7)
    lo = np.maximum(hi - 1, 0)
    gap = np.where(GRID[hi] == a, np.float32(1.0), GRID[hi] - GRID[lo])
    p = ((a - GRID[lo]) / gap).astype(np.float32)
    thr = np.floor(p.astype(np.float64) * 65536.0).astype(np.int64)
    for d in (-2, -1, 0, 1, 2):
        u = np.clip(thr + d, 0, 65535).astype(np.uint32)
        _check(a, u)
