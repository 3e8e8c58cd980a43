"""Pins for oracle.formats and oracle.philox against sources outside the oracle.

* E4M3 decode: the OCP FP8 specification's values (golden fixture) and
  torch's independent float8_e4m3fn implementation for all 256 bytes.
* Inner-scale rounding: exact (fp64) arithmetic, up to one fp32 product rounding.
* E4M3 round-to-nearest-even: torch's fp32 -> float8_e4m3fn conversion.
* E2M1 grid: derived from the bit-field definition (bias 1, 1 mantissa bit).
* Philox4x32-10: the algorithm authors' published known-answer vectors.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import philox as P
from oracle.quant import mx_exponent


def _read_table(path):
    rows = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def test_e4m3_decode_matches_ocp_examples(golden_dir):
    for byte, val in _read_table(os.path.join(golden_dir, "e4m3_ocp.txt")):
        got = F.e4m3_decode(np.uint8(int(byte, 16)))
        if val == "nan":
            assert np.isnan(got)
        else:
            assert got == float(val), byte


def test_e4m3_decode_matches_torch_all_bytes():
    b = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = F.e4m3_decode(b)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])


def _inner_scale_cases(rng):
    """(a_i, s_o) pairs: random magnitudes, and group maxima placed exactly on, and a few
    fp32 ulps around, the top value 6 sigma s_o of every candidate scale sigma."""
    s_o = np.exp2(rng.uniform(-60, 60, 4000)).astype(np.float32)
    a = (s_o.astype(np.float64) * rng.uniform(0, 2688 * 1.2, 4000)).astype(np.float32)
    sig = F.e4m3_decode(rng.integers(0x01, 0x7F, 6000).astype(np.uint8))
    so2 = np.exp2(rng.uniform(-60, 60, 6000)).astype(np.float32)
    on = (6 * sig * so2.astype(np.float64)).astype(np.float32)
    near = [on]
    for k in (1, 2, 3):
        up, dn = on.copy(), on.copy()
        for _ in range(k):
            up = np.nextafter(up, np.float32(np.inf))
            dn = np.nextafter(dn, np.float32(0))
        near += [up, dn]
    tiny = np.exp2(rng.uniform(-40, 0, 2000)) * 2688 * s_o[:2000].astype(np.float64)
    a_all = np.concatenate([a] + near + [tiny.astype(np.float32), np.zeros(3, np.float32)])
    s_all = np.concatenate([s_o] + [so2] * 7 + [s_o[:2000], np.ones(3, np.float32)])
    return a_all, s_all


def test_inner_scale_against_exact_arithmetic():
    """The inner scale is, up to the fp32 rounding of one product, the smallest normal
    E4M3 value sigma with 6 sigma s_o >= a_i in exact arithmetic (fp64 holds 6 sigma s_o
    exactly: 6 sigma has at most 6 significant bits, s_o 24).  It may sit one step lower
    only where the exact top value of that lower scale is within half an fp32 ulp below
    a_i, so that rounding the product lifts it onto a_i."""
    rng = np.random.default_rng(0)
    a_all, s_all = _inner_scale_cases(rng)
    got = F.e4m3_inner_scale_byte(a_all, s_all)
    normal = [(b, float(F.e4m3_decode(np.uint8(b)))) for b in range(0x08, 0x7F)]
    lower = 0
    for ai, so, gb in zip(a_all.astype(np.float64), s_all.astype(np.float64), got):
        if ai == 0:
            assert gb == 0
            continue
        fits = [b for b, v in normal if 6 * v * so >= ai]
        exact = fits[0] if fits else 0x7E
        if gb == exact:
            continue
        assert gb == exact - 1 and gb >= 0x08, (ai, so, gb, exact)
        top = 6 * float(F.e4m3_decode(np.uint8(gb))) * so
        assert top < ai and (ai - top) <= 0.5 * np.spacing(np.float32(ai)), (ai, so, gb)
        lower += 1
    assert lower > 0                     # the boundary cases were reached


def test_inner_scale_is_normal_and_never_clips():
    """Every nonzero group gets a normal E4M3 scale (>= 2^-6), and its maximum scaled
    by 1/(s_i s_o) stays within the E2M1 range up to the rounding of that division."""
    rng = np.random.default_rng(1)
    a_all, s_all = _inner_scale_cases(rng)
    sb = F.e4m3_inner_scale_byte(a_all, s_all)
    nz = a_all > 0
    assert np.all(sb[nz] >= 0x08) and np.all(sb[nz] <= 0x7E) and np.all(sb[~nz] == 0)
    s = F.e4m3_decode(sb[nz]) * s_all[nz].astype(np.float64)
    inside = sb[nz] < 0x7E               # 448 is a clamp: the largest amax of a block
    v = a_all[nz].astype(np.float64) / s
    assert np.all(v[inside] <= 6 * (1 + 2.0 ** -22))


def test_e4m3_rne_matches_torch():
    rng = np.random.default_rng(1)
    vals = np.array([F.e4m3_decode(np.uint8(b)) for b in range(0x7F)])
    x = np.concatenate([
        vals, -vals, (vals[1:] + vals[:-1]) / 2, -(vals[1:] + vals[:-1]) / 2,
        rng.standard_normal(50000) * 50, np.exp2(rng.uniform(-14, 8.8, 50000)),
    ]).astype(np.float32)
    x = x[np.abs(x) < 464]                      # torch does not saturate beyond 464
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = F.e4m3_rne_satfinite_byte(x)
    assert np.array_equal(ref, got)
    # saturation: everything beyond the largest finite value clamps to +-448
    big = np.array([448.0, 460.0, 470.0, 1e5, -1e5, -470.0], dtype=np.float32)
    assert list(F.e4m3_rne_satfinite_byte(big)) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]


def test_e2m1_grid_from_bit_fields():
    # E2M1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit; exponent 0 is subnormal
    vals = []
    for e in range(4):
        for m in range(2):
            vals.append((m / 2) * 2.0 ** 0 if e == 0 else (1 + m / 2) * 2.0 ** (e - 1))
    assert list(F.E2M1_GRID.astype(np.float64)) == vals
    # the pages' example: 0 and 0.5 are adjacent representable values
    assert F.E2M1_GRID[0] == 0.0 and F.E2M1_GRID[1] == 0.5
    assert F.e2m1_decode(0x8 | 7) == -6.0 and F.e2m1_decode(0x8) == 0.0


def test_ue8m0():
    assert F.ue8m0_decode(127) == 1.0
    assert F.ue8m0_decode(0) == 2.0 ** -127
    assert F.ue8m0_decode(254) == 2.0 ** 127


def test_mx_exponent_brute_force():
    rng = np.random.default_rng(2)
    a = np.concatenate([
        448.0 * np.exp2(np.arange(-40, 40, dtype=np.float64)),
        np.nextafter((448.0 * np.exp2(np.arange(-40, 40))).astype(np.float32), np.float32(np.inf)),
        np.exp2(rng.uniform(-60, 60, 5000)),
    ]).astype(np.float32).astype(np.float64)
    E = mx_exponent(a)
    for ai, ei in zip(a, E):
        assert 448.0 * 2.0 ** ei >= ai
        assert 448.0 * 2.0 ** (ei - 1) < ai


def test_philox_known_answers(golden_dir):
    for row in _read_table(os.path.join(golden_dir, "philox4x32_10_kat.txt")):
        v = [int(h, 16) for h in row]
        out = P.philox4x32_10(*v[:6])
        assert [int(o) for o in out] == v[6:]


def test_sr_uniform16_word_mapping_and_uniformity():
    e = np.arange(1 << 16, dtype=np.uint64)
    u = P.sr_uniform16(e, seed=123, tag=1)
    # element 8g+j reads 16-bit half (j & 1) of word (j >> 1) of call g
    w = P.philox4x32_10(5, 0, 1, 0, *P.seed_key(123))
    for j in range(8):
        assert u[8 * 5 + j] == (int(w[j >> 1]) >> (16 * (j & 1))) & 0xFFFF
    # uniformity: mean and per-bit frequencies of 65536 draws
    assert abs(u.mean() / 65535.0 - 0.5) < 0.005
    bits = ((u[:, None] >> np.arange(16)) & 1).mean(axis=0)
    assert np.all(np.abs(bits - 0.5) < 0.01)
    # distinct tags and seeds give distinct streams
    assert not np.array_equal(u, P.sr_uniform16(e, seed=123, tag=2))
    assert not np.array_equal(u, P.sr_uniform16(e, seed=124, tag=1))


def test_rht_signs_balanced():
    d = P.rht_signs(7, 0x100)
    assert set(np.unique(d)) <= {-1.0, 1.0}
    assert abs(d.sum()) < 40
    assert not np.array_equal(d, P.rht_signs(7, 0x101))
