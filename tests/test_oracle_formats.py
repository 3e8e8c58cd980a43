"""Pins for oracle.formats and oracle.philox against sources outside the oracle.

* E4M3 decode: the OCP FP8 specification's values (golden fixture) and
  torch's independent float8_e4m3fn implementation for all 256 bytes.
* E4M3 round-up: brute-force "smallest representable >= t".
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


def test_e4m3_ceil_brute_force():
    rng = np.random.default_rng(0)
    vals = np.array([F.e4m3_decode(np.uint8(b)) for b in range(0x7F)])   # 0 .. 448
    # every representable value, its neighbours in fp32, midpoints, random values
    t = np.concatenate([
        vals,
        np.nextafter(vals.astype(np.float32), np.float32(np.inf)).astype(np.float64),
        np.nextafter(vals.astype(np.float32), np.float32(0)).astype(np.float64),
        (vals[1:] + vals[:-1]) / 2,
        rng.uniform(0, 448, 20000),
        np.exp2(rng.uniform(-14, 9, 20000)),
        [449.0, 500.0, 1e6],
    ]).astype(np.float32).astype(np.float64)
    t = t[t >= 0]
    got = F.e4m3_decode(F.e4m3_ceil_byte(t))
    for ti, gi in zip(t, got):
        if ti > 448:
            assert gi == 448
            continue
        # brute force: the smallest representable value >= ti
        expect = min(v for v in vals if v >= ti)
        assert gi == expect, (ti, gi, expect)


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
