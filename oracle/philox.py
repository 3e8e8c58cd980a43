"""Philox4x32-10 counter-based generator.

Test infrastructure only (see the package docstring).

Algorithm: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel
Random Numbers: As Easy as 1, 2, 3", SC'11.  A 128-bit counter and a 64-bit
key go through 10 rounds; each round multiplies counter words 0 and 2 by the
constants M0, M1 into 64-bit products, swaps/xors the halves with the other
counter words and the round key, and the key is bumped by the Weyl constants
W0, W1 between rounds.

The pages do not name a generator; stochastic rounding (§2.A) and the random
signs of the RHT (§2.C) need reproducible uniform bits, and a counter-based
generator keyed by (seed, element index) lets every element be drawn
independently of launch order.
"""
import numpy as np

PHILOX_M0 = np.uint64(0xD2511F53)
PHILOX_M1 = np.uint64(0xCD9E8D57)
PHILOX_W0 = np.uint64(0x9E3779B9)
PHILOX_W1 = np.uint64(0xBB67AE85)
_MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Vectorised Philox4x32-10.  All arguments are uint32-valued arrays/scalars.

    Returns a tuple of four uint64 arrays holding the 32-bit output words.
    """
    c = [np.asarray(v, dtype=np.uint64) & _MASK32 for v in (c0, c1, c2, c3)]
    k0 = np.asarray(k0, dtype=np.uint64) & _MASK32
    k1 = np.asarray(k1, dtype=np.uint64) & _MASK32
    for rnd in range(10):
        p0 = PHILOX_M0 * c[0]                      # < 2^64, exact in uint64
        p1 = PHILOX_M1 * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
        if rnd != 9:
            k0 = (k0 + PHILOX_W0) & _MASK32
            k1 = (k1 + PHILOX_W1) & _MASK32
    return tuple(c)


def seed_key(seed):
    """64-bit seed -> (k0, k1) = (low 32 bits, high 32 bits)."""
    s = int(seed) & 0xFFFFFFFFFFFFFFFF
    return np.uint64(s & 0xFFFFFFFF), np.uint64(s >> 32)


def sr_uniform16(elem_index, seed, tag):
    """16-bit uniforms for stochastic rounding, one per element index.

    Reading (SR resolution): element e of a quantized operand (e = row * Lp +
    col in the operand's quantized layout) uses Philox with counter
    (g lo32, g hi32, tag, 0), g = e >> 3, key = seed; of the 128 output bits,
    word (e & 7) >> 1 supplies the 16 bits, the low half for even e.
    """
    e = np.asarray(elem_index, dtype=np.uint64)
    g = e >> np.uint64(3)
    k0, k1 = seed_key(seed)
    w = philox4x32_10(g & _MASK32, g >> np.uint64(32), np.uint64(tag), np.uint64(0), k0, k1)
    words = np.stack(w, axis=0)                                    # [4, ...]
    sel = ((e & np.uint64(7)) >> np.uint64(1)).astype(np.int64)
    word = np.take_along_axis(words, sel[None, ...], axis=0)[0]
    shift = (e & np.uint64(1)) * np.uint64(16)
    return ((word >> shift) & np.uint64(0xFFFF)).astype(np.uint32)


def rht_signs(seed, tag, n=128):
    """The ±1 diagonal of the random Hadamard transform (§2.C).

    One Philox call with counter (0, 0, tag, 0) and key = seed; bit i of the
    128 output bits (word i >> 5, bit i & 31) set means d[i] = -1.
    """
    assert n == 128
    k0, k1 = seed_key(seed)
    w = philox4x32_10(0, 0, tag, 0, k0, k1)
    d = np.empty(n, dtype=np.float32)
    for i in range(n):
        bit = (int(w[i >> 5]) >> (i & 31)) & 1
        d[i] = -1.0 if bit else 1.0
    return d
