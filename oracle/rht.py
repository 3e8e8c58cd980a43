"""128-point random Hadamard transform (RHT).

Test infrastructure only (see the package docstring).

TetraJet-v2 technical summary §2.C: the RHT is applied to the backward
contractions (dX and dW) to spread outlier energy over channels and lower the
quantization variance.  Reading (the pages give neither the size nor the sign
rule): blocks of 128 along the contraction dimension, y = H_128 (d * x) with
the unnormalised Sylvester Hadamard matrix and a random +-1 diagonal d drawn
from Philox (oracle.philox.rht_signs).  Both operands of one GEMM use the same
d, so H^T H = 128 I makes the transformed product exactly 128 times the
original; the GEMM multiplies by 2^-7 to undo it.

The butterfly runs in fp32 in a fixed stage order h = 1, 2, 4, ..., 64; at
stage h every pair (i, i + h) with i & h == 0 becomes (a + b, a - b).
"""
import numpy as np

F32 = np.float32
RHT_N = 128


def fwht128_f32(x):
    """Unnormalised Walsh-Hadamard transform of each 128-block of the last axis (fp32)."""
    y = np.array(x, dtype=F32, copy=True)
    assert y.shape[-1] % RHT_N == 0
    lead, nblk = y.shape[:-1], y.shape[-1] // RHT_N
    y = y.reshape(*lead, nblk, RHT_N)          # (an explicit block count: rows may be empty)
    h = 1
    while h < RHT_N:
        idx = np.arange(RHT_N)
        i = idx[(idx & h) == 0]
        a = y[..., i].copy()
        b = y[..., i + h].copy()
        y[..., i] = (a + b).astype(F32)
        y[..., i + h] = (a - b).astype(F32)
        h *= 2
    return y.reshape(*lead, nblk * RHT_N)


def rht_f32(x, d):
    """RHT of each 128-block of the last axis of x (already zero-padded): H (d * x)."""
    x = np.asarray(x, dtype=F32)
    L = x.shape[-1]
    assert L % RHT_N == 0
    dd = np.tile(np.asarray(d, dtype=F32), L // RHT_N)
    return fwht128_f32((x * dd).astype(F32))
