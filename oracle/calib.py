"""OutControl static outlier calibration.

Test infrastructure only (see the package docstring).

TetraJet-v2 technical summary §2.C: outlier channels are structurally
consistent (the same channels always have large norms), so the top p% of
channels (e.g. 10%) are found once, during a short calibration window, and
kept in higher precision from then on.

Readings: channels are the input features of the linear layer;
they are ranked by the squared L2 norm summed over the calibration batches;
k = ceil(p * K); ties go to the lower channel index; the result is returned
in ascending order together with its ascending complement.  The fp64 sum
runs in a fixed order so that any implementation can reproduce it bit for
bit: per channel, over the tokens of each 128-token chunk in order, then over
the chunks in order, then added to the running total of earlier batches.
"""
import numpy as np

CHUNK = 128


def accumulate_sumsq(x, sumsq):
    """Add this batch's per-channel sum of squares (fp64, fixed order) to sumsq [K]."""
    x = np.asarray(x, dtype=np.float64)               # bf16/fp32 -> fp64 is exact
    M, K = x.shape
    batch = np.zeros(K, dtype=np.float64)
    for c0 in range(0, M, CHUNK):
        chunk = np.zeros(K, dtype=np.float64)
        for t in range(c0, min(c0 + CHUNK, M)):
            chunk = chunk + x[t] * x[t]               # x*x is exact in fp64
        batch = batch + chunk
    return np.asarray(sumsq, dtype=np.float64) + batch


def top_k_channels(sumsq, k):
    """(outlier indices ascending [k], normal indices ascending [K-k])."""
    s = np.asarray(sumsq, dtype=np.float64)
    K = len(s)
    order = sorted(range(K), key=lambda c: (-s[c], c))
    out = np.array(sorted(order[:k]), dtype=np.int64)
    mask = np.ones(K, dtype=bool)
    mask[out] = False
    return out, np.nonzero(mask)[0].astype(np.int64)


def outlier_count(K, percent):
    """k = ceil(percent * K / 100) in integer arithmetic."""
    return (int(percent) * int(K) + 99) // 100
