"""Pins for the oracle's RHT and linear-layer compositions.

* FWHT equals multiplication by scipy's Sylvester Hadamard matrix (a library
  routine), H H^T = 128 I, the transform inverts as D H / 128, one-hot inputs
  give signed columns of H.
* The forward on grid-valued inputs (which quantize exactly) equals a plain
  fp64 matmul, with and without an FP8 outlier slice.
* The backward is unbiased: averaged over seeds, dX and dW converge to
  dY W-hat and dY^T X-hat at the 1/sqrt(n) rate (SR is unbiased and the
  random Hadamard factors cancel, which is why the pages use both).
"""
import numpy as np
import scipy.linalg

from oracle import linear as Lin
from oracle import quant as Q
from oracle.philox import rht_signs
from oracle.rht import fwht128_f32, rht_f32
from test_oracle_quant import grid_tensor

F32 = np.float32


def test_fwht_matches_sylvester_matrix():
    H = scipy.linalg.hadamard(128).astype(np.float64)
    assert np.array_equal(H @ H.T, 128 * np.eye(128))
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 384)).astype(F32)
    y = fwht128_f32(x).astype(np.float64)
    ref = (x.astype(np.float64).reshape(5, 3, 128) @ H.T).reshape(5, 384)
    # 7 fp32 butterfly stages: error bounded by 7 * 2^-24 * sum |x| per output
    bound = 7 * 2.0 ** -24 * np.abs(x).reshape(5, 3, 128).sum(axis=2).repeat(128, axis=1) * 1.01
    assert np.all(np.abs(y - ref) <= bound)
    # one-hot e_j -> column j of H, exactly
    e = np.zeros((128, 128), dtype=F32)
    e[np.arange(128), np.arange(128)] = 1
    assert np.array_equal(fwht128_f32(e).astype(np.float64), H.T)


def test_rht_inverse_and_signs():
    rng = np.random.default_rng(1)
    d = rht_signs(11, 0x100)
    x = rng.standard_normal((4, 256)).astype(F32)
    y = rht_f32(x, d)
    back = (np.tile(d, 2) * fwht128_f32(y)).astype(np.float64) / 128.0
    assert np.allclose(back, x, rtol=0, atol=1e-5)
    # the transformed product is 128 times the plain product (same d on both sides)
    z = rng.standard_normal((3, 256)).astype(F32)
    prod = rht_f32(x, d).astype(np.float64) @ rht_f32(z, d).astype(np.float64).T
    assert np.allclose(prod * Lin.ALPHA_RHT, x.astype(np.float64) @ z.astype(np.float64).T, atol=1e-4)


def test_forward_on_grid_inputs_is_plain_matmul():
    rng = np.random.default_rng(2)
    X = grid_tensor(rng, 32, 256)
    W = grid_tensor(rng, 48, 256)
    Y, fx, fw = Lin.forward(X, W, [])
    assert np.array_equal(Y, X.astype(np.float64) @ W.astype(np.float64).T)


def test_forward_with_outlier_slice_on_representable_inputs():
    rng = np.random.default_rng(3)
    K, k = 256 + 32, 32
    X = np.zeros((16, K), dtype=F32)
    W = np.zeros((24, K), dtype=F32)
    o = np.sort(rng.choice(K, k, replace=False))
    nc = Lin.normal_channels(K, o)
    X[:, nc] = grid_tensor(rng, 16, 256)
    W[:, nc] = grid_tensor(rng, 24, 256)
    # outlier columns: integers up to 2^4 times 2^e (exact in E4M3 with a UE8M0 scale)
    X[:, o] = (rng.integers(-16, 17, (16, k)) * 4.0).astype(F32)
    X[:, o[0]] = 448.0 * 4.0
    W[:, o] = (rng.integers(-16, 17, (24, k)) / 64.0).astype(F32)
    W[:, o[0]] = 448.0 / 64.0
    Y, fx, fw = Lin.forward(X, W, o)
    assert np.array_equal(Y, X.astype(np.float64) @ W.astype(np.float64).T)
    # the saved forward operand dequantizes to X itself on both channel sets
    assert np.array_equal(Lin.deq_normal_f32(fx), X[:, nc])
    assert np.array_equal(Lin.deq_outlier_f32(fx), X[:, o])


def _mean_error(fn, exact, seeds):
    acc = np.zeros_like(exact)
    errs = {}
    for i, s in enumerate(seeds, 1):
        acc += fn(s)
        if i in (1, len(seeds)):
            errs[i] = np.linalg.norm(acc / i - exact) / np.linalg.norm(exact)
    return errs


def test_backward_is_unbiased_over_seeds():
    rng = np.random.default_rng(4)
    M, N, K = 128, 256, 128
    X = rng.standard_normal((M, K)).astype(F32)
    W = (rng.standard_normal((N, K)) * 0.05).astype(F32)
    dY = (rng.standard_normal((M, N)) * 1e-3).astype(F32)
    dY[:, 5] *= 20                                          # an outlier column in dY
    _, fx, fw = Lin.forward(X, W, [])
    W_hat = Lin.deq_normal_f32(fw).astype(np.float64)
    X_hat = Lin.deq_normal_f32(fx).astype(np.float64)
    seeds = list(range(100, 164))
    ex = dY.astype(np.float64) @ W_hat
    e = _mean_error(lambda s: Lin.bwd_dx(dY, fw, [], s), ex, seeds)
    assert e[64] < 0.2 * e[1]                                # ~1/8 expected for 64 seeds
    ew = dY.astype(np.float64).T @ X_hat
    e = _mean_error(lambda s: Lin.bwd_dw(dY, fx, [], s), ew, seeds)
    assert e[64] < 0.2 * e[1]


def test_backward_outlier_columns_use_fp8_slice():
    rng = np.random.default_rng(5)
    M, N, K = 64, 128, 160
    o = np.array([3, 77, 150])
    X = rng.standard_normal((M, K)).astype(F32)
    X[:, o] *= 40
    W = (rng.standard_normal((N, K)) * 0.05).astype(F32)
    dY = (rng.standard_normal((M, N)) * 1e-3).astype(F32)
    _, fx, fw = Lin.forward(X, W, o)
    dX = Lin.bwd_dx(dY, fw, o, 7)
    dW = Lin.bwd_dw(dY, fx, o, 7)
    W_o = Lin.deq_outlier_f32(fw).astype(np.float64)
    X_o = Lin.deq_outlier_f32(fx).astype(np.float64)
    # FP8 slices: relative error of each operand <= 2^-4, no RHT / SR noise
    ref_dx = dY.astype(np.float64) @ W_o
    ref_dw = dY.astype(np.float64).T @ X_o
    mag_dx = np.abs(dY).astype(np.float64) @ np.abs(W_o)
    mag_dw = np.abs(dY).astype(np.float64).T @ np.abs(X_o)
    assert np.all(np.abs(dX[:, o] - ref_dx) <= mag_dx * (2 * 2.0 ** -4 + 2.0 ** -8) + 1e-12)
    assert np.all(np.abs(dW[:, o] - ref_dw) <= mag_dw * (2 * 2.0 ** -4 + 2.0 ** -8) + 1e-12)
    # FP8 slice is deterministic (no seed dependence); FP4 columns are seeded
    assert np.array_equal(Lin.bwd_dx(dY, fw, o, 8)[:, o], dX[:, o])
    assert not np.array_equal(Lin.bwd_dx(dY, fw, o, 8)[:, 0], dX[:, 0])


# ---------------------------------------------------------------------------
# FP8 linear baseline (technical summary §4's comparison): exact on tensors whose
# every 32-block, along rows and along columns, reaches +-448 with E4M3 values, so
# that forward, dX and dW reduce to the plain matmul; otherwise within the E4M3
# rounding bound of both operands.
# ---------------------------------------------------------------------------
def _exact_fp8_tensor(rng, R, C):
    from oracle import formats as Fm
    vals = Fm.e4m3_decode(rng.integers(0, 0x7F, (R, C)).astype(np.uint8))
    vals *= rng.choice([-1.0, 1.0], (R, C))
    i = np.arange(R)[:, None] % 32
    j = np.arange(C)[None, :] % 32
    vals = np.where(i == j, 448.0 * rng.choice([-1.0, 1.0], (R, C)), vals)
    return (vals * 2.0 ** -9).astype(F32)       # one global power of two: still exact


def test_fp8_baseline_exact_reduces_to_matmul():
    rng = np.random.default_rng(31)
    M, N, K = 96, 160, 224
    X = _exact_fp8_tensor(rng, M, K)
    W = _exact_fp8_tensor(rng, N, K)
    dY = _exact_fp8_tensor(rng, M, N)
    X64, W64, dY64 = (a.astype(np.float64) for a in (X, W, dY))
    Y, _, _ = Lin.fp8_forward(X, W)
    dX, _, _ = Lin.fp8_bwd_dx(dY, W)
    dW, _, _ = Lin.fp8_bwd_dw(dY, X)
    assert np.array_equal(Y, X64 @ W64.T)
    assert np.array_equal(dX, dY64 @ W64)
    assert np.array_equal(dW, dY64.T @ X64)


def test_fp8_baseline_error_bound():
    rng = np.random.default_rng(32)
    M, N, K = 64, 96, 200
    X = (rng.standard_normal((M, K)) * 3).astype(F32)
    W = (rng.standard_normal((N, K)) * 0.02).astype(F32)
    Y, _, _ = Lin.fp8_forward(X, W)
    ref = X.astype(np.float64) @ W.astype(np.float64).T
    mag = np.abs(X.astype(np.float64)) @ np.abs(W.astype(np.float64)).T
    # each E4M3 operand is within 2^-4 relative (normal range) of its input, plus the
    # absolute step of the block's subnormals
    assert np.all(np.abs(Y - ref) <= mag * (2 * 2.0 ** -4 + 2.0 ** -8) + 1e-6)
