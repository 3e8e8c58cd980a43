"""GPU parity: OsciReset and OutControl calibration, bit for bit.

OsciReset: several steps of a synthetic trajectory whose learning rate crosses
the threshold; every piece of state (master weight, w_prev, dist_Q, dist_M, the
emitted forward NVFP4 weight, the reset mask) must equal the oracle's exactly.
Calibration: fixed-order fp64 sums of squares over ragged batches, and the
top-k selection with its tie rule.
"""
import numpy as np
import pytest
import torch

from layouts import assert_nvfp4_equal
from oracle import calib as OC
from oracle import osci as OO
from oracle import quant as Q

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tj():
    from nvfp4_bit_fully_gb300 import tj as _tj

    _tj.load()
    return _tj


def _mask_bits(mask_words, rows, cols):
    w = mask_words.cpu().numpy().view(np.uint32).reshape(rows, -1)
    bits = (w[:, :, None] >> np.arange(32, dtype=np.uint32)) & 1
    return bits.reshape(rows, -1)[:, :cols].astype(bool)


# the odd column counts take the kernel's scalar path (rows not 16-byte aligned) and leave a
# ragged last mask word and a ragged last 128-element block
ODD_SHAPES = [(1, 1), (3, 130), (129, 33), (50, 517)]


@pytest.mark.parametrize("rows,cols", [(64, 256), (100, 200)] + ODD_SHAPES)
def test_osci_reset_trajectory_bit_exact(tj, rows, cols):
    rng = np.random.default_rng(rows + cols)
    w0 = (rng.standard_normal((rows, cols)) * 0.02).astype(np.float32)
    # make some elements oscillate around bin midpoints: alternate +-d
    osc = rng.random((rows, cols)) < 0.05
    state = OO.init_state(w0)
    w_dev = torch.from_numpy(w0.copy()).cuda()
    w_prev = w_dev.clone()
    dq = torch.zeros_like(w_dev)
    dm = torch.zeros_like(w_dev)
    q_prev = tj.quantize_nvfp4(w_dev)
    q_out = tj.NVFP4.empty(rows, cols)
    mask = torch.empty(rows * ((cols + 31) // 32), dtype=torch.int32, device="cuda")
    w = w0
    lrs = [1e-3, 8e-4, 5e-4, 2e-4, 9e-5, 5e-5, 2e-5, 1e-5]
    for t, lr in enumerate(lrs):
        step = (rng.standard_normal((rows, cols)) * lr).astype(np.float32)
        step = np.where(osc, np.float32(3e-4 * (1 if t % 2 == 0 else -1)), step).astype(np.float32)
        w = (w + step).astype(np.float32)
        w_dev.copy_(torch.from_numpy(w))
        w, state, m_ref, q_ref = OO.osci_reset_step(w, state, lr, 1e-4, 4.0)
        tj.osci_reset(w_dev, w_prev, dq, dm, q_prev, q_out, mask, lr, 1e-4, 4.0)
        torch.cuda.synchronize()
        assert np.array_equal(w_dev.cpu().numpy(), w), t
        assert np.array_equal(w_prev.cpu().numpy(), state["w_prev"]), t
        assert np.array_equal(dq.cpu().numpy(), state["dist_q"]), t
        assert np.array_equal(dm.cpu().numpy(), state["dist_m"]), t
        assert np.array_equal(_mask_bits(mask, rows, cols), m_ref), t
        assert_nvfp4_equal(q_out, q_ref, "Q step %d" % t)
        q_prev, q_out = q_out, q_prev
    assert state["dist_m"].max() > 0


@pytest.mark.parametrize("rows,cols", [(64, 256), (37, 200)] + ODD_SHAPES)
def test_adamw_osci_reset_trajectory_bit_exact(tj, rows, cols):
    """The fused training-step pass (AdamW, then OsciReset of the updated weights) equals the
    oracle's AdamW step followed by its OsciReset step, bit for bit, over a schedule whose
    learning rate falls below the threshold; a low risk threshold makes resets happen."""
    rng = np.random.default_rng(3 * rows + cols)
    w0 = (rng.standard_normal((rows, cols)) * 0.02).astype(np.float32)
    state = OO.init_state(w0)
    m = np.zeros_like(w0)
    v = np.zeros_like(w0)
    w_dev = torch.from_numpy(w0.copy()).cuda()
    m_dev, v_dev = torch.zeros_like(w_dev), torch.zeros_like(w_dev)
    w_prev = w_dev.clone()
    dq = torch.zeros_like(w_dev)
    dm = torch.zeros_like(w_dev)
    q_prev = tj.quantize_nvfp4(w_dev)
    q_out = tj.NVFP4.empty(rows, cols)
    mask = torch.empty(rows * ((cols + 31) // 32), dtype=torch.int32, device="cuda")
    w = w0
    osc = rng.random((rows, cols)) < 0.2
    lrs = [1e-3, 5e-4, 2e-4, 9e-5, 5e-5, 2e-5, 1e-5, 1e-5]
    resets = 0
    for t, lr in enumerate(lrs, start=1):
        g = (rng.standard_normal((rows, cols)) * 1e-2).astype(np.float32)
        g = np.where(osc, np.float32(0.05 * (1 if t % 2 else -1)), g).astype(np.float32)
        w, m, v, state, m_ref, q_ref = OO.adamw_osci_reset_step(w, g, m, v, state, lr, 0.9, 0.95, 1e-8, 0.1, t,
                                                                 1e-4, 0.5)
        tj.adamw_osci_reset(w_dev, torch.from_numpy(g).cuda(), m_dev, v_dev, w_prev, dq, dm, q_prev, q_out, mask,
                            lr, 0.9, 0.95, 1e-8, 0.1, t, 1e-4, 0.5)
        torch.cuda.synchronize()
        assert np.array_equal(w_dev.cpu().numpy(), w), t
        assert np.array_equal(m_dev.cpu().numpy(), m), t
        assert np.array_equal(v_dev.cpu().numpy(), v), t
        assert np.array_equal(w_prev.cpu().numpy(), state["w_prev"]), t
        assert np.array_equal(dq.cpu().numpy(), state["dist_q"]), t
        assert np.array_equal(dm.cpu().numpy(), state["dist_m"]), t
        assert np.array_equal(_mask_bits(mask, rows, cols), m_ref), t
        assert_nvfp4_equal(q_out, q_ref, "Q step %d" % t)
        resets += int(m_ref.sum())
        q_prev, q_out = q_out, q_prev
    if rows * cols >= 1024:                   # enough weights for some of them to oscillate
        assert resets > 0


def test_osci_reset_in_place_q(tj):
    """q_out may be the same tensor as q_prev: it then holds Q of the new weights."""
    rows, cols = 32, 128
    w = torch.randn(rows, cols, device="cuda") * 0.02
    q = tj.quantize_nvfp4(w)
    w_prev = w.clone()
    w2 = w + 1e-4
    w2_before = w2.cpu().numpy().copy()
    dq = torch.zeros_like(w)
    dm = torch.zeros_like(w)
    mask = torch.empty(rows * 4, dtype=torch.int32, device="cuda")
    tj.osci_reset(w2, w_prev, dq, dm, q, q, mask, 1e-5, 1e-4, 4.0)
    torch.cuda.synchronize()
    assert_nvfp4_equal(q, Q.quantize_nvfp4(w2_before, 0), "in-place Q")


def test_osci_reset_keeps_q_on_the_gpu(tj):
    """A reset moves a weight onto its bin centre without moving its quantized value
    (§2.B): after a pass that resets many weights, the GPU quantizer applied to the
    reset weights gives back the Q the pass emitted (codes up to the sign of zero),
    and both equal the oracle's quantization of the pre-reset weights."""
    rows, cols = 256, 1024
    rng = np.random.default_rng(77)
    w0 = (rng.standard_normal((rows, cols)) * 0.02).astype(np.float32)
    w1 = (w0 + rng.standard_normal((rows, cols)).astype(np.float32) * np.float32(2e-3)).astype(np.float32)
    w_dev = torch.from_numpy(w1.copy()).cuda()
    w_prev = torch.from_numpy(w0.copy()).cuda()
    dq = torch.zeros_like(w_dev)
    dm = torch.zeros_like(w_dev)
    q_prev = tj.quantize_nvfp4(w_prev)
    q_out = tj.NVFP4.empty(rows, cols)
    mask = torch.empty(rows * (cols // 32), dtype=torch.int32, device="cuda")
    # risk threshold 0.5 and lr below the threshold: a large share of the weights reset
    tj.osci_reset(w_dev, w_prev, dq, dm, q_prev, q_out, mask, 1e-5, 1e-4, 0.5)
    q_again = tj.quantize_nvfp4(w_dev)
    torch.cuda.synchronize()
    m = _mask_bits(mask, rows, cols)
    assert m.sum() > rows * cols // 100
    ref = Q.quantize_nvfp4(w1, 0)
    assert_nvfp4_equal(q_out, ref, "Q of the pass")
    from layouts import nvfp4_to_logical
    a, b = nvfp4_to_logical(q_again), nvfp4_to_logical(q_out)
    strip = lambda c: np.where((c & 7) == 0, 0, c)
    assert np.array_equal(strip(a[0]), strip(b[0])), "codes moved by a reset"
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2]), "scales moved by a reset"
    qh = Q.dequantize_nvfp4_f32(*ref)
    assert np.array_equal(w_dev.cpu().numpy()[m], qh[m])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_calibration_bit_exact(tj, dtype):
    g = torch.Generator().manual_seed(5)
    K = 300
    heavy = torch.randperm(K, generator=g)[:12]
    sumsq = torch.zeros(K, dtype=torch.float64, device="cuda")
    s_ref = np.zeros(K)
    for b, M in enumerate((1000, 300, 4096)):
        x = torch.randn(M, K, generator=g)
        x[:, heavy] *= 40
        x = x.to(dtype)
        tj.outlier_calibrate(x.cuda(), sumsq)
        s_ref = OC.accumulate_sumsq(x.float().numpy(), s_ref)
    k = OC.outlier_count(K, 10)
    outl, normal = tj.outlier_calibrate(None, sumsq, finalize=True, k=k)
    torch.cuda.synchronize()
    assert np.array_equal(sumsq.cpu().numpy(), s_ref)
    o_ref, n_ref = OC.top_k_channels(s_ref, k)
    assert np.array_equal(outl.cpu().numpy(), o_ref)
    assert np.array_equal(normal.cpu().numpy(), n_ref)
    assert set(heavy.numpy()) <= set(o_ref)


def test_calibration_ties(tj):
    s = torch.tensor([5.0, 7.0, 7.0, 1.0, 7.0, 0.0], dtype=torch.float64, device="cuda")
    outl, normal = tj.outlier_calibrate(None, s, finalize=True, k=2)
    torch.cuda.synchronize()
    assert outl.cpu().tolist() == [1, 2] and normal.cpu().tolist() == [0, 3, 4, 5]
