"""Pins for the oracle's OsciReset and OutControl calibration.

OsciReset (technical summary §2.B) is pinned by closed-form trajectories:
  * the pages' own example (golden fixture): a weight alternating around the
    midpoint 0.25 of the bins 0 and 0.5 has risk = step / (2 delta) and is
    reset at the first step whose learning rate is below the threshold;
  * a weight drifting monotonically away from a grid point never reaches
    risk 4 (each bin change needs at least half a bin of travel);
  * a reset puts the master weight exactly on Q-hat and zeroes its distances;
  * a reset leaves the quantization unchanged: re-quantizing after resetting 1%,
    50% or all of the weights, or exactly the group and block maxima, of random
    and adversarial rows gives the same values, scales and codes (RTN is
    idempotent), and a planted rounding slip makes this pin fail.
Calibration (§2.C) is pinned by planted heavy channels, a full-sort brute
force with the tie rule, and exact integer sums.
"""
import os

import numpy as np
import pytest

from oracle import calib as C
from oracle import osci as O

F32 = np.float32


def _fixture(golden_dir):
    vals = {}
    with open(os.path.join(golden_dir, "oscillation_example.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, *v = line.split()
                vals[k] = [float(t) for t in v]
    return vals


def _row_with_grid_step_half(centre):
    """One 128-wide row whose outer block and the tracked element's 16-block both
    reach 6, so the tracked element sees the grid {0, 0.5, 1, ...} (scale ~1)."""
    w = np.zeros((1, 128), dtype=F32)
    w[0, 1:] = 0.013
    w[0, 0] = 6.0
    w[0, 65] = 6.0
    w[0, 64] = centre
    return w


def test_pages_oscillation_example_resets_on_schedule(golden_dir):
    fx = _fixture(golden_dir)
    centre, delta = fx["centre"][0], fx["delta"][0]
    w = _row_with_grid_step_half(centre - delta)        # tracking starts on the low side
    state = O.init_state(w)
    resets = []
    for t, lr in enumerate(fx["lr_schedule"]):
        w = w.copy()
        w[0, 64] = F32(centre + delta * (1 if t % 2 == 0 else -1))
        qh, _ = O.qhat_f32(w)
        assert qh[0, 64] in (np.float32(fx["grid_low"][0]), O.qhat_f32(_row_with_grid_step_half(0.5))[0][0, 64])
        w, state, mask, _ = O.osci_reset_step(w, state, lr, fx["lr_threshold"][0], fx["risk_threshold"][0])
        if not mask[0, 64]:
            risk = state["dist_q"][0, 64] / state["dist_m"][0, 64]
            assert abs(risk - fx["risk_per_step"][0]) < 0.01 * fx["risk_per_step"][0]
        else:
            resets.append(t)
            assert w[0, 64] == qh[0, 64]                      # moved onto the bin centre
            assert state["dist_q"][0, 64] == 0 and state["dist_m"][0, 64] == 0
            break
        assert not mask[0, :64].any() and not mask[0, 65:].any()  # only the tracked element
    assert resets == [int(fx["first_reset_step"][0])]


def test_monotone_drift_from_grid_point_never_resets():
    w = _row_with_grid_step_half(0.5)
    state = O.init_state(w)
    for t in range(400):
        w = w.copy()
        w[0, 64] = F32(0.5 + 0.004 * (t + 1))                 # drifts across several bins
        w, state, mask, _ = O.osci_reset_step(w, state, 1e-5, 1e-4, 4.0)
        assert not mask.any()
    assert state["dist_q"][0, 64] > 0                         # it did change bins


def test_reset_condition_and_state_update():
    rng = np.random.default_rng(0)
    w0 = (rng.standard_normal((8, 256)) * 0.02).astype(F32)
    state = O.init_state(w0)
    w = w0
    for t in range(30):
        w = (w + rng.standard_normal(w.shape).astype(F32) * F32(3e-4)).astype(F32)
        lr = 1e-3 if t < 20 else 5e-5
        pre = state
        w_new, state, mask, q = O.osci_reset_step(w, state, lr, 1e-4, 4.0)
        dist_m = (pre["dist_m"] + np.abs(w - pre["w_prev"])).astype(F32)
        qh, _ = O.qhat_f32(w)
        dist_q = (pre["dist_q"] + np.abs(qh - pre["qhat_prev"])).astype(F32)
        expect = (lr < 1e-4) & (dist_m > 0) & (dist_q > F32(4.0) * dist_m)
        assert np.array_equal(mask, expect)
        assert np.array_equal(w_new[mask], qh[mask]) and np.array_equal(w_new[~mask], w[~mask])
        assert np.all(state["dist_q"][mask] == 0)
        if t < 20:
            assert not mask.any()
        w = w_new
    assert state["dist_m"].max() > 0


# ---------------------------------------------------------------------------
# A reset lands the master weight on the centre of its current bin (technical summary
# §2.B), so it must not move the weight's quantized value, nor that of any other weight
# of its block: re-quantizing after any set of resets gives the same quantization.
# ---------------------------------------------------------------------------
def _requantize_after_reset(x, mask):
    """Quantize x, move the masked elements onto their Q-hat, quantize again."""
    qh, (c, s, o) = O.qhat_f32(x)
    x2 = np.where(mask, qh, x).astype(F32)
    qh2, (c2, s2, o2) = O.qhat_f32(x2)
    return (qh, c, s, o), (qh2, c2, s2, o2), x2


def _reset_invariance_failures(x, mask):
    """Counts of everything a reset changed.  Byte for byte: the outer scales; the inner
    scale byte of every group holding a nonzero quantized value; every code, once a
    magnitude-0 code's sign bit is cleared (a reset element whose Q-hat is -0 becomes
    the weight -0, which quantizes as code 0).  The only other byte that may move is the
    scale of a group every element of which dequantizes to zero before and after: a
    group whose elements were all reset to zero has amax 0 and scale byte 0."""
    (qh, c, s, o), (qh2, c2, s2, o2), x2 = _requantize_after_reset(x, mask)
    R, L = x.shape
    zero_grp = (qh.reshape(R, -1, 16) == 0).all(axis=2) if L % 16 == 0 else None
    live = ~zero_grp if zero_grp is not None else np.ones(s.shape, bool)[:, : L // 16]
    strip = lambda cc: np.where((cc & 7) == 0, 0, cc)
    return {
        "values": int((qh2 != qh).sum()),
        "outer": int((o2.view(np.uint32) != o.view(np.uint32)).sum()),
        "inner": int((s2[:, : L // 16] != s[:, : L // 16])[live].sum()),
        "codes": int((strip(c2) != strip(c)).sum()),
        "landed": int((x2[mask] != qh[mask]).sum()),
    }


def _adversarial_rows(rng, R=256, L=1024):
    """Rows built to sit on the scale rules' edges: group amaxima spread over 40 binades
    below their block's maximum (tiny groups get the smallest normal scale), maxima
    placed exactly on and one ulp around the top value 6 sigma s_o of a scale, ties of
    the E2M1 grid, repeated block maxima, and signed values that round to -0."""
    x = rng.standard_normal((R, L)).astype(F32)
    g = np.exp2(-rng.integers(0, 40, (R, L // 16))).astype(F32)
    x = (x.reshape(R, -1, 16) * g[:, :, None]).reshape(R, L).astype(F32)
    qh, (c, s, o) = O.qhat_f32(x)
    from oracle import formats as Fm
    for r in range(0, R, 4):                       # group maxima on a scale's top value
        b, j = rng.integers(0, L // 128), rng.integers(0, 8)
        sig = float(Fm.e4m3_decode(np.uint8(rng.integers(0x08, 0x7E))))
        top = F32(F32(6.0 * sig) * o[r, b])
        seg = slice(b * 128 + j * 16, b * 128 + j * 16 + 16)
        x[r, seg] = (x[r, seg] / np.abs(x[r, seg]).max() * top * F32(0.9)).astype(F32)
        x[r, b * 128 + j * 16] = [top, np.nextafter(top, F32(0)), np.nextafter(top, F32(np.inf))][r % 3]
    for r in range(1, R, 4):                       # E2M1 ties and a repeated block maximum
        x[r, :128] = (np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0] * 16, F32) * F32(2.0 ** -5))
        x[r, 127] = F32(6.0 * 2.0 ** -5)
    x[2::4, 5::7] = -1e-30                         # negatives that quantize to -0
    return x


@pytest.mark.parametrize("frac", [0.01, 0.5, 1.0])
def test_reset_keeps_quantization_random_weights(frac):
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((512, 1024)) * 0.02).astype(F32)
    fails = _reset_invariance_failures(x, rng.random(x.shape) < frac)
    assert fails == dict.fromkeys(fails, 0), fails


@pytest.mark.parametrize("frac", [0.01, 0.5, 1.0])
def test_reset_keeps_quantization_adversarial_rows(frac):
    rng = np.random.default_rng(12)
    x = _adversarial_rows(rng)
    fails = _reset_invariance_failures(x, rng.random(x.shape) < frac)
    assert fails == dict.fromkeys(fails, 0), fails


def test_reset_of_group_and_block_maxima():
    """Resetting exactly the elements that set the scales: every group maximum, and
    every block maximum."""
    rng = np.random.default_rng(13)
    for x in ((rng.standard_normal((256, 1024)) * 0.02).astype(F32), _adversarial_rows(rng)):
        ax = np.abs(x).reshape(x.shape[0], -1, 16)
        gmax = (ax == ax.max(axis=2, keepdims=True)).reshape(x.shape)
        bx = np.abs(x).reshape(x.shape[0], -1, 128)
        bmax = (bx == bx.max(axis=2, keepdims=True)).reshape(x.shape)
        for mask in (gmax, bmax):
            fails = _reset_invariance_failures(x, mask)
            assert fails == dict.fromkeys(fails, 0), fails


def test_rtn_is_idempotent():
    """Q(Q-hat(x)) = Q(x): a fully dequantized tensor quantizes back to itself (values,
    outer scales, codes up to the sign of zero, and the scale of every live group)."""
    rng = np.random.default_rng(14)
    for x in ((rng.standard_normal((128, 1152)) * rng.uniform(1e-3, 1e3)).astype(F32), _adversarial_rows(rng, 64)):
        fails = _reset_invariance_failures(x, np.ones(x.shape, bool))
        assert fails == dict.fromkeys(fails, 0), fails


def test_osci_reset_step_leaves_q_unchanged():
    """Through OsciReset itself: weights oscillating across bin boundaries at a low
    learning rate get reset, and the reset weights quantize to the Q the step emitted."""
    rng = np.random.default_rng(15)
    w = (rng.standard_normal((64, 512)) * 0.02).astype(F32)
    state = O.init_state(w)
    resets = 0
    for t in range(12):
        kick = (rng.standard_normal(w.shape) * 2e-3 * (1 if t % 2 == 0 else -1)).astype(F32)
        w = (w + kick).astype(F32)
        w, state, mask, q = O.osci_reset_step(w, state, 5e-5, 1e-4, 4.0)
        resets += int(mask.sum())
        _, (c2, s2, o2) = O.qhat_f32(w)
        strip = lambda cc: np.where((cc & 7) == 0, 0, cc)
        assert np.array_equal(strip(c2), strip(q[0])) and np.array_equal(s2, q[1])
        assert np.array_equal(o2, q[2])
    assert resets > 100


def test_planted_ratio_ceiling_breaks_reset_invariance(monkeypatch):
    """The pin above catches the rounding slip it was written for: deciding the inner
    scale as the E4M3 ceiling of the fp32 quotient a_i / (6 s_o) (subnormal scales
    allowed) lets a reset group maximum bump its scale one step and re-quantize its
    neighbours.  Planted in the oracle, on the CPU."""
    from oracle import formats as Fm
    from oracle import quant as Qm
    pos = np.arange(0, 0x7F, dtype=np.uint8)
    vals = Fm.e4m3_decode(pos)

    def ratio_ceiling(a_i, s_o):
        m = (np.asarray(s_o, F32) * F32(6.0)).astype(F32)
        with np.errstate(divide="ignore", invalid="ignore"):
            t = np.where(a_i > 0, (a_i / np.where(m > 0, m, F32(1))).astype(F32), F32(0))
        idx = np.minimum(np.searchsorted(vals, t.astype(np.float64), side="left"), len(pos) - 1)
        return np.where(a_i > 0, pos[idx], 0).astype(np.uint8)

    monkeypatch.setattr(Qm, "e4m3_inner_scale_byte", ratio_ceiling)
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((512, 1024)) * 0.02).astype(F32)
    fails = _reset_invariance_failures(x, rng.random(x.shape) < 0.01)
    assert fails["values"] > 0 and fails["inner"] > 0


def test_calibration_planted_channels_and_brute_force():
    rng = np.random.default_rng(1)
    M, K = 300, 96
    heavy = np.sort(rng.choice(K, 6, replace=False))
    s = np.zeros(K)
    for b in range(3):
        x = rng.standard_normal((M, K)).astype(F32)
        x[:, heavy] *= 40
        s = C.accumulate_sumsq(x, s)
    k = C.outlier_count(K, 10)
    assert k == 10
    out, normal = C.top_k_channels(s, k)
    assert set(heavy) <= set(out)
    assert np.array_equal(np.sort(np.concatenate([out, normal])), np.arange(K))
    ref = np.sort(np.argsort(-s, kind="stable")[:k])      # library sort, stable = lower index first
    assert np.array_equal(out, ref)


def test_calibration_ties_and_exact_sums():
    x = np.zeros((260, 8), dtype=F32)
    x[:, 2] = 3.0
    x[:, 5] = 3.0
    x[:, 6] = -3.0
    s = C.accumulate_sumsq(x, np.zeros(8))
    assert np.array_equal(s, np.array([0, 0, 2340, 0, 0, 2340, 2340, 0], dtype=np.float64))
    out, _ = C.top_k_channels(s, 2)
    assert list(out) == [2, 5]                               # ties -> lower channel index
    assert C.outlier_count(1024, 10) == 103 and C.outlier_count(4096, 10) == 410


# ---------------------------------------------------------------------------
# AdamW step of the fused training-step pass, pinned against closed forms and against
# torch.optim.AdamW (an independent implementation whose rounding order differs, so it
# agrees within a few fp32 ulp).
# ---------------------------------------------------------------------------
def test_adamw_first_step_closed_form():
    """Step 1 without weight decay: m-hat = g and v-hat = g^2, so w moves by
    lr * g / (|g| + eps), i.e. by about lr against the sign of g."""
    rng = np.random.default_rng(4)
    w = (rng.standard_normal((4, 64)) * 0.02).astype(F32)
    g = (rng.standard_normal((4, 64)) * 1e-2).astype(F32)
    z = np.zeros_like(w)
    lr, eps = 1e-3, 1e-8
    w1, m1, v1 = O.adamw_step(w, g, z, z, lr, 0.9, 0.95, eps, 0.0, 1)
    # from m = 0 the first moment is exactly (1 - beta1) g, beta1 being the fp32 argument
    assert np.array_equal(m1, (F32(1.0 - float(F32(0.9))) * g).astype(F32))
    exact = w.astype(np.float64) - lr * g.astype(np.float64) / (np.abs(g.astype(np.float64)) + eps)
    assert np.allclose(w1, exact, rtol=0, atol=4e-9)


def test_adamw_weight_decay_alone_is_one_product():
    """A zero gradient leaves m = v = 0 and the update is exactly w * fp32(1 - lr wd)."""
    w = (np.random.default_rng(5).standard_normal((2, 128)) * 0.02).astype(F32)
    z = np.zeros_like(w)
    w1, m1, v1 = O.adamw_step(w, z, z, z, 1e-3, 0.9, 0.95, 1e-8, 0.1, 7)
    assert not m1.any() and not v1.any()
    assert np.array_equal(w1, (w * F32(1.0 - 1e-3 * 0.1)).astype(F32))


def test_adamw_matches_torch_optim_adamw():
    torch = __import__("torch")
    rng = np.random.default_rng(6)
    w = (rng.standard_normal((8, 96)) * 0.02).astype(F32)
    m = np.zeros_like(w)
    v = np.zeros_like(w)
    p = torch.nn.Parameter(torch.from_numpy(w.copy()))
    opt = torch.optim.AdamW([p], lr=1e-3, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1, foreach=False)
    for t in range(1, 9):
        g = (rng.standard_normal(w.shape) * 1e-2).astype(F32)
        w, m, v = O.adamw_step(w, g, m, v, 1e-3, 0.9, 0.95, 1e-8, 0.1, t)
        p.grad = torch.from_numpy(g.copy())
        opt.step()
        st = opt.state[p]
        assert np.allclose(w, p.detach().numpy(), rtol=1e-6, atol=1e-9), t
        mt, vt = st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()
        # m can cancel to near zero, where the two rounding orders differ most in relative terms
        assert np.allclose(m, mt, rtol=1e-5, atol=1e-6 * float(np.abs(mt).max())), t
        assert np.allclose(v, vt, rtol=1e-5, atol=0), t
