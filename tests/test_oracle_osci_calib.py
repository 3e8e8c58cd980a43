"""Pins for the oracle's OsciReset and OutControl calibration.

OsciReset (technical summary §2.B) is pinned by closed-form trajectories:
  * the pages' own example (golden fixture): a weight alternating around the
    midpoint 0.25 of the bins 0 and 0.5 has risk = step / (2 delta) and is
    reset at the first step whose learning rate is below the threshold;
  * a weight drifting monotonically away from a grid point never reaches
    risk 4 (each bin change needs at least half a bin of travel);
  * a reset puts the master weight exactly on Q-hat and zeroes its distances.
Calibration (§2.C) is pinned by planted heavy channels, a full-sort brute
force with the tie rule, and exact integer sums.
"""
import os

import numpy as np

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
