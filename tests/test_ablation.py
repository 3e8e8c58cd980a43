"""CPU tests of the ablation harness's host logic (nvfp4_bit_fully_gb300.ablation):
the metrics against closed forms, the sweep grid, and the synthetic targets."""
import numpy as np

from nvfp4_bit_fully_gb300 import ablation as A


def test_rel_err_closed_forms():
    rng = np.random.default_rng(0)
    r = rng.standard_normal((8, 16))
    assert A.rel_err(r, r) == 0.0
    assert abs(A.rel_err(2 * r, r) - 1.0) < 1e-12
    assert abs(A.rel_err(r + 0.5 * r, r) - 0.5) < 1e-12
    assert A.rel_err(np.ones(3), np.zeros(3)) == np.sqrt(3)


def test_bias_and_spread_tells_unbiased_from_biased():
    rng = np.random.default_rng(1)
    ref = rng.standard_normal((32, 32))
    S = 64
    noise = rng.standard_normal((S, 32, 32))
    unb = A.bias_and_spread(ref + noise, ref)
    # unbiased: the mean's error falls like 1/sqrt(S) of one sample's
    assert abs(unb["bias"] * np.sqrt(S) / unb["per_seed"] - 1.0) < 0.1
    biased = A.bias_and_spread(1.1 * ref + noise, ref)
    assert abs(biased["bias"] - np.sqrt(0.1 ** 2 + 1.0 / S)) < 0.02
    assert unb["seeds"] == S


def test_flips_counts_changes():
    h = np.array([[0, 1], [0, 2], [1, 2], [1, 2], [0, 2]], dtype=np.float32)
    assert A.flips(h) == 3
    assert A.flips(h[:1]) == 0


def test_cosine_lr_and_sweep_grid():
    assert abs(A.cosine_lr(0, 200) - 1e-3) < 1e-15 and abs(A.cosine_lr(200, 200) - 1e-5) < 1e-15
    # the learning rate crosses the 1e-4 threshold at about step 162 of 200
    first = next(t for t in range(201) if A.cosine_lr(t, 200) < A.LR_THR)
    assert 160 <= first <= 165
    names = [c["name"] for c in A.osci_configs()]
    assert names[0] == "off" and len(names) == 1 + len(A.OSCI_THRESHOLDS) + len(A.OSCI_START_STEPS) - 1
    assert all(c["track"] for c in A.osci_configs()[1:])


def test_synthetic_targets_sit_on_bin_boundaries():
    rng = np.random.default_rng(2)
    t = A.synthetic_targets(rng, 16, 256)
    assert t.shape == (16, 256) and t.dtype == np.float32
    blk = np.abs(t.reshape(16, 2, 128))
    # the picked targets are E2M1 midpoints times one unit of their block (amax / 6)
    mids = {0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0}
    unit = blk.max(axis=2, keepdims=True) / 6.0
    ratio = blk / unit
    on_mid = np.isin(np.round(ratio * 4) / 4, list(mids)) & (np.abs(ratio - np.round(ratio * 4) / 4) < 1e-4)
    assert on_mid.mean() > 0.3


def test_unpack_codes_layout_and_zero_sign():
    # row 0: codes 1..15 then 0; byte j holds elements 2j (low nibble) and 2j + 1
    codes = np.zeros((2, 256), dtype=np.uint8)
    codes[0, :16] = np.arange(1, 17) % 16
    codes[1, 5] = 8                                      # -0: the same bin as +0
    raw = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    got = A.unpack_codes(raw.reshape(-1), 2, 200)
    assert got.shape == (2, 200)
    want = codes[:, :200].copy()
    want[1, 5] = 0
    want[0, 7] = 0                                       # code 8 = -0 in row 0 as well
    assert np.array_equal(got, want)
