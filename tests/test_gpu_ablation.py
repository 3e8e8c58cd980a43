"""GPU run of the ablation harness (small sweep) through the library: the table is
written and shows what the components must do on the synthetic tensors."""
import json

import pytest

pytestmark = pytest.mark.gpu


def test_small_ablation_sweep(tmp_path):
    from nvfp4_bit_fully_gb300 import ablation as A

    out = tmp_path / "ablation.json"
    table = A.run(str(out), small=True)
    assert json.loads(out.read_text())["osci_reset"] == table["osci_reset"]
    osci = {r["config"]: r for r in table["osci_reset"]}
    assert osci["off"]["resets"] == 0
    # a higher reset threshold never resets more weights
    rs = [osci["r=%g" % r]["resets"] for r in A.OSCI_THRESHOLDS]
    assert all(a >= b for a, b in zip(rs, rs[1:])) and rs[0] > 0
    # resetting oscillating weights leaves fewer flips of the quantized weights
    assert osci["r=4"]["flip_rate"] <= osci["off"]["flip_rate"]
    oc = {r["outlier_pct"]: r for r in table["outcontrol"]}
    # FP8 outlier channels lower the forward error on activations with heavy channels
    assert oc[10]["fwd_rel_err"] < oc[0]["fwd_rel_err"]
    for r in table["outcontrol"]:
        # unbiased backward estimates: the mean over seeds is closer than one seed
        assert r["dx"]["bias"] < 0.8 * r["dx"]["per_seed"] and r["dw"]["bias"] < 0.8 * r["dw"]["per_seed"]


def test_slice_format_ablation(tmp_path):
    """The FP6 x FP4 slices run through the layer; the FP8 slice, with three mantissa bits on
    both sides, gives the smallest slice error."""
    import torch

    from nvfp4_bit_fully_gb300 import ablation as A
    from nvfp4_bit_fully_gb300 import tj

    tj.load()
    rows = A.run_slice_formats(tj, torch, 256, 256, 512, 10, 4, 13)
    errs = {r["slice"]: r["slice_fwd_rel_err"] for r in rows}
    assert set(errs) == {n for n, _, _ in A.SLICE_FORMATS}
    assert all(0 < e < 1 for e in errs.values())
    assert errs["e4m3 x e4m3"] == min(errs.values())
    sizes = {r["slice"]: r["slice_code_bytes"] for r in rows}
    assert sizes["e2m3 x e2m1"] < sizes["e4m3 x e4m3"]
