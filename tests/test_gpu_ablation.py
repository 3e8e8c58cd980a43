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
