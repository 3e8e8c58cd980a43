"""The oracle's pins catch plausible mistakes (CPU only).

Each case below plants one slip in the oracle's source, the kind a restatement of the
method could make: a wrong constant, a swapped comparison or sign, a transposed
operand, a dropped factor, the wrong tie rule or index.  The mutated source is executed
in place of the module (names other modules bound to its functions follow it), and the
listed pins from the oracle's own test files are run against it: at least one of them
must fail.  The module is put back afterwards.  This checks the pins, not the kernels;
nothing here touches the CUDA library.
"""
import contextlib
import importlib
import inspect
import sys
import types

import pytest

import test_oracle_formats as TF
import test_oracle_mx_formats as TM
import test_oracle_osci_calib as TO
import test_oracle_quant as TQ
import test_oracle_rht_linear as TR
from oracle import formats as F
from oracle import quant as Q


@contextlib.contextmanager
def mutant(modname, old, new):
    """Run the module `modname` with `old` replaced by `new` in its source."""
    mod = importlib.import_module(modname)
    src = inspect.getsource(mod)
    assert src.count(old) == 1, (modname, old)
    saved = dict(mod.__dict__)
    exec(compile(src.replace(old, new), mod.__file__, "exec"), mod.__dict__)
    rebound = []
    holders = [m for n, m in list(sys.modules.items())
               if m is not mod and (n.startswith("oracle") or n.startswith("test_") or n == "layouts")]
    for name, obj in saved.items():
        if isinstance(obj, types.FunctionType) and obj.__module__ == modname:
            for other in holders:
                d = other.__dict__
                for k, v in list(d.items()):
                    if v is obj:
                        d[k] = mod.__dict__[name]
                        rebound.append((d, k, obj))
    try:
        yield
    finally:
        for d, k, obj in rebound:
            d[k] = obj
        mod.__dict__.clear()
        mod.__dict__.update(saved)


def _golden():
    import os

    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# (case, module, original text, planted text, pins that must not all pass)
CASES = [
    ("outer scale from the E4M3 maximum alone", "oracle.quant",
     "s_o = (a_o / F32(6.0 * 448.0)).astype(F32)", "s_o = (a_o / F32(448.0)).astype(F32)",
     [lambda: TQ.test_codes_scales_and_error_bound(Q.RTN), TQ.test_block_maximum_takes_top_scale_and_code]),
    ("RTN ties to the odd grid point", "oracle.quant",
     "((d_hi == d_lo) & (hi % 2 == 0))", "((d_hi == d_lo) & (hi % 2 == 1))",
     [TQ.test_rtn_is_nearest_grid_point_ties_even]),
    ("SR rounds up with the complementary probability", "oracle.quant",
     "p = ((a - g_lo) / gap).astype(F32)", "p = ((g_hi - a) / gap).astype(F32)",
     [TQ.test_sr_sampled_mean_converges]),
    ("code sign bit dropped", "oracle.quant",
     "sign = np.where(xb < 0, 8, 0).astype(np.uint8)", "sign = np.where(xb < 0, 0, 0).astype(np.uint8)",
     [lambda: TQ.test_codes_scales_and_error_bound(Q.RTN), TQ.test_grid_tensors_quantize_exactly]),
    ("MX block exponent one step too high", "oracle.quant",
     "E = np.where(mant <= 0.875, ex - 9, ex - 8)", "E = np.where(mant <= 0.875, ex - 8, ex - 8)",
     [TF.test_mx_exponent_brute_force, TQ.test_mxfp8_roundtrip_and_bound]),
    ("inner scale rounded down instead of up", "oracle.formats",
     "ok = top >= a[:, None]\n        first = np.where(ok.any(axis=1), ok.argmax(axis=1), len(_INNER_BYTES) - 1)",
     "ok = top > a[:, None]\n        first = np.maximum(np.where(ok.any(axis=1), ok.argmax(axis=1), len(_INNER_BYTES)) - 1, 0)",
     [TF.test_inner_scale_against_exact_arithmetic, lambda: TQ.test_codes_scales_and_error_bound(Q.RTN)]),
    ("E4M3 exponent bias 8", "oracle.formats",
     "nor = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)",
     "nor = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 8.0)",
     [TF.test_e4m3_decode_matches_torch_all_bytes]),
    ("butterfly difference reversed", "oracle.rht",
     "y[..., i + h] = (a - b).astype(F32)", "y[..., i + h] = (b - a).astype(F32)",
     [TR.test_fwht_matches_sylvester_matrix]),
    ("RHT sign diagonal not applied", "oracle.rht",
     "return fwht128_f32((x * dd).astype(F32))", "return fwht128_f32(x)",
     [TR.test_rht_inverse_and_signs]),
    ("GEMM with a transposed operand", "oracle.linear",
     "return alpha * (a @ b.T)", "return alpha * (a.T @ b)",
     [TR.test_forward_on_grid_inputs_is_plain_matmul]),
    ("RHT normalisation 2^-6 instead of 2^-7", "oracle.linear",
     "ALPHA_RHT = 2.0 ** -7", "ALPHA_RHT = 2.0 ** -6",
     [TR.test_backward_is_unbiased_over_seeds]),
    ("dX operands transformed with different sign diagonals", "oracle.linear",
     "s_dy = sr_rht_rows(dY, seed, TAG_DY_ROW, TAG_RHT_DX)", "s_dy = sr_rht_rows(dY, seed, TAG_DY_ROW, TAG_RHT_DW)",
     [TR.test_backward_is_unbiased_over_seeds]),
    ("OsciReset risk test with the distances swapped", "oracle.osci",
     "risky = (dist_m > 0) & (dist_q > (F32(risk_thr) * dist_m).astype(F32))",
     "risky = (dist_q > 0) & (dist_m > (F32(risk_thr) * dist_q).astype(F32))",
     [lambda: TO.test_pages_oscillation_example_resets_on_schedule(_golden()), TO.test_reset_condition_and_state_update]),
    ("OsciReset resets to the previous weight", "oracle.osci",
     "w_new = np.where(mask, qh, w).astype(F32)", "w_new = np.where(mask, state[\"w_prev\"], w).astype(F32)",
     [TO.test_reset_condition_and_state_update, TO.test_osci_reset_step_leaves_q_unchanged]),
    ("calibration ties go to the higher channel", "oracle.calib",
     "key=lambda c: (-s[c], c)", "key=lambda c: (-s[c], -c)",
     [TO.test_calibration_ties_and_exact_sums]),
    ("Philox with nine rounds", "oracle.philox",
     "for rnd in range(10):", "for rnd in range(9):",
     [lambda: TF.test_philox_known_answers(_golden())]),
    ("SR uniforms always from the low half-word", "oracle.philox",
     "shift = (e & np.uint64(1)) * np.uint64(16)", "shift = (e & np.uint64(0)) * np.uint64(16)",
     [TF.test_sr_uniform16_word_mapping_and_uniformity]),
    ("AdamW without the first-moment bias correction", "oracle.osci",
     '"step_size": F32(lr / (1.0 - b1 ** t))', '"step_size": F32(lr)',
     [TO.test_adamw_first_step_closed_form, TO.test_adamw_matches_torch_optim_adamw]),
    ("outlier channels kept among the normal ones", "oracle.linear",
     "mask[np.asarray(outlier_idx, dtype=np.int64)] = False", "mask[np.asarray(outlier_idx, dtype=np.int64)] = True",
     [TR.test_forward_with_outlier_slice_on_representable_inputs]),
    ("dW slice operands not transposed", "oracle.linear",
     "dYt = np.ascontiguousarray(np.asarray(dY, dtype=F32).T)", "dYt = np.ascontiguousarray(np.asarray(dY, dtype=F32))",
     [TR.test_backward_is_unbiased_over_seeds]),
    ("dist_Q accumulates the step of the weight, not of Q-hat", "oracle.osci",
     "dist_q = (state[\"dist_q\"] + np.abs((qh - state[\"qhat_prev\"]).astype(F32))).astype(F32)",
     "dist_q = (state[\"dist_q\"] + np.abs((w - state[\"w_prev\"]).astype(F32))).astype(F32)",
     [lambda: TO.test_pages_oscillation_example_resets_on_schedule(_golden()), TO.test_reset_condition_and_state_update]),
    ("calibration sums |x| instead of x^2", "oracle.calib",
     "chunk = chunk + x[t] * x[t]", "chunk = chunk + np.abs(x[t])",
     [TO.test_calibration_ties_and_exact_sums, TO.test_calibration_planted_channels_and_brute_force]),
    ("E2M3 exponent bias 2", "oracle.formats",
     "(1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 1.0))", "(1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 2.0))",
     [lambda: TM.test_decode_matches_the_hand_tables(F.MX_E2M3)]),
    ("MX element ties away from zero", "oracle.formats",
     "((d_hi == d_lo) & ((codes[hi] & 1) == 0))", "(d_hi == d_lo)",
     [lambda: TM.test_rne_by_brute_force(F.MX_E3M2), lambda: TM.test_rne_by_brute_force(F.MX_E2M3)]),
    ("MX block scale applied the wrong way", "oracle.quant",
     "scale_inv = np.exp2(-E.astype(np.float64))\n    y = xb.astype(np.float64)",
     "scale_inv = np.exp2(E.astype(np.float64))\n    y = xb.astype(np.float64)",
     [lambda: TM.test_grid_inputs_quantize_exactly_and_the_product_is_a_matmul(F.MX_E2M3)]),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_a_planted_slip_fails_a_pin(case):
    name, modname, old, new, pins = case
    failed = []
    with mutant(modname, old, new):
        for pin in pins:
            try:
                pin()
            except (AssertionError, ValueError, IndexError, FloatingPointError) as e:
                failed.append(type(e).__name__)
    assert failed, "no pin caught: " + name


def test_the_pins_pass_on_the_oracle_itself():
    """The same pins, on the unmodified oracle (after every mutant was put back)."""
    for _, _, _, _, pins in CASES:
        for pin in pins:
            pin()
