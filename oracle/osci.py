"""OsciReset: oscillation tracking and reset of master weights.

Test infrastructure only (see the package docstring).

TetraJet-v2 technical summary §2.B: follow each weight's optimisation
trajectory; the oscillation risk is dist_Q / dist_M, the distance travelled by
the quantized weight over the distance travelled by the master weight.  When
the learning rate is low and the risk exceeds a threshold, the master weight
of the oscillating element is set to the centre of its current quantization
bin.

Readings:
  * distances are cumulative L1 path lengths in fp32, summed step by step
    from the start of tracking and zeroed on a reset;
  * Q-hat is the fp32 dequantized RTN double-block quantization of the master
    weight, rows quantized along their length (the forward weight layout,
    without an outlier split);
  * "bin centre" is the grid point itself, i.e. Q-hat.  The quantizer decides
    its scales on dequantized values (quant / formats.e4m3_inner_scale_byte),
    so it is idempotent: a weight moved onto its Q-hat quantizes to the same
    code and scales, and so do the other weights of its block;
  * reset  <=>  track and lr < lr_thr and dist_M > 0 and dist_Q > r * dist_M
    (fp32 product); 0/0 never resets;
  * after the step, w_prev <- w and Q-hat_prev <- Q-hat.
"""
import numpy as np

from . import quant as Q

F32 = np.float32


def qhat_f32(w):
    """fp32 Q-hat of a master weight matrix [rows, cols] (cols padded to 128 internally)."""
    w = np.asarray(w, dtype=F32)
    c, s, o = Q.quantize_nvfp4(w, Q.RTN)
    return Q.dequantize_nvfp4_f32(c, s, o)[:, : w.shape[1]], (c, s, o)


def init_state(w0):
    """State at the start of tracking: w_prev = w0, Q-hat_prev = Q-hat(w0), distances 0."""
    w0 = np.asarray(w0, dtype=F32)
    qh, _ = qhat_f32(w0)
    z = np.zeros_like(w0)
    return {"w_prev": w0.copy(), "qhat_prev": qh, "dist_q": z.copy(), "dist_m": z.copy()}


def osci_reset_step(w, state, lr, lr_thr, risk_thr, track=True):
    """One OsciReset pass after an optimizer step.  Returns (w_new, state_new, mask, q).

    q is the RTN double-block quantization (codes, sf, outer) of the
    pre-reset w, i.e. the next forward's weight operand.
    """
    w = np.asarray(w, dtype=F32)
    dist_m = (state["dist_m"] + np.abs((w - state["w_prev"]).astype(F32))).astype(F32)
    qh, q = qhat_f32(w)
    dist_q = (state["dist_q"] + np.abs((qh - state["qhat_prev"]).astype(F32))).astype(F32)
    lr_low = bool(np.float32(lr) < np.float32(lr_thr))
    risky = (dist_m > 0) & (dist_q > (F32(risk_thr) * dist_m).astype(F32))
    mask = risky & bool(track) & lr_low
    w_new = np.where(mask, qh, w).astype(F32)
    dist_q = np.where(mask, F32(0.0), dist_q).astype(F32)
    dist_m = np.where(mask, F32(0.0), dist_m).astype(F32)
    new_state = {"w_prev": w_new.copy(), "qhat_prev": qh, "dist_q": dist_q, "dist_m": dist_m}
    return w_new, new_state, mask, q


# ---------------------------------------------------------------------------
# Training-step fusion around OsciReset: the optimizer update that precedes the pass.
# The pages apply OsciReset to the master weights after the optimizer step and name no
# optimizer; this follows AdamW (Loshchilov & Hutter, decoupled weight decay), the usual
# choice for the OLMo-2-class models the pages train, in the form
#     m <- beta1 m + (1 - beta1) g
#     v <- beta2 v + (1 - beta2) g g
#     w <- w (1 - lr wd) - (lr / (1 - beta1^t)) * m / (sqrt(v) / sqrt(1 - beta2^t) + eps)
# with every operation an fp32 round-to-nearest step in exactly this order (products
# before sums, no fused multiply-add), and the per-step constants formed in double
# precision and rounded once to fp32.
# ---------------------------------------------------------------------------
def adamw_constants(lr, beta1, beta2, eps, weight_decay, step):
    """The fp32 constants of one AdamW step t = step >= 1.  The hyperparameters are fp32
    values (as the C ABI takes them); each constant is formed from them in double precision
    and rounded once to fp32."""
    t = int(step)
    lr, b1, b2, wd = (float(F32(a)) for a in (lr, beta1, beta2, weight_decay))
    return {
        "b1": F32(b1), "b2": F32(b2), "om1": F32(1.0 - b1), "om2": F32(1.0 - b2),
        "decay": F32(1.0 - lr * wd), "step_size": F32(lr / (1.0 - b1 ** t)),
        "bc2": F32(np.sqrt(1.0 - b2 ** t)), "eps": F32(eps),
    }


def adamw_step(w, g, m, v, lr, beta1, beta2, eps, weight_decay, step):
    """One AdamW update in fp32.  Returns (w_new, m_new, v_new)."""
    c = adamw_constants(lr, beta1, beta2, eps, weight_decay, step)
    w, g, m, v = (np.asarray(a, dtype=F32) for a in (w, g, m, v))
    m1 = (c["b1"] * m).astype(F32) + (c["om1"] * g).astype(F32)
    m1 = m1.astype(F32)
    gg = (g * g).astype(F32)
    v1 = ((c["b2"] * v).astype(F32) + (c["om2"] * gg).astype(F32)).astype(F32)
    denom = ((np.sqrt(v1).astype(F32) / c["bc2"]).astype(F32) + c["eps"]).astype(F32)
    upd = (c["step_size"] * (m1 / denom).astype(F32)).astype(F32)
    w1 = ((w * c["decay"]).astype(F32) - upd).astype(F32)
    return w1, m1, v1


def adamw_osci_reset_step(w, g, m, v, state, lr, beta1, beta2, eps, weight_decay, step, lr_thr, risk_thr,
                          track=True):
    """The fused training-step pass: AdamW, then OsciReset of the updated weights (and their
    forward quantization).  Returns (w_new, m_new, v_new, state_new, mask, q)."""
    w1, m1, v1 = adamw_step(w, g, m, v, lr, beta1, beta2, eps, weight_decay, step)
    w_new, state_new, mask, q = osci_reset_step(w1, state, lr, lr_thr, risk_thr, track)
    return w_new, m1, v1, state_new, mask, q
