"""CPU pin of the kernels' inner-scale recipe against the oracle's definition.

The kernels do not search all 119 candidate scales.  They take c, the E4M3 ceiling
of a first guess of the quotient a_i / fl(6 s_o) (a_i times an approximate
reciprocal, the ceiling formed from its fp32 bits), clamped to the normal bytes
0x08 .. 0x7E.  Where s_o >= 2^-110 the top values fl(fl(6 sigma) s_o) of c - 1 and c
decide between c - 1, c and c + 1; elsewhere they compute the top values of c - 2 .. c + 1,
step once up or down, and walk further only where that step is not enough
(fp32-subnormal products, or a far start).  That recipe is restated here in numpy, from the exact quotient
and from starts perturbed by a few ulps as an approximate reciprocal gives them, and
checked equal to ``oracle.formats.e4m3_inner_scale_byte`` (the brute-force
definition) on group maxima placed on and around every scale's top value, random
magnitudes over the fp32 range, and fp32-subnormal products.
"""
import numpy as np

from oracle import formats as F

F32 = np.float32
_ALL = np.arange(0, 0x7F, dtype=np.uint8)
_ALL_VALS = F.e4m3_decode(_ALL)


def _top(b, s_o):
    v = F.e4m3_decode(np.asarray(b).astype(np.uint8)).astype(F32)
    with np.errstate(over="ignore"):
        return ((F32(6.0) * v).astype(F32) * s_o).astype(F32)


FAST_S_O = F32(2.0 ** -110)        # at or above: every candidate top value is a normal fp32 number


def _ceil_byte(t):
    """The kernels' branch-free E4M3 ceiling of t >= 0: the fp32 bits rounded up to 3
    mantissa bits, rebiased (127 -> 7), clamped to the normal bytes 0x08 .. 0x7E."""
    bits = np.asarray(t, dtype=F32).view(np.uint32).astype(np.int64)
    c = ((bits + 0xFFFFF) >> 20) - 960
    return np.clip(c, 0x08, 0x7E)


def _recipe(a_i, s_o, rel=None, stats=None):
    """The kernels' selection: start c, the branch-free ceiling of the quotient.  With
    s_o >= 2^-110 the top values of c - 1 and c decide between c - 1, c and c + 1; below,
    the top values of c - 2 .. c + 1, one step, and walks where that step is not enough."""
    m6 = (s_o * F32(6.0)).astype(F32)
    with np.errstate(divide="ignore", over="ignore", invalid="ignore"):
        t = (a_i / m6).astype(F32)
        if rel is not None:                         # a first guess off by some ulps
            t = (t.astype(np.float64) * (1.0 + rel)).astype(F32)
    t = np.where(np.isnan(t), F32(np.inf), t)
    c = _ceil_byte(t)
    ref_c = np.maximum(_ALL[np.minimum(np.searchsorted(_ALL_VALS, t.astype(np.float64), side="left"), 0x7E)]
                       .astype(np.int64), 0x08)
    assert np.array_equal(c, ref_c)                 # the bit form is the E4M3 ceiling
    cp = np.where(c < 0x7E, c + 1, c)
    cm = np.where(c > 0x08, c - 1, c)
    cmm = np.where(cm > 0x08, cm - 1, cm)
    tp, t0, tm, tmm = _top(cp, s_o), _top(c, s_o), _top(cm, s_o), _top(cmm, s_o)
    up = t0 < a_i
    down = ~up & (cm < c) & (tm >= a_i)
    sb = np.where(up, cp, np.where(down, cm, c))
    fast = s_o >= FAST_S_O                          # the fast path ends here: no check, no walk
    more = ~fast & ((up & (cp < 0x7E) & (tp < a_i)) | (down & (cmm < cm) & (tmm >= a_i)))
    if stats is not None:
        stats["walks"] = int(more.sum())
        stats["fast_short"] = int((fast & ((up & (cp < 0x7E) & (tp < a_i)) | (down & (cmm < cm) & (tmm >= a_i)))).sum())
    for _ in range(120):                            # the walks, on the groups that need them
        step = more & (sb < 0x7E) & (_top(sb, s_o) < a_i)
        if not step.any():
            break
        sb = np.where(step, sb + 1, sb)
    for _ in range(120):
        step = more & (sb > 0x08) & (_top(np.maximum(sb - 1, 0), s_o) >= a_i)
        if not step.any():
            break
        sb = np.where(step, sb - 1, sb)
    return np.where(a_i > 0, sb, 0).astype(np.uint8)


def _cases(rng, n):
    s_o = np.exp2(rng.uniform(-126, 110, n)).astype(F32)
    sig = F.e4m3_decode(rng.integers(0x01, 0x7F, n).astype(np.uint8))
    on = (6 * sig * s_o.astype(np.float64)).astype(F32)
    out_a, out_s = [on], [s_o]
    for k in (1, 2, 5):
        up, dn = on.copy(), on.copy()
        for _ in range(k):
            up, dn = np.nextafter(up, F32(np.inf)), np.nextafter(dn, F32(0))
        out_a += [up, dn]
        out_s += [s_o, s_o]
    rnd = (s_o.astype(np.float64) * np.exp2(rng.uniform(-30, np.log2(2688 * 1.1), n))).astype(F32)
    out_a.append(rnd)
    out_s.append(s_o)
    # fp32-subnormal products: tiny outer scales (down to 2^-149) with amaxima near them
    s_t = np.exp2(-rng.integers(130, 150, n).astype(np.float64)).astype(F32)
    a_t = (s_t.astype(np.float64) * rng.uniform(0, 3000, n)).astype(F32)
    out_a.append(a_t)
    out_s.append(s_t)
    return np.concatenate(out_a), np.concatenate(out_s)


def test_recipe_equals_definition():
    rng = np.random.default_rng(21)
    a, s = _cases(rng, 100000)
    keep = np.isfinite(a)
    a, s = a[keep], s[keep]
    ref = F.e4m3_inner_scale_byte(a, s)
    assert np.array_equal(_recipe(a, s), ref)
    assert np.array_equal(_recipe(a, s, rng.uniform(-2.0 ** -20, 2.0 ** -20, a.size)), ref)
    # the walking path reaches the answer from any start; the fast path relies on the first
    # guess being a few ulps off at most (an approximate reciprocal and one product)
    slow = s < FAST_S_O
    assert np.array_equal(_recipe(a[slow], s[slow], rng.uniform(-0.3, 0.3, int(slow.sum()))), ref[slow])


def test_fast_path_never_needs_a_second_step():
    """With s_o >= 2^-110 the kernels stop after one step from c without checking it: over
    every case (tops on and around every scale, random magnitudes, starts a few ulps off),
    a second step would never have been needed."""
    rng = np.random.default_rng(23)
    a, s = _cases(rng, 100000)
    s_fast = np.exp2(rng.uniform(-110, -100, a.size)).astype(F32)      # the fast path's low edge
    a2 = (a.astype(np.float64) / s.astype(np.float64) * s_fast.astype(np.float64)).astype(F32)
    for aa, ss in ((a, s), (a2, s_fast)):
        ok = np.isfinite(aa) & (aa > 0)
        aa, ss = aa[ok], ss[ok]
        for rel in (None, rng.uniform(-2.0 ** -20, 2.0 ** -20, aa.size)):
            stats = {}
            assert np.array_equal(_recipe(aa, ss, rel, stats), F.e4m3_inner_scale_byte(aa, ss))
            assert stats["fast_short"] == 0


def test_walks_only_for_subnormal_products():
    """Where every product is a normal fp32 number, one step from the start decides the
    scale: the walks never run, from the exact quotient or from a start a few ulps off."""
    rng = np.random.default_rng(22)
    a, s = _cases(rng, 50000)
    ok = np.isfinite(a) & (s >= F32(2.0 ** -110)) & (a > 0)
    a, s = a[ok], s[ok]
    ref = F.e4m3_inner_scale_byte(a, s)
    for rel in (None, rng.uniform(-2.0 ** -20, 2.0 ** -20, a.size)):
        stats = {}
        assert np.array_equal(_recipe(a, s, rel, stats), ref)
        assert stats["walks"] == 0
