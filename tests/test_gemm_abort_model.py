"""CPU model of the GEMM kernel's synchronisation, normal and aborted.

k_gemm_nvfp4 (gemm.cu) has three roles per CTA: producer warps fill a 5-stage operand
ring (mbarriers full / empty, outer-scale slots sempty), the MMA warp turns each 128-K
block into a tensor-memory partial in a 3-slot ring (commit -> mbarrier pfull), and
eight promotion warps read each partial and release its slot through hardware named
barriers (one per slot, 9 warps per generation: the MMA warp meets it with a sync
before it reuses the slot; a live promotion warp arrives without waiting).  Each
promotion warp also hands an FP4 block's outer-scale slot back once its math is done
(sempty completes a phase after eight arrivals).  Every
mbarrier wait is bounded; a wait that runs out sets the CTA's abort flag, after which
the roles stop working but keep the named-barrier protocol, which has no time bound.

This model restates that protocol at the level of the barriers (one actor per warp, a
random interleaving and random relative speeds per trial) and checks, over thousands of
interleavings with and without an injected fault (a stage whose loads are never issued,
or a wait that runs out at a random moment), that every actor finishes, that no warp
takes part twice in one named-barrier generation, and that no block's outer scales are
overwritten before its promotion (a planted mistake, producers that do not wait for the
slot's hand-back, is caught).  A promotion warp that stops being live must first
see the MMA warp meet the slot's previous generation (the kernel's `met` counters,
compared by parity with the slot's phase, which the model checks is enough);
without that gate the model finds the double participation that would derail the
generations, which the last test shows.
"""
import random

import pytest

STAGES, PSLOTS, PROD, PROMO, SSLOTS = 5, 3, 3, 8, 8
COUNT = 1 + PROMO                       # warps per named-barrier generation


class Violation(Exception):
    pass


class Model:
    def __init__(self, works, skip_stage=None, gate=True, rng=None, timeout_at=None, wait_sempty=True):
        self.works = works                   # per CTA work list: (nkb4, nk8)
        self.wait_sempty = wait_sempty       # False: planted mistake, outer-scale slots reloaded unasked
        self.skip = skip_stage
        self.gate = gate
        self.rng = rng or random.Random(0)
        self.timeout_at = timeout_at         # force a bounded wait to run out after this many steps
        self.steps = 0
        self.abort = False
        self.timeouts = 0
        self.full = [0] * STAGES             # completed phases per mbarrier
        self.empty = [0] * STAGES
        self.pfull = [0] * PSLOTS
        self.sempty = [0] * SSLOTS             # completed phases of each outer-scale slot
        self.sempty_arrivals = [0] * SSLOTS
        self.sload = [0] * SSLOTS              # outer-scale loads landed per slot
        self.met = [0] * PSLOTS              # generations the MMA warp has met per slot
        self.bar = {s: {"gen": 0, "members": set()} for s in range(PSLOTS)}

    # --- primitives (generators yield until they can proceed) ---------------------------
    def wait_bounded(self, arr, idx, phase):
        """Wait until arr[idx] > phase; False when it runs out or the CTA has aborted."""
        while True:
            if self.abort:
                return False
            if arr[idx] > phase:
                return True
            if self.timeout_at is not None and self.steps >= self.timeout_at:
                self.timeout_at = None
                self.abort = True
                self.timeouts += 1
                return False
            yield ("wait", arr is self.full and "full" or "other")

    def stalled_timeout(self):
        """All actors blocked: a bounded wait runs out (the hardware clock bound)."""
        self.abort = True
        self.timeouts += 1

    def arrive(self, s, warp):
        b = self.bar[s]
        if warp in b["members"]:
            raise Violation("warp %s takes part twice in generation %d of slot %d" % (warp, b["gen"], s))
        b["members"].add(warp)
        if len(b["members"]) == COUNT:
            b["gen"] += 1
            b["members"] = set()

    def sync(self, s, warp):
        b = self.bar[s]
        gen = b["gen"]
        self.arrive(s, warp)
        while self.bar[s]["gen"] == gen:
            yield ("named", s)

    # --- roles ---------------------------------------------------------------------------
    def stages(self):
        for w in self.works:
            nkb4, nk8 = w
            nst4 = (nkb4 + 1) // 2
            for st in range(nst4 + nk8):
                yield w, st, nst4

    def producer(self, warp):
        it, fbase, issued, ok = 0, 0, set(), True
        for w in self.works:
            if not ok:
                break
            nkb4, nk8 = w
            nst4 = (nkb4 + 1) // 2
            for st in range(nst4 + nk8):
                if it % PROD != warp:
                    it += 1
                    continue
                slot = it % STAGES
                if it >= STAGES:
                    ok = yield from self.wait_bounded(self.empty, slot, it // STAGES - 1)
                    if not ok:
                        break
                nkbs = min(2, nkb4 - 2 * st) if st < nst4 else 0
                for j in range(nkbs):
                    f = fbase + 2 * st + j
                    if f >= SSLOTS and ok and self.wait_sempty:
                        ok = yield from self.wait_bounded(self.sempty, f % SSLOTS, f // SSLOTS - 1)
                if not ok:
                    break
                if it != self.skip:
                    self.full[slot] += 1          # expect_tx + copies land
                    for j in range(nkbs):         # with the outer scales of the stage's blocks
                        self.sload[(fbase + 2 * st + j) % SSLOTS] += 1
                    issued.add(it)
                it += 1
            fbase += nkb4
        # drain: the copies it issued have landed (they complete by themselves in the model)

    def mma(self):
        it, pc, live = 0, 0, True
        for w, st, nst4 in self.stages():
            nkb4, nk8 = w
            slot = it % STAGES
            if live:
                live = yield from self.wait_bounded(self.full, slot, it // STAGES)
            if st < nst4:
                for kbl in range(min(2, nkb4 - 2 * st)):
                    ps = pc % PSLOTS
                    if pc >= PSLOTS:
                        yield from self.sync(ps, "mma")
                        self.met[ps] += 1
                    if live:
                        self.pfull[ps] += 1       # MMAs complete, commit arrives
                    pc += 1
            else:
                s8 = st - nst4
                ps = pc % PSLOTS
                if s8 == 0 and pc >= PSLOTS:
                    yield from self.sync(ps, "mma")
                    self.met[ps] += 1
                if live and s8 == nk8 - 1:
                    self.pfull[ps] += 1
                if s8 == nk8 - 1:
                    pc += 1
            if live:
                self.empty[slot] += 1             # the stage's MMAs complete
            it += 1
        for j in range(max(pc - PSLOTS, 0), pc):
            yield from self.sync(j % PSLOTS, "mma")
            self.met[j % PSLOTS] += 1

    def promo(self, warp):
        live, blk, f4c = True, 0, 0
        for w in self.works:
            nkb4, nk8 = w
            nblk = nkb4 + (1 if nk8 else 0)
            for kb in range(nblk):
                ps = blk % PSLOTS
                if live:
                    live = yield from self.wait_bounded(self.pfull, ps, blk // PSLOTS)
                if live and kb < nkb4 and self.sload[f4c % SSLOTS] != f4c // SSLOTS + 1:
                    raise Violation("outer scales of block %d overwritten before their promotion" % f4c)
                if live:
                    self.arrive(ps, warp)
                    if kb < nkb4:                 # the math is done with the block's outer scales
                        s = f4c % SSLOTS
                        self.sempty_arrivals[s] += 1
                        if self.sempty_arrivals[s] % PROMO == 0:
                            self.sempty[s] += 1
                        f4c += 1
                else:
                    if self.gate:
                        # the slot's previous generation must have been met by the MMA warp.  The
                        # kernel compares parities: this is use u of the slot and met is u - 1 or u
                        u = blk // PSLOTS
                        while (self.met[ps] & 1) != (u & 1):
                            if self.met[ps] not in (u - 1, u):
                                raise Violation("met %d at use %d of slot %d" % (self.met[ps], u, ps))
                            yield ("gate", ps)
                        if self.met[ps] != u:
                            raise Violation("gate passed with met %d at use %d" % (self.met[ps], u))
                    yield from self.sync(ps, warp)
                blk += 1

    # --- scheduler -------------------------------------------------------------------------
    def run(self, max_steps=200000):
        actors = {("prod", p): self.producer(p) for p in range(PROD)}
        actors["mma"] = self.mma()
        actors.update({("promo", q): self.promo(("promo", q)) for q in range(PROMO)})
        pending = dict(actors)
        # each actor takes 1 to 3 steps per round (drawn per trial), so that some trials run
        # a role several blocks ahead of another
        speed = {name: self.rng.choice((1, 1, 2, 3)) for name in actors}
        blocked_rounds = 0
        while pending:
            self.steps += 1
            if self.steps > max_steps:
                raise Violation("no progress: " + str(sorted(map(str, pending))))
            progressed = False
            for name in self.rng.sample(list(pending), len(pending)):
                for _ in range(speed[name]):
                    before = self.snapshot()
                    try:
                        next(pending[name])
                    except StopIteration:
                        del pending[name]
                        progressed = True
                        break
                    if self.snapshot() != before:
                        progressed = True
            if progressed:
                blocked_rounds = 0
            else:
                blocked_rounds += 1
                if blocked_rounds > 3:
                    if self.abort:
                        raise Violation("deadlock after abort: " + str(sorted(map(str, pending))))
                    self.stalled_timeout()
                    blocked_rounds = 0
        return self

    def snapshot(self):
        return (tuple(self.full), tuple(self.empty), tuple(self.pfull), tuple(self.met), tuple(self.sload),
                tuple(self.sempty),
                tuple(self.sempty_arrivals), self.abort,
                tuple((b["gen"], len(b["members"])) for b in self.bar.values()))


WORK_SETS = [
    [(4, 0)] * 3,                  # FP4 only, three tiles
    [(7, 0), (7, 0)],              # odd number of blocks
    [(8, 2), (8, 2)],              # FP4 and an FP8 slice of two stages
    [(0, 6), (2, 0), (0, 3)],      # FP8-only works between FP4 ones (pair launches)
]


@pytest.mark.parametrize("works", WORK_SETS)
def test_normal_runs_complete_without_timeouts(works):
    for seed in range(50):
        m = Model(works, rng=random.Random(seed)).run()
        assert m.timeouts == 0 and not m.abort
        assert all(len(b["members"]) == 0 for b in m.bar.values())


@pytest.mark.parametrize("works", WORK_SETS)
def test_skipped_stage_aborts_and_every_warp_finishes(works):
    nst = sum((a + 1) // 2 + b for a, b in works)
    for seed in range(200):
        rng = random.Random(seed)
        m = Model(works, skip_stage=rng.randrange(nst), rng=rng).run()
        assert m.abort and m.timeouts >= 1
        assert all(len(b["members"]) == 0 for b in m.bar.values())   # no generation left open


@pytest.mark.parametrize("works", WORK_SETS)
def test_timeout_at_any_moment(works):
    for seed in range(300):
        rng = random.Random(1000 + seed)
        m = Model(works, rng=rng, timeout_at=rng.randrange(1, 400)).run()
        assert all(len(b["members"]) == 0 for b in m.bar.values())


def test_without_the_gate_a_warp_can_take_part_twice():
    """Planted in the model: a warp that stops being live syncs at once.  Some
    interleaving then makes it join a generation it already arrived on."""
    found = False
    for seed in range(3000):
        rng = random.Random(seed)
        try:
            Model([(8, 0), (8, 0)], gate=False, rng=rng, timeout_at=rng.randrange(1, 300)).run()
        except Violation as e:
            found = "twice" in str(e) or "deadlock" in str(e)
            if found:
                break
    assert found


def test_outer_scale_slots_need_the_hand_back():
    """Planted in the model: the producers load a stage without waiting for its blocks'
    outer-scale slots to be handed back.  Some interleaving then overwrites a block's outer
    scales before every promotion warp has used them."""
    found = False
    for seed in range(500):
        try:
            Model([(16, 0), (16, 0)], rng=random.Random(seed), wait_sempty=False).run()
        except Violation as e:
            found = "overwritten" in str(e)
            if found:
                break
    assert found
