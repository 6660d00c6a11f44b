"""Randomised simulation of the barrier protocol of the GEMM's multicast
plans (csrc/rs_gemm.cu: 256-row activation tiles without K split, the two
CTAs of a (2,1,1) cluster sharing each activation tile).

Per CTA and stage s: full[s] (one arrival with the expected bytes from the
CTA's own producer; the bytes complete from its weight copy, its own half of
the activation tile and the partner's half, in any order, possibly before
the arrival), sfr[s] (four scale warps), empty[s] (two arrivals: both CTAs'
MMA commits; the commits of the last S units, whose stages are never
refilled, stay local), and one accumulator (accum_full, accum_empty with
eight epilogue arrivals).  mbarrier semantics: a phase completes when its
pending arrivals and its transaction count are both zero; the count may go
below zero first.  Checks that every actor finishes (no deadlock), that no
copy lands in a stage whose previous unit the MMAs of that CTA still read,
that the scale warps never rewrite a stage's scale columns before its
previous MMAs are done, and that nothing is in flight at the end."""
import random

import pytest


class Bar:
    def __init__(self, count):
        self.count = count
        self.pending = count
        self.tx = 0
        self.phase = 0  # completed phases

    def _check(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def arrive(self, expect_tx=0):
        self.tx += expect_tx
        self.pending -= 1
        assert self.pending >= 0
        self._check()

    def complete_tx(self, n):
        self.tx -= n
        self._check()

    def done(self, parity):
        return (self.phase & 1) != parity


W, H = 3, 2  # bytes of a stage's weight copy and of each activation half (units)


def simulate(S, ntl, chunks, seed, commit_both=True):
    """commit_both=False plants a mistake: each CTA's commit arrives only on its
    own empty barrier (count 1)."""
    rng = random.Random(seed)
    nu = ntl * chunks
    ec = 2 if commit_both else 1
    cta = [dict(full=[Bar(1) for _ in range(S)], empty=[Bar(ec) for _ in range(S)], sfr=[Bar(4) for _ in range(S)],
                accum_full=Bar(1), accum_empty=Bar(8)) for _ in range(2)]
    # per CTA and stage: the unit whose bytes it holds / still waits for, and
    # the last unit whose MMAs are done with it
    landed = [[dict() for _ in range(S)] for _ in range(2)]  # stage -> {unit: bytes landed}
    mma_done = [[-1] * S for _ in range(2)]
    sf_unit = [[-1] * S for _ in range(2)]
    inflight = []  # (dst cta, stage, unit, bytes)

    def issue(dst, s, u, n):
        # a copy may only target a stage whose previous unit's MMAs are done
        assert mma_done[dst][s] >= u - S, (dst, s, u, mma_done[dst][s])
        inflight.append((dst, s, u, n))

    def producer(r):
        s, ph = 0, 0
        for u in range(nu):
            if u >= S:
                while not cta[r]["empty"][s].done(ph ^ 1):
                    yield
            cta[r]["full"][s].arrive(expect_tx=W + 2 * H)
            issue(r, s, u, W)              # own weights
            issue(r, s, u, H)              # own half, multicast to both
            issue(1 - r, s, u, H)
            yield
            s += 1
            if s == S:
                s, ph = 0, ph ^ 1

    def land():
        while True:
            if inflight and rng.random() < 0.5:
                r, s, u, n = inflight.pop(rng.randrange(len(inflight)))
                landed[r][s][u] = landed[r][s].get(u, 0) + n
                cta[r]["full"][s].complete_tx(n)
            yield

    def scale_warp(r):
        s, ph = 0, 0
        for u in range(nu):
            while not cta[r]["full"][s].done(ph):
                yield
            assert landed[r][s].get(u, 0) == W + 2 * H, (r, s, u, landed[r][s])
            assert mma_done[r][s] >= u - S  # the previous unit's MMAs no longer read the columns
            sf_unit[r][s] = u
            yield
            cta[r]["sfr"][s].arrive()
            s += 1
            if s == S:
                s, ph = 0, ph ^ 1

    def mma(r):
        s, ph, u = 0, 0, 0
        for j in range(ntl):
            if j > 0:
                while not cta[r]["accum_empty"].done((j - 1) & 1):
                    yield
            for _ in range(chunks):
                while not (cta[r]["full"][s].done(ph) and cta[r]["sfr"][s].done(ph)):
                    yield
                assert landed[r][s].get(u, 0) == W + 2 * H and sf_unit[r][s] == u
                for _ in range(rng.randrange(1, 4)):
                    yield  # MMAs run
                mma_done[r][s] = u
                del landed[r][s][u]
                if commit_both and u + S < nu:
                    for d in range(2):
                        cta[d]["empty"][s].arrive()
                else:
                    cta[r]["empty"][s].arrive()  # never waited on
                u += 1
                s += 1
                if s == S:
                    s, ph = 0, ph ^ 1
            cta[r]["accum_full"].arrive()

    def epilogue(r):
        for j in range(ntl):
            while not cta[r]["accum_full"].done(j & 1):
                yield
            yield  # read the accumulator
            cta[r]["accum_empty"].arrive()

    actors = [producer(r) for r in (0, 1)] + [scale_warp(r) for r in (0, 1) for _ in range(4)]
    actors += [mma(r) for r in (0, 1)] + [epilogue(r) for r in (0, 1) for _ in range(8)]
    lander = land()
    alive = list(actors)
    steps = 0
    while alive:
        steps += 1
        assert steps < 400000, "deadlock"
        next(lander)
        a = rng.choice(alive)
        try:
            next(a)
        except StopIteration:
            alive.remove(a)
    assert not inflight
    return steps


@pytest.mark.parametrize("S", [2, 3, 4])
@pytest.mark.parametrize("ntl,chunks", [(1, 1), (1, 5), (2, 3), (3, 8), (7, 4)])
def test_multicast_protocol_finishes_and_never_refills_early(S, ntl, chunks):
    for seed in range(10):
        simulate(S, ntl, chunks, seed)


def test_local_commits_would_refill_early():
    """With each CTA's commit arriving only on its own empty barrier, a CTA may
    multicast into its partner's stage while the partner's MMAs still read it:
    the model catches that (which pins the count-2 barrier and the multicast
    commit)."""
    caught = 0
    for seed in range(30):
        try:
            simulate(3, 3, 4, seed, commit_both=False)
        except AssertionError:
            caught += 1
    assert caught > 0
