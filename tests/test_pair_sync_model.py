"""Randomised simulation of the barrier protocol of the paired-CTA GEMM
(csrc/rs_gemm_pair.cu; mbarrier
phase semantics: a barrier completes a phase when its pending arrivals reach
zero; try_wait(parity P) succeeds once the phase with parity P is complete,
i.e. the barrier's current phase parity differs from P).  Checks that every
actor finishes (no deadlock) and that no stage is overwritten before the
MMAs that read it are done, for several stage counts, tile counts and chunk
counts, under random interleavings."""
import random


class Bar:
    def __init__(self, count):
        self.count = count
        self.pending = count
        self.phase = 0  # completed phases

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def done(self, parity):
        return (self.phase & 1) != parity


def simulate(S, ntl, chunks, seed):
    rng = random.Random(seed)
    nu = ntl * chunks
    cta = [dict(full=[Bar(1) for _ in range(S)], empty=[Bar(1) for _ in range(S)], accum_full=Bar(1)) for _ in range(2)]
    pfull = [Bar(1) for _ in range(S)]
    accum_empty = Bar(8)
    stage_owner = [[None] * S for _ in range(2)]  # unit loaded into stage s of each CTA, None when free
    inflight = []  # (cta, stage, unit) copies in flight
    mma_reading = {}

    def producer(r):
        s, ph = 0, 0
        for u in range(nu):
            if u >= S:
                while not cta[r]["empty"][s].done(ph ^ 1):
                    yield
            assert stage_owner[r][s] is None or stage_owner[r][s] < u - S + 1
            inflight.append((r, s, u))
            yield
            s += 1
            if s == S:
                s, ph = 0, ph ^ 1

    def land():
        # copies land in any order, some time later
        while True:
            if inflight and rng.random() < 0.5:
                r, s, u = inflight.pop(rng.randrange(len(inflight)))
                stage_owner[r][s] = u
                cta[r]["full"][s].arrive()
            yield

    def relay():
        s, ph = 0, 0
        for u in range(nu):
            while not cta[1]["full"][s].done(ph):
                yield
            pfull[s].arrive()
            yield
            s += 1
            if s == S:
                s, ph = 0, ph ^ 1

    def mma():
        s, ph = 0, 0
        u = 0
        for j in range(ntl):
            if j > 0:
                while not accum_empty.done((j - 1) & 1):
                    yield
            for i in range(chunks):
                while not (cta[0]["full"][s].done(ph) and pfull[s].done(ph)):
                    yield
                assert stage_owner[0][s] == u and stage_owner[1][s] == u, (stage_owner, s, u)
                yield  # MMAs run
                # multicast commit: both CTAs' empty[s]
                for r in range(2):
                    stage_owner[r][s] = None
                    cta[r]["empty"][s].arrive()
                u += 1
                s += 1
                if s == S:
                    s, ph = 0, ph ^ 1
            for r in range(2):
                cta[r]["accum_full"].arrive()

    def epilogue(r):
        for j in range(ntl):
            while not cta[r]["accum_full"].done(j & 1):
                yield
            yield  # read the accumulator
            accum_empty.arrive()

    actors = [producer(0), producer(1), relay(), mma()] + [epilogue(r) for r in (0, 1) for _ in range(4)]
    lander = land()
    alive = list(actors)
    steps = 0
    while alive:
        steps += 1
        assert steps < 200000, "deadlock"
        next(lander)
        a = rng.choice(alive)
        try:
            next(a)
        except StopIteration:
            alive.remove(a)
    return steps


import pytest


@pytest.mark.parametrize("S", [2, 3, 5, 6])
@pytest.mark.parametrize("ntl,chunks", [(1, 1), (1, 32), (2, 3), (5, 3), (5, 32)])
def test_pair_protocol_finishes_and_never_refills_early(S, ntl, chunks):
    for seed in range(12):
        simulate(S, ntl, chunks, seed)
