"""Host model of the backward kernel's exit after a wait gives up.

A bounded wait that runs out of time sets the CTA's abort flag and returns
false, and from then on every wait of the CTA returns false at once (the
flag is read while polling).  The kernel must still end: every warp reaches
the final block-wide barrier, and the four drain warps, which meet at a
named barrier twice per step, must all take it the same number of times (a
warp that left the loop early would leave the others waiting forever).

The model runs the warps' programs (producer, issuers A and B, four P/dS
warps, four drain warps; products and loads complete on their own), makes
one randomly chosen wait give up, and checks that every warp finishes.
Waits that ignore the flag (an issuer waiting for its own products, the
producer for its own loads) are modelled as such: they end because what
they wait for always completes.  A drain that breaks out of its loop after
a failed wait is shown to hang.
"""
import random

import pytest

SBUFS = STAGES = 3
WARPS = 4


def sbuf(it):
    return it % SBUFS


def spar(it):
    return (it // SBUFS) & 1


class Bar:
    def __init__(self, count):
        self.count, self.pending, self.completed = count, 0, 0

    def arrive(self):
        self.pending += 1
        if self.pending == self.count:
            self.pending, self.completed = 0, self.completed + 1

    def passes(self, parity):
        return (self.completed & 1) != parity


class Named:
    """bar.sync of a fixed thread count: generation g opens when all arrived."""

    def __init__(self, count):
        self.count, self.arrived, self.gen = count, 0, 0

    def arrive(self):
        self.arrived += 1
        g = self.gen
        if self.arrived == self.count:
            self.arrived, self.gen = 0, self.gen + 1
        return g


def run(n, fail_at, rng, early_break_drain=False):
    bar = {
        "stage_full": [Bar(1) for _ in range(STAGES)], "s_full": [Bar(1) for _ in range(SBUFS)],
        "sm_done": [Bar(WARPS) for _ in range(SBUFS)], "dq_full": [Bar(1) for _ in range(SBUFS)],
        "dq_free": [Bar(WARPS) for _ in range(SBUFS)], "dp_full": [Bar(1)], "dp_read": [Bar(WARPS)],
        "acc_done": [Bar(1)], "a_done": [Bar(1)],
    }
    drain_bar = Named(WARPS)
    st = {"abort": False, "waits": 0, "loads": [], "pipe": []}

    def wait(name, i, parity, honours_abort=True):
        """A program step: yields until the wait passes or fails; returns its result."""
        while True:
            if honours_abort and st["abort"]:
                return False
            if bar[name][i].passes(parity):
                st["waits"] += 1
                if st["waits"] == fail_at and honours_abort:  # this one runs out of time instead
                    st["abort"] = True
                    return False
                return True
            yield

    def mma(*targets):
        st["pipe"].append(targets)

    def producer():
        issued = 0
        for it in range(n):
            if it >= STAGES:
                j = it - STAGES
                ok = yield from wait("dq_full", sbuf(j), spar(j))
                if not ok:
                    break
            st["loads"].append(("stage_full", it % STAGES))
            issued += 1
        for c in range(max(0, issued - STAGES), issued):  # its own loads land whatever happened
            yield from wait("stage_full", c % STAGES, (c // STAGES) & 1, honours_abort=False)

    def issuer_a():
        ok = True
        def s_step(step):
            ok = yield from wait("stage_full", step % STAGES, (step // STAGES) & 1)
            if ok:
                mma(("s_full", sbuf(step)))
            return ok
        if n > 0:
            ok = yield from s_step(0)
            if ok:
                mma(("dp_full", 0))
            step = 1
            while ok and step < min(SBUFS, n):
                ok = yield from s_step(step)
                step += 1
        it = 0
        while ok and it < n:
            if it + 1 < n:
                ok = yield from wait("dp_read", 0, it & 1)
                if not ok:
                    break
                mma(("dp_full", 0))
            nxt = it + SBUFS - 1
            if it >= 1 and nxt < n:
                ok = yield from wait("dq_free", sbuf(it - 1), spar(it - 1))
                if not ok:
                    break
                ok = yield from s_step(nxt)
            it += 1
        mma(("a_done", 0))
        yield from wait("a_done", 0, 0, honours_abort=False)  # its own products always complete

    def issuer_b():
        for it in range(n):
            ok = yield from wait("sm_done", sbuf(it), spar(it))
            if not ok:
                break
            mma(("dq_full", sbuf(it)))
        mma(("acc_done", 0))
        yield from wait("acc_done", 0, 0, honours_abort=False)

    def pds_warp():
        for it in range(n):
            ok = True
            if it >= 2:
                ok = yield from wait("dq_full", sbuf(it - 2), spar(it - 2))
            ok = ok and (yield from wait("stage_full", it % STAGES, (it // STAGES) & 1))
            ok = ok and (yield from wait("s_full", sbuf(it), spar(it)))
            if not ok:
                break
            ok = yield from wait("dp_full", 0, it & 1)
            if not ok:
                break
            bar["dp_read"][0].arrive()
            bar["sm_done"][sbuf(it)].arrive()
        yield from wait("acc_done", 0, 0)  # the dV epilogue, skipped on an abort

    def drain_warp():
        ok = True
        for it in range(n):
            w = ok and (yield from wait("dq_full", sbuf(it), spar(it)))
            ok = w
            if w:
                bar["dq_free"][sbuf(it)].arrive()
            elif early_break_drain:
                break
            for _ in range(2):  # the two named barriers of the step, whatever w was
                g = drain_bar.arrive()
                while drain_bar.gen == g:
                    yield
        yield from wait("acc_done", 0, 0)  # the dK epilogue, skipped on an abort

    progs = [producer(), issuer_a(), issuer_b()] + [pds_warp() for _ in range(WARPS)] + [drain_warp() for _ in range(WARPS)]
    live = list(range(len(progs)))
    for _ in range(200000):
        if not live and not st["loads"] and not st["pipe"]:
            return True
        choices = list(live) + (["load"] if st["loads"] else []) + (["pipe"] if st["pipe"] else [])
        c = rng.choice(choices)
        if c == "load":
            name, i = st["loads"].pop(rng.randrange(len(st["loads"])))
            bar[name][i].arrive()
        elif c == "pipe":
            for name, i in st["pipe"].pop(0):
                bar[name][i].arrive()
        else:
            try:
                next(progs[c])
            except StopIteration:
                live.remove(c)
    return False  # some warp never finished


@pytest.mark.parametrize("n", [1, 3, 4, 8])
def test_every_warp_finishes_after_a_wait_gives_up(n):
    rng = random.Random(n)
    for fail_at in list(range(1, 40)) + [10 ** 9]:  # 10**9: no wait gives up
        for _ in range(4):
            assert run(n, fail_at, rng), (n, fail_at)


def test_a_drain_that_leaves_early_hangs():
    rng = random.Random(2)
    hung = any(not run(6, fail_at, rng, early_break_drain=True) for fail_at in range(5, 40) for _ in range(3))
    assert hung
