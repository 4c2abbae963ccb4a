"""Host model of the backward kernel's barriers, buffers and parity waits.

One CTA of the backward walks n query steps with five kinds of workers: the
producer (each step's Q/dO stage, three deep, reloaded once dQ^T of the step
that last used it is done), issuer A (S^T into one of three tensor-memory
buffers, dP^T into its single buffer), four P/dS warps, issuer B (dV, dK and
dQ^T of a step), and four drain warps (dQ^T out of its buffer).  Products
complete in issue order (one tensor core), loads in any order.

Every mbarrier wait in the kernel is a parity wait, sound only if the
waiter has seen the barrier's previous completion and the next one cannot
come first.  The model runs the kernel's programs, in the kernel's order of
waits, under random schedules and checks

  - every passed wait against the completion the waiter meant (a pass on an
    older completion of the same parity is a stale wait);
  - every buffer access against the accesses it must follow: a stage is
    loaded again only after every reader of its previous step is done, S^T
    goes into a buffer only after the drain has read that buffer's dQ^T,
    dP^T is overwritten only after the warps have read it, a dS^T tile is
    written only after the dQ^T that read it last is complete, and every
    read finds the data of its own step;
  - that every schedule runs to the end (no stall).

Mutations, each dropping one wait of the protocol, must be caught, so that
the checks are shown to bite.
"""
import random

import pytest

SBUFS = 3     # S^T buffers in tensor memory (one per step in turn)
STAGES = 3    # Q/dO stages in shared memory
WARPS = 4     # P/dS warps, and drain warps


def sbuf(it):
    return it % SBUFS


def spar(it):
    return (it // SBUFS) & 1


class Barrier:
    def __init__(self, count):
        self.count, self.pending, self.completed = count, 0, 0

    def arrive(self):
        self.pending += 1
        if self.pending == self.count:
            self.pending, self.completed = 0, self.completed + 1

    def passes(self, parity):
        return (self.completed & 1) != parity


class Model:
    def __init__(self, n, rng, skip=()):
        self.n, self.rng, self.skip = n, rng, set(skip)
        b = Barrier
        self.bar = {
            "stage_full": [b(1) for _ in range(STAGES)],
            "s_full": [b(1) for _ in range(SBUFS)],
            "sm_done": [b(WARPS) for _ in range(SBUFS)],
            "dq_full": [b(1) for _ in range(SBUFS)],
            "dq_free": [b(WARPS) for _ in range(SBUFS)],
            "dp_full": [b(1)],
            "dp_read": [b(WARPS)],
        }
        self.errors = []
        self.loads = []          # (stage, step) in flight
        self.pipe = []           # products in issue order: (label, step, on_complete)
        # what each buffer holds, and what has happened to each step
        self.stage_holds = [None] * STAGES   # step whose Q/dO/L/D landed there
        self.stage_readers = {}              # step -> readers not done
        self.tmem_s = [None] * SBUFS         # ("S"|"PdS"|"dQ", step)
        self.drained = set()                 # steps whose dQ^T the drain has read (all warps)
        self.drain_reads = {}                # step -> drain warps that read it
        self.dp_holds = None                 # step of the dP^T in its buffer
        self.dp_reads = {}                   # step -> P/dS warps that read dP^T
        self.tile = [None, None]             # step whose dS^T a tile holds
        self.tile_writes = {}                # step -> warps that wrote their dS^T rows
        self.pds_done = {}                   # step -> warps done with P, dS
        self.dq_done = set()                 # steps whose dQ^T product completed

    def err(self, msg):
        self.errors.append(msg)

    # -- the workers' programs: generators yielding ("wait", name, index, parity, meant)
    # or ("act", fn); `meant` is the completion count the wait is meant to see
    def producer(self):
        for it in range(self.n):
            st = it % STAGES
            if it >= STAGES and "stage_release" not in self.skip:
                j = it - STAGES
                yield ("wait", "dq_full", sbuf(j), spar(j), j // SBUFS + 1)
            def load(it=it, st=st):
                prev = it - STAGES
                if prev >= 0 and self.stage_readers.get(prev):
                    self.err(f"stage {st} reloaded for step {it} while {sorted(self.stage_readers[prev])} of step {prev} read it")
                self.stage_readers[it] = {"S", "dP", "dVdK"} | {f"w{w}" for w in range(WARPS)}
                self.loads.append((st, it))
            yield ("act", load)

    def issuer_a(self):
        n = self.n

        def s_step(step):
            yield ("wait", "stage_full", step % STAGES, (step // STAGES) & 1, step // STAGES + 1)
            def issue(step=step):
                b = sbuf(step)
                if self.stage_holds[step % STAGES] != step:
                    self.err(f"S^T({step}) issued on stage data of step {self.stage_holds[step % STAGES]}")
                prev = step - SBUFS
                if prev >= 0 and prev not in self.drained:
                    self.err(f"S^T({step}) issued into buffer {b} before the drain read dQ^T({prev})")
                def done(step=step, b=b):
                    self.tmem_s[b] = ("S", step)
                    self.stage_readers[step].discard("S")
                    self.bar["s_full"][b].arrive()
                self.pipe.append(("S", step, done))
            yield ("act", issue)

        def dp_step(step):
            def issue(step=step):
                if self.stage_holds[step % STAGES] != step:
                    self.err(f"dP^T({step}) issued on stage data of step {self.stage_holds[step % STAGES]}")
                if step > 0 and len(self.dp_reads.get(step - 1, ())) < WARPS:
                    self.err(f"dP^T({step}) issued before every warp read dP^T({step - 1})")
                def done(step=step):
                    self.dp_holds = step
                    self.stage_readers[step].discard("dP")
                    self.bar["dp_full"][0].arrive()
                self.pipe.append(("dP", step, done))
            yield ("act", issue)

        if n > 0:
            yield from s_step(0)
            yield from dp_step(0)
            for step in range(1, min(SBUFS, n)):
                yield from s_step(step)
        for it in range(n):
            if it + 1 < n:
                if "dp_read" not in self.skip:
                    yield ("wait", "dp_read", 0, it & 1, it + 1)
                yield from dp_step(it + 1)
            nxt = it + SBUFS - 1
            if it >= 1 and nxt < n:
                if "dq_free" not in self.skip:
                    yield ("wait", "dq_free", sbuf(it - 1), spar(it - 1), (it - 1) // SBUFS + 1)
                yield from s_step(nxt)

    def pds_warp(self, w):
        for it in range(self.n):
            b, st = sbuf(it), it % STAGES
            if it >= 2 and "tile" not in self.skip:
                yield ("wait", "dq_full", sbuf(it - 2), spar(it - 2), (it - 2) // SBUFS + 1)
            yield ("wait", "stage_full", st, (it // STAGES) & 1, it // STAGES + 1)
            yield ("wait", "s_full", b, spar(it), it // SBUFS + 1)
            def p_phase(it=it, b=b, st=st):
                if self.tmem_s[b] != ("S", it):
                    self.err(f"warp {w} read S^T({it}) from a buffer holding {self.tmem_s[b]}")
                if self.stage_holds[st] != it:
                    self.err(f"warp {w} read L of step {it} from a stage holding step {self.stage_holds[st]}")
            yield ("act", p_phase)
            yield ("wait", "dp_full", 0, it & 1, it + 1)
            def ds_phase(it=it, b=b, st=st):
                if self.dp_holds != it:
                    self.err(f"warp {w} read dP^T({it}) from a buffer holding step {self.dp_holds}")
                self.dp_reads.setdefault(it, set()).add(w)
                self.bar["dp_read"][0].arrive()
                if it >= 2 and (it - 2) not in self.dq_done:
                    self.err(f"warp {w} wrote dS^T({it}) into tile {it & 1} before dQ^T({it - 2}) read it")
                self.tile_writes.setdefault(it, set()).add(w)
                if len(self.tile_writes[it]) == WARPS:
                    self.tile[it & 1] = it
                self.stage_readers[it].discard(f"w{w}")
                self.pds_done.setdefault(it, set()).add(w)
                if len(self.pds_done[it]) == WARPS:
                    self.tmem_s[b] = ("PdS", it)
                self.bar["sm_done"][b].arrive()
            yield ("act", ds_phase)

    def issuer_b(self):
        for it in range(self.n):
            b = sbuf(it)
            yield ("wait", "sm_done", b, spar(it), it // SBUFS + 1)
            def issue(it=it, b=b):
                if self.tmem_s[b] != ("PdS", it):
                    self.err(f"dV, dK({it}) issued on a buffer holding {self.tmem_s[b]}")
                if self.tile[it & 1] != it:
                    self.err(f"dQ^T({it}) issued on tile {it & 1} holding step {self.tile[it & 1]}")
                def dvdk_done(it=it):
                    self.stage_readers[it].discard("dVdK")
                def dq_done(it=it, b=b):
                    self.tmem_s[b] = ("dQ", it)
                    self.dq_done.add(it)
                    self.bar["dq_full"][b].arrive()
                self.pipe.append(("dVdK", it, dvdk_done))
                self.pipe.append(("dQ", it, dq_done))
            yield ("act", issue)

    def drain_warp(self, w):
        for it in range(self.n):
            b = sbuf(it)
            yield ("wait", "dq_full", b, spar(it), it // SBUFS + 1)
            def read(it=it, b=b):
                if self.tmem_s[b] != ("dQ", it):
                    self.err(f"drain warp {w} read dQ^T({it}) from a buffer holding {self.tmem_s[b]}")
                self.drain_reads.setdefault(it, set()).add(w)
                if len(self.drain_reads[it]) == WARPS:
                    self.drained.add(it)
                self.bar["dq_free"][b].arrive()
            yield ("act", read)

    def run(self):
        agents = [self.producer(), self.issuer_a(), self.issuer_b()]
        agents += [self.pds_warp(w) for w in range(WARPS)] + [self.drain_warp(w) for w in range(WARPS)]
        cur = [next(a, None) for a in agents]
        while True:
            choices = []
            for i, c in enumerate(cur):
                if c is None:
                    continue
                if c[0] == "act" or self.bar[c[1]][c[2]].passes(c[3]):
                    choices.append(i)
            if self.loads:
                choices.append("load")
            if self.pipe:
                choices.append("pipe")
            if not choices:
                break
            ch = self.rng.choice(choices)
            if ch == "load":
                st, it = self.loads.pop(self.rng.randrange(len(self.loads)))
                self.stage_holds[st] = it
                self.bar["stage_full"][st].arrive()
            elif ch == "pipe":
                _, _, done = self.pipe.pop(0)  # the tensor core completes in issue order
                done()
            else:
                c = cur[ch]
                if c[0] == "wait":
                    got = self.bar[c[1]][c[2]].completed
                    if got != c[4]:
                        self.err(f"wait on {c[1]}[{c[2]}] passed at completion {got}, meant {c[4]}")
                else:
                    c[1]()
                cur[ch] = next(agents[ch], None)
        finished = all(c is None for c in cur) and not self.loads and not self.pipe
        return self.errors, finished


def sweep(n, runs, seed, **kw):
    rng = random.Random(seed)
    errors, stopped = [], 0
    for _ in range(runs):
        e, finished = Model(n, rng, **kw).run()
        errors += e
        stopped += not finished
    return errors, stopped


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 10])
def test_backward_protocol_is_sound(n):
    errors, stopped = sweep(n, runs=150, seed=n)
    assert stopped == 0 and not errors, (stopped, errors[:5])


@pytest.mark.parametrize("skip,expect", [
    ("tile", "before dQ^T"),                  # P/dS warps: dQ^T(it-2) before the dS^T tile
    ("stage_release", "reloaded"),            # producer: dQ^T(it-3) before the stage
    ("dq_free", "before the drain read"),     # issuer A: the drain before S^T(it+2)
    ("dp_read", "before every warp read"),    # issuer A: the warps before dP^T(it+1)
])
def test_model_catches_a_missing_wait(skip, expect):
    errors, _ = sweep(8, runs=200, seed=1, skip=(skip,))
    assert any(expect in e for e in errors), errors[:3]
