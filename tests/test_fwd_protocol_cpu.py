"""Host model of the forward kernel's barriers and buffers.

One CTA of the forward runs a chunk of key-tile steps per item, with two
query tiles t = 0, 1 (two tiles of one head, or one tile of each of two
paired heads).  Workers: the producer (each tile's Q once per chunk in which
the tile has keys, then every step's K and V through a ring of slots), two
MMA issuers taking strict turns (issuer t's group for step s is
O_t += P_t(s-1) V(s-1) and S_t(s) = Q_t K(s)^T), and four softmax warps per
tile (S_t(j) in, P_t(j) written over it, O_t rescaled when a row's reference
moves, and the epilogue reading O_t).  Products complete in issue order,
loads in any order; a tile's chunk may end before the chunk's last step
(causal), and then its issuer releases the K/V tiles it skips.

The model runs the kernel's programs with the kernel's order of waits under
random schedules, and checks that every parity wait passes on the
completion it means, that every read finds the data of its own step and
chunk (Q, K, V, S, P, and O accumulated exactly through the previous step
before a rescale or the epilogue), that no buffer is overwritten while
needed (Q before the chunk's last S of the tile, O before the previous
chunk's epilogue has read it), and that no schedule stalls.  Dropping the
producer's q_empty wait or the issuers' p_ready wait is caught.  Dropping
the o_free wait is not: the first P.V of a chunk also waits for the
chunk's first P, which each softmax warp writes only after its epilogue of
the previous chunk has read O, so o_free only restates that order.
"""
import random

import pytest

WARPS = 4  # softmax warps per tile


class Barrier:
    def __init__(self, count, initial=0):
        self.count, self.pending, self.completed = count, 0, initial

    def arrive(self, k=1):
        for _ in range(k):
            self.pending += 1
            if self.pending == self.count:
                self.pending, self.completed = 0, self.completed + 1

    def passes(self, parity):
        return (self.completed & 1) != parity


class Model:
    def __init__(self, chunks, paired, ring, rng, skip=()):
        # chunks: (kb, ke, ne0, ne1): the chunk's steps [kb, ke), tile t has keys in [kb, ne_t)
        self.chunks, self.paired, self.ring, self.rng, self.skip = chunks, paired, ring, rng, set(skip)
        self.kvps = 4 if paired else 2
        self.rel = 2 if paired else 1
        B = Barrier
        self.q_full = [B(1), B(1)]
        self.q_empty = [B(1), B(1)]
        self.s_full = [B(1), B(1)]
        self.p_ready = [B(WARPS), B(WARPS)]
        self.o_done = [B(1), B(1)]
        self.o_free = [B(WARPS), B(WARPS)]
        self.turn = [B(1, initial=1), B(1)]   # tile 0 takes the first turn
        self.kv_full = [B(1) for _ in range(ring)]
        self.kv_empty = [B(2) for _ in range(ring)]
        self.errors = []
        self.loads, self.pipe = [], []
        self.q_holds = [None, None]                       # chunk whose Q_t is in shared memory
        self.kv_holds = [None] * ring                     # position whose tile is in the slot
        self.sbuf = [[None] * WARPS, [None] * WARPS]      # per tile and warp quadrant: (kind, chunk, step)
        self.o = [None, None]                             # (chunk, last step accumulated) of O_t
        self.o_read = [set(), set()]                      # chunks whose epilogue read O_t
        self.s_done = [set(), set()]                      # (chunk, step) of S_t complete
        self.base = []
        pos = 0
        for kb, ke, _, _ in chunks:
            self.base.append(pos - self.kvps * kb)
            pos += self.kvps * (ke - kb)
        self.n_pos = pos

    def err(self, m):
        self.errors.append(m)

    def ne(self, c, t):
        return self.chunks[c][2 + t]

    def pos(self, c, t, kind, j):
        # K then V of each step (unpaired), or K of both heads then V of both
        heads = 2 if self.paired else 1
        return self.base[c] + self.kvps * j + (heads if kind == "V" else 0) + (t if self.paired else 0)

    def wait(self, bar, parity, meant, what):
        return ("wait", bar, parity, meant, what)

    # -- programs ----------------------------------------------------------
    def producer(self):
        q_loads = [0, 0]
        n = 0
        for c, (kb, ke, _, _) in enumerate(self.chunks):
            for t in (0, 1):
                if self.ne(c, t) <= kb:
                    continue
                if "q_empty" not in self.skip:
                    yield self.wait(self.q_empty[t], (q_loads[t] & 1) ^ 1, q_loads[t], f"q_empty[{t}]")
                def load_q(c=c, t=t):
                    prev = [cc for cc in range(c) if self.ne(cc, t) > self.chunks[cc][0]]
                    if prev:
                        pc = prev[-1]
                        need = {(pc, j) for j in range(self.chunks[pc][0], self.ne(pc, t))}
                        if not need <= self.s_done[t]:
                            self.err(f"Q_{t} reloaded for chunk {c} before chunk {pc}'s S products were done")
                    self.loads.append(("q", t, c))
                yield ("act", load_q)
                q_loads[t] += 1
            heads = 2 if self.paired else 1
            for j in range(kb, ke):
                for k in range(2 * heads):
                    slot, fill = n % self.ring, n // self.ring
                    yield self.wait(self.kv_empty[slot], (fill & 1) ^ 1, fill, f"kv_empty[{slot}]")
                    def load_kv(n=n):
                        self.loads.append(("kv", n % self.ring, n))
                    yield ("act", load_kv)
                    n += 1

    def issuer(self, t):
        q_uses = pr = turns = 0
        of = 1
        for c, (kb, ke, _, _) in enumerate(self.chunks):
            ne = self.ne(c, t)
            if ne > kb:
                yield self.wait(self.q_full[t], q_uses & 1, q_uses + 1, f"q_full[{t}]")
                q_uses += 1
            for s in range(kb, ke + 1):
                do_pv = kb <= s - 1 < ne
                do_s = s < ne
                cv = self.pos(c, t, "V", s - 1) if s - 1 >= kb else None
                ck = self.pos(c, t, "K", s) if s < ke else None

                def kv_waits():
                    if do_pv:
                        yield self.wait(self.kv_full[cv % self.ring], (cv // self.ring) & 1, cv // self.ring + 1, "kv_full V")
                    if do_s:
                        yield self.wait(self.kv_full[ck % self.ring], (ck // self.ring) & 1, ck // self.ring + 1, "kv_full K")

                if not self.paired:
                    yield from kv_waits()
                if do_pv:
                    if s == kb + 1 and "o_free" not in self.skip:
                        yield self.wait(self.o_free[t], of, None, f"o_free[{t}]")
                        of ^= 1
                    if "p_ready" not in self.skip:
                        yield self.wait(self.p_ready[t], pr & 1, pr + 1, f"p_ready[{t}]")
                    pr += 1
                yield self.wait(self.turn[t], turns & 1, turns + 1, f"turn[{t}]")
                turns += 1
                if self.paired:
                    yield from kv_waits()

                def issue(c=c, s=s, do_pv=do_pv, do_s=do_s, cv=cv, ck=ck, ne=ne, kb=kb):
                    if do_pv:
                        for w in range(WARPS):
                            if self.sbuf[t][w] != ("P", c, s - 1):
                                self.err(f"P.V_{t}({c},{s - 1}) issued on {self.sbuf[t][w]}")
                        if self.kv_holds[cv % self.ring] != cv:
                            self.err(f"P.V_{t}({c},{s - 1}) issued on slot holding position {self.kv_holds[cv % self.ring]}")
                    if do_s:
                        if self.q_holds[t] != c:
                            self.err(f"S_{t}({c},{s}) issued on Q of chunk {self.q_holds[t]}")
                        if self.kv_holds[ck % self.ring] != ck:
                            self.err(f"S_{t}({c},{s}) issued on slot holding position {self.kv_holds[ck % self.ring]}")
                    def done():
                        if do_pv:
                            if s == kb + 1:
                                prev = [cc for cc in range(c) if self.ne(cc, t) > self.chunks[cc][0]]
                                if prev and prev[-1] not in self.o_read[t]:
                                    self.err(f"O_{t} overwritten by chunk {c} before chunk {prev[-1]}'s epilogue read it")
                                self.o[t] = (c, s - 1)
                            else:
                                if self.o[t] != (c, s - 2):
                                    self.err(f"O_{t} accumulated step {s - 1} onto {self.o[t]}")
                                self.o[t] = (c, s - 1)
                            self.kv_empty[cv % self.ring].arrive(self.rel)
                        if do_s:
                            for w in range(WARPS):
                                self.sbuf[t][w] = ("S", c, s)
                            self.s_done[t].add((c, s))
                            self.kv_empty[ck % self.ring].arrive(self.rel)
                            self.s_full[t].arrive()
                            if s == ne - 1:
                                self.q_empty[t].arrive()
                        if do_pv and not do_s:
                            self.o_done[t].arrive()
                    self.pipe.append(done)
                    self.turn[1 - t].arrive()
                yield ("act", issue)
                # K/V tiles this tile skips (past its keys) are released unread
                for p, used in ((cv, do_pv), (ck, do_s)):
                    if p is not None and not used:
                        yield self.wait(self.kv_full[p % self.ring], (p // self.ring) & 1, p // self.ring + 1, "kv_full skip")
                        def release(p=p):
                            self.kv_empty[p % self.ring].arrive(self.rel)
                        yield ("act", release)

    def softmax(self, t, w):
        s_par = od = 0
        n_s = 0
        for c, (kb, ke, _, _) in enumerate(self.chunks):
            ne = self.ne(c, t)
            if ne <= kb:
                continue
            for j in range(kb, ne):
                yield self.wait(self.s_full[t], s_par, n_s + 1, f"s_full[{t}]")
                s_par ^= 1
                n_s += 1
                def tile(c=c, j=j, kb=kb):
                    if self.sbuf[t][w] != ("S", c, j):
                        self.err(f"softmax {t}.{w} read S({c},{j}) from {self.sbuf[t][w]}")
                    if j > kb and self.rng.random() < 0.5:  # a row's reference moved: rescale O
                        if self.o[t] != (c, j - 1):
                            self.err(f"softmax {t}.{w} rescaled O({c}) holding {self.o[t]} at step {j}")
                    self.sbuf[t][w] = ("P", c, j)
                    self.p_ready[t].arrive()
                yield ("act", tile)
            yield self.wait(self.o_done[t], od, None, f"o_done[{t}]")
            od ^= 1
            def epilogue(c=c, ne=ne):
                if self.o[t] != (c, ne - 1):
                    self.err(f"epilogue {t}.{w} of chunk {c} read O holding {self.o[t]}")
                self._o_reads = getattr(self, "_o_reads", {})
                self._o_reads.setdefault((t, c), set()).add(w)
                if len(self._o_reads[(t, c)]) == WARPS:
                    self.o_read[t].add(c)
                self.o_free[t].arrive()
            yield ("act", epilogue)

    def run(self):
        agents = [self.producer(), self.issuer(0), self.issuer(1)]
        agents += [self.softmax(t, w) for t in (0, 1) for w in range(WARPS)]
        cur = [next(a, None) for a in agents]
        while True:
            ch = []
            for i, c in enumerate(cur):
                if c is not None and (c[0] == "act" or c[1].passes(c[2])):
                    ch.append(i)
            if self.loads:
                ch.append("load")
            if self.pipe:
                ch.append("pipe")
            if not ch:
                break
            x = self.rng.choice(ch)
            if x == "load":
                kind, a, b = self.loads.pop(self.rng.randrange(len(self.loads)))
                if kind == "q":
                    self.q_holds[a] = b
                    self.q_full[a].arrive()
                else:
                    self.kv_holds[a] = b
                    self.kv_full[a].arrive()
            elif x == "pipe":
                self.pipe.pop(0)()
            else:
                c = cur[x]
                if c[0] == "wait":
                    if c[3] is not None and c[1].completed != c[3]:
                        self.err(f"wait on {c[4]} passed at completion {c[1].completed}, meant {c[3]}")
                else:
                    c[1]()
                cur[x] = next(agents[x], None)
        return self.errors, all(c is None for c in cur) and not self.loads and not self.pipe


def random_chunks(rng, paired, causal):
    chunks, kb = [], 0
    for _ in range(rng.randint(1, 4)):
        n = rng.randint(1, 6)
        kb = rng.randint(0, 2) if rng.random() < 0.5 else 0  # a part of an item may start inside it
        ke = kb + n
        if causal and not paired:
            ne0 = rng.randint(kb, ke)                 # tile 0 ends at or before tile 1
            ne1 = rng.randint(max(ne0, kb + 1), ke)
        else:
            ne0 = ne1 = ke
        chunks.append((kb, ke, ne0, ne1))
    return chunks


@pytest.mark.parametrize("paired,causal,ring", [
    (False, False, 5), (False, True, 5), (False, False, 9), (False, True, 9), (True, False, 5), (True, False, 9),
])
def test_forward_protocol_is_sound(paired, causal, ring):
    rng = random.Random(hash((paired, causal, ring)) & 0xffff)
    for _ in range(120):
        chunks = random_chunks(rng, paired, causal)
        errors, finished = Model(chunks, paired, ring, rng).run()
        assert finished and not errors, (chunks, errors[:4])


@pytest.mark.parametrize("skip,expect", [
    ("q_empty", "reloaded"),   # producer: Q_t of the next chunk over one still read
    ("p_ready", "issued on"),  # issuer: P.V on S instead of P
])
def test_model_catches_a_missing_wait(skip, expect):
    rng = random.Random(5)
    caught = False
    for _ in range(300):
        chunks = random_chunks(rng, False, False)
        errors, _ = Model(chunks, False, 5, rng, skip=(skip,)).run()
        caught |= any(expect in e for e in errors)
    assert caught


def test_o_free_restates_the_p_ready_order():
    rng = random.Random(6)
    for _ in range(200):
        chunks = random_chunks(rng, False, rng.random() < 0.5)
        errors, finished = Model(chunks, False, 5, rng, skip=("o_free",)).run()
        assert finished and not errors, (chunks, errors[:3])
