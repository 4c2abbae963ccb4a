"""Host model of the forward kernel's K/V ring and its parity waits.

The forward streams K and V tiles through a ring of shared-memory slots.  A
slot's "full" mbarrier completes once per fill, and a waiter tests it by
phase parity, which tells fill n of the slot from fill n-1 but not from fill
n-2.  A wait is therefore sound only if the waiter knows that fill n-1 of
the slot is complete when it tests for fill n.

This model runs the producer (fills in ring order, each slot refilled once
its previous tile is released), the two MMA issuers taking strict turns
(issuer t's group for step s reads V_t(s-1) and K_t(s) and releases them
when its products complete), and the asynchronous completions (loads and
products land in any order), under random schedules.  It checks every
passed full-wait against the fill the issuer meant, and that every schedule
runs to the end.  Ring sizes are those of the kernel instances (5 slots at
d = 128 bf16, 9 at d = 64) and a few more.

Without head pairing both issuers read every tile, so each waits for every
position in order; with pairing a step's four tiles (K of both heads, then V
of both) each have one reader, and the kernel waits for a group's K/V only
after the issuer has the turn.  The model finds the stale fill when a paired
issuer waits before the turn (what the kernel once did) on the five-slot
ring, and none otherwise.  With five slots and four tiles a step, the slot
of tile 0's next K last held tile 1's V of the step before, which tile 1
reads only in the group after tile 0's; from six slots on, every slot's
previous tile was read by a group already issued, so the earlier order was
sound there too.
"""
import random

import pytest


class Barrier:
    """An mbarrier reduced to what the waits use: completed phases."""

    def __init__(self, count):
        self.count = count
        self.pending = 0
        self.completed = 0

    def arrive(self):
        self.pending += 1
        if self.pending == self.count:
            self.pending = 0
            self.completed += 1

    def test_parity(self, parity):
        # try_wait.parity(p) succeeds once the phase of parity p has
        # completed: the barrier's current phase bit differs from p
        return (self.completed & 1) != parity


def run(ring, paired, wait_after_turn, chunks, rng):
    """One random schedule over chunks of the given step counts (a CTA's
    items, or parts of items, in turn).  Returns (stale_waits, finished)."""
    heads = 2 if paired else 1
    per_step = 2 * heads                     # K of each head, then V of each
    n_pos = per_step * sum(chunks)
    # every issuer walks the same groups: chunk c's groups s = 0 .. chunks[c],
    # group s reading V(s-1) and K(s) of the chunk
    groups = [(c, s) for c in range(len(chunks)) for s in range(chunks[c] + 1)]
    base = [per_step * sum(chunks[:c]) for c in range(len(chunks))]
    full = [Barrier(1) for _ in range(ring)]
    empty = [Barrier(2) for _ in range(ring)]  # two releases per fill either way

    def pos_k(t, c, s):
        return base[c] + per_step * s + (t if paired else 0)

    def pos_v(t, c, s):
        return base[c] + per_step * s + heads + (t if paired else 0)

    # producer state
    prod_next = 0
    loads_in_flight = []                     # positions whose fill has not landed
    # issuer state: index into `groups`
    group = [0, 0]
    kv_idx = [0, 0]                          # the group's K/V waits passed so far
    turn = 0
    mma_in_flight = []                       # (tile, positions) whose products have not completed
    stale = 0

    def needs(t, g):
        c, s = groups[g]
        ps = []
        if s >= 1:
            ps.append(pos_v(t, c, s - 1))
        if s < chunks[c]:
            ps.append(pos_k(t, c, s))
        return ps

    def kv_done(t):
        return kv_idx[t] == len(needs(t, group[t]))

    def kv_ready(t):
        # the group's next wait (V(s-1), then K(s), as issued) would pass
        p = needs(t, group[t])[kv_idx[t]]
        return full[p % ring].test_parity((p // ring) & 1)

    def pass_kv(t):
        nonlocal stale
        p = needs(t, group[t])[kv_idx[t]]
        if full[p % ring].completed != p // ring + 1:  # passed on an earlier fill: a stale tile
            stale += 1
        kv_idx[t] += 1

    while True:
        actions = []
        # producer: next position, once its slot's previous fill is released
        if prod_next < n_pos:
            slot, n = prod_next % ring, prod_next // ring
            if n == 0 or empty[slot].test_parity((n - 1) & 1):
                actions.append("produce")
        if loads_in_flight:
            actions.append("land")
        if mma_in_flight:
            actions.append("mma_done")
        for t in (0, 1):
            if group[t] == len(groups):
                continue
            if not kv_done(t) and (not wait_after_turn or turn == t) and kv_ready(t):
                actions.append(("kv", t))
            if kv_done(t) and turn == t:
                actions.append(("issue", t))
        if not actions:
            break
        a = rng.choice(actions)
        if a == "produce":
            loads_in_flight.append(prod_next)
            prod_next += 1
        elif a == "land":
            p = loads_in_flight.pop(rng.randrange(len(loads_in_flight)))
            full[p % ring].arrive()
        elif a == "mma_done":
            t, ps = mma_in_flight.pop(rng.randrange(len(mma_in_flight)))
            for p in ps:
                for _ in range(2 if paired else 1):
                    empty[p % ring].arrive()
        elif a[0] == "kv":
            pass_kv(a[1])
        else:  # issue the group, hand over the turn
            t = a[1]
            mma_in_flight.append((t, needs(t, group[t])))
            group[t] += 1
            kv_idx[t] = 0
            turn = 1 - t
    finished = group[0] == len(groups) and group[1] == len(groups) and prod_next == n_pos
    return stale, finished


def sweep(ring, paired, wait_after_turn, runs=300, chunks=(12,), seed=0):
    """(stale waits, schedules that stopped before the end) over random schedules."""
    rng = random.Random(seed)
    stale = stopped = 0
    for _ in range(runs):
        s, finished = run(ring, paired, wait_after_turn, list(chunks), rng)
        stale += s
        stopped += not finished
    return stale, stopped


@pytest.mark.parametrize("ring", [5, 6, 7, 9])
def test_unpaired_waits_before_the_turn_are_sound(ring):
    assert sweep(ring, paired=False, wait_after_turn=False) == (0, 0)


@pytest.mark.parametrize("ring", [5, 6, 7, 9])
def test_paired_waits_after_the_turn_are_sound(ring):
    assert sweep(ring, paired=True, wait_after_turn=True) == (0, 0)


def test_paired_waits_before_the_turn_can_take_a_stale_fill():
    # the ordering the kernel had before, on the d = 128 ring: the model must
    # find the stale fill
    stale, _ = sweep(5, paired=True, wait_after_turn=False)
    assert stale > 0


@pytest.mark.parametrize("ring", [6, 7, 9, 13])
def test_paired_waits_before_the_turn_are_sound_from_six_slots(ring):
    assert sweep(ring, paired=True, wait_after_turn=False) == (0, 0)


@pytest.mark.parametrize("chunks", [(1, 1, 1, 1, 1, 1), (3, 8, 2), (5, 1, 7)])
@pytest.mark.parametrize("ring", [5, 9])
def test_chunk_boundaries(ring, chunks):
    # a CTA's chunks in turn (the first and last group of a chunk read one
    # tile each); paired items under the causal mask with at most 128 rows
    # take one step each
    assert sweep(ring, paired=False, wait_after_turn=False, runs=150, chunks=chunks) == (0, 0)
    assert sweep(ring, paired=True, wait_after_turn=True, runs=150, chunks=chunks) == (0, 0)
