"""Host model of the forward's in-launch merge of split items.

The plan cuts the concatenated key-tile steps of all items into one equal
range per CTA, so a range boundary can fall inside an item: each side then
computes a part (O over its keys and that part's logsumexp) and the parts
meet through one counter per (item, query tile, warp quadrant).  A CTA's
warp handles its chunks in order:

  - a part in the CTA's last chunk reads the counter first: if every other
    part is in, the warp merges without publishing (its own part is still in
    tensor memory); otherwise it publishes its part, counts its arrival, and
    merges if that arrival completed the parts;
  - a part in the CTA's first chunk (when more chunks follow) is published
    at once but its arrival is made at the start of the next chunk (or at
    the end), and the warp merges the item at the end if that arrival
    completed the parts;
  - the merging warp resets the counter for the next launch.

The model cuts random items over random grids exactly as the plan does
(range c = [W c / G, W (c + 1) / G) of W steps), interleaves the CTAs'
actions at random (sequentially consistent: it checks the counting logic,
not the memory ordering, which the fences and acquire loads provide), and
checks that every split item is merged exactly once, by a warp that finds
every other part published, and that every counter is zero afterwards.
A mutation (arriving for the first chunk's part without publishing it
first) must be caught.
"""
import random

import pytest


def plan(steps, grid):
    """Per CTA: its chunks as (item, part_slot or None, last)."""
    start = [0]
    for s in steps:
        start.append(start[-1] + s)
    W = start[-1]
    ctas = []
    for c in range(grid):
        g0, g1 = W * c // grid, W * (c + 1) // grid
        chunks = []
        for item in range(len(steps)):
            lo, hi = max(g0, start[item]), min(g1, start[item + 1])
            if lo < hi:
                part = lo > start[item] or hi < start[item + 1]
                chunks.append([item, part])
        for i, ch in enumerate(chunks):
            ch.append(i == len(chunks) - 1)
        ctas.append(chunks)
    parts = {}
    for c, chunks in enumerate(ctas):
        for item, part, _ in chunks:
            if part:
                parts.setdefault(item, []).append(c)
    return ctas, parts


def warp_program(c, chunks, parts, st, defer_publish_bug=False):
    """One warp quadrant of CTA c; yields actions (callables) in order."""
    count = {k: len(v) for k, v in parts.items()}
    state = {"arrival": -2, "first_item": None, "pend": []}

    def arrive(item):
        old = st["ctr"][item]
        st["ctr"][item] += 1
        return old

    for q, (item, part, last) in enumerate(chunks):
        if state["arrival"] == -1:
            def deferred():
                state["arrival"] = arrive(state["first_item"])
            yield deferred
        if not part:
            continue
        if last:
            outcome = {}
            def check(item=item, outcome=outcome):
                outcome["all_in"] = st["ctr"][item] == count[item] - 1
            yield check
            if outcome["all_in"]:
                state["pend"].append((item, "tmem"))
                continue
            def publish_and_arrive(item=item):
                st["published"].add((item, c))
                if arrive(item) == count[item] - 1:
                    state["pend"].append((item, "tmem"))
            yield publish_and_arrive
        else:  # the first chunk of several: published now, arrival deferred
            def publish(item=item):
                if not defer_publish_bug:
                    st["published"].add((item, c))
                state["arrival"] = -1
                state["first_item"] = item
            yield publish
    if state["arrival"] == -1:
        def final_arrival():
            state["arrival"] = arrive(state["first_item"])
        yield final_arrival
    if state["arrival"] >= 0 and state["arrival"] == count[state["first_item"]] - 1:
        state["pend"].insert(0, (state["first_item"], "slot"))
    for item, own in state["pend"]:
        def merge(item=item, own=own):
            for other in parts[item]:
                if other != c and (item, other) not in st["published"]:
                    st["errors"].append(f"item {item} merged by CTA {c} before CTA {other}'s part was published")
            if own == "slot" and (item, c) not in st["published"]:
                st["errors"].append(f"item {item}: CTA {c} merged its own part from a slot it never wrote")
            st["merges"][item] = st["merges"].get(item, 0) + 1
            st["ctr"][item] = 0
        yield merge


def run(steps, grid, rng, **kw):
    ctas, parts = plan(steps, grid)
    st = {"ctr": {k: 0 for k in parts}, "published": set(), "merges": {}, "errors": []}
    progs = [warp_program(c, chunks, parts, st, **kw) for c, chunks in enumerate(ctas)]
    live = list(range(len(progs)))
    while live:
        i = rng.choice(live)
        action = next(progs[i], None)
        if action is None:
            live.remove(i)
        else:
            action()
    for k in parts:
        if st["merges"].get(k, 0) != 1:
            st["errors"].append(f"item {k} merged {st['merges'].get(k, 0)} times")
        if st["ctr"][k] != 0:
            st["errors"].append(f"item {k}'s counter left at {st['ctr'][k]}")
    return st["errors"], parts


@pytest.mark.parametrize("seed", range(6))
def test_every_split_item_is_merged_once_with_every_part(seed):
    rng = random.Random(seed)
    split = 0
    for _ in range(150):
        steps = [rng.randint(1, 9) for _ in range(rng.randint(1, 12))]
        grid = rng.randint(2, 2 * len(steps) + 3)
        errors, parts = run(steps, grid, rng)
        assert not errors, (steps, grid, errors[:3])
        split += len(parts)
    assert split > 50  # the sweep does cut items


def test_three_and_more_parts():
    # one long item over many CTAs (the decode shape): parts in the middle are
    # a CTA's only chunk, first and last at once
    rng = random.Random(7)
    for grid in range(2, 9):
        errors, parts = run([40], grid, rng)
        assert not errors and len(parts[0]) == grid


def test_model_catches_an_unpublished_part():
    rng = random.Random(3)
    caught = False
    for _ in range(200):
        steps = [rng.randint(2, 9) for _ in range(rng.randint(2, 8))]
        errors, _ = run(steps, rng.randint(3, 12), rng, defer_publish_bug=True)
        caught |= any("before CTA" in e or "never wrote" in e for e in errors)
    assert caught
