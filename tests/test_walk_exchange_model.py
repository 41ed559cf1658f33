"""Host model of the greedy walk's per-step exchange (the walk from the root, one cluster of
eight CTAs per sequence). Every warp of every CTA writes its (max, index) pair into its own
CTA's slot of the step's parity, all threads meet at one cluster barrier, then every warp
reads all 8 x 16 pairs and goes on to the next step without another barrier. A slot of one
parity is written again two steps later.

The model runs the 128 warps as interleaved programs under a random scheduler. The barrier
admits no warp past step k's barrier until all have arrived. It checks that no slot is
overwritten while a reader of the step that wrote it has yet to read it, and that every warp
reads the values of its own step. The same schedule with the parity buffer reduced to one
slot fails that check: the parity is what makes one barrier per step enough."""

import random

CTAS, WARPS = 8, 16


def _run(steps, parities, seed):
    rng = random.Random(seed)
    n = CTAS * WARPS
    slot = {}                       # (parity, warp id) -> step whose value it holds
    pc = [0] * n                    # per warp: position in its program
    arrived = [0] * (steps + 1)     # warps arrived at each step's barrier
    reads_left = {}                 # (step, writer) -> readers still to read it
    bad = []

    def program(w):
        for k in range(steps):
            yield ("write", k)
            yield ("arrive", k)
            yield ("wait", k)
            for r in range(n):
                yield ("read", k, r)

    progs = [program(w) for w in range(n)]
    pending = [next(p) for p in progs]
    live = set(range(n))
    while live:
        runnable = [w for w in live if not (pending[w][0] == "wait" and arrived[pending[w][1]] < n)]
        w = rng.choice(runnable)
        op = pending[w]
        if op[0] == "write":
            k = op[1]
            key = (k % parities, w)
            old = slot.get(key)
            if old is not None and reads_left.get((old, w), 0) > 0:
                bad.append(("overwrite", w, old, k))
            slot[key] = k
            reads_left[(k, w)] = n
        elif op[0] == "arrive":
            arrived[op[1]] += 1
        elif op[0] == "read":
            k, r = op[1], op[2]
            if slot.get((k % parities, r)) != k:
                bad.append(("stale", w, r, k))
            reads_left[(k, r)] -= 1
        try:
            pending[w] = next(progs[w])
        except StopIteration:
            live.discard(w)
    return bad


def test_two_parities_one_barrier_per_step():
    for seed in range(3):
        assert _run(4, 2, seed) == []


def test_one_parity_would_not_suffice():
    assert any(_run(3, 1, seed) for seed in range(3))
