"""A discrete-event model of the tensor-core attention CTA's barrier protocol, run on the CPU.

The model mirrors the waits and arrivals of `attn_tc_kernel` (csrc/attn_tc.cu):
- the TMA producer;
- for the FP8 cache, the four converter warps;
- the two MMA-issuing threads;
- the eight softmax warps (four per M-tile).

It runs the asynchronous parts with random, heavy-tailed delays: TMA copies, and MMAs that
complete in issue order per thread. The mbarriers follow the hardware rule: a wait on parity p
passes when the barrier's phase count has the other parity.

Checks, over many random schedules:
- no deadlock;
- every wait passes for the phase it means, not one phase early or late (a parity wait cannot
  tell a barrier two phases behind from a current one);
- no shared-memory stage or TMEM buffer is written while another party reads or writes it.

Two planted mistakes must be caught:
- the first FP8 ring ownership, where the producer also loaded the tree blocks;
- a softmax warp that skips its wait for the previous PV before touching O.
"""

import random

import pytest


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.tx, self.phase = name, count, count, 0, 0

    def arrive(self, tx=0):
        self.tx += tx
        self.pending -= 1
        assert self.pending >= 0, f"arrival overflow on {self.name}"
        self._step()

    def complete_tx(self, n):
        self.tx -= n
        assert self.tx >= 0, self.name
        self._step()

    def _step(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def passed(self, parity):
        return (self.phase & 1) != parity


class Violation(AssertionError):
    pass


def run_cta(npb, ntree, fp8, seed, old_ring=False, skip_pv_wait=False, ntiles=2):
    """One CTA: npb prefix blocks, ntree tree blocks. Raises Violation on any broken check."""
    rnd = random.Random(seed)
    S16 = 3 if fp8 else 4      # bf16 ring stages
    S8 = 3                     # code ring stages (FP8 cache)
    nb = npb + ntree
    heavy = lambda lo, hi: rnd.uniform(lo, hi) * (50 if rnd.random() < 0.05 else 1)
    kvf = [Bar(f"kv_full{i}", 4 if fp8 else 1) for i in range(S16)]
    kve = [Bar(f"kv_empty{i}", ntiles) for i in range(S16)]
    f8f = [Bar(f"f8_full{i}", 1) for i in range(S8)]
    f8e = [Bar(f"f8_empty{i}", 4) for i in range(S8)]
    sf = [[Bar(f"s_full{t}{i}", 1) for i in range(2)] for t in range(ntiles)]
    pf = [Bar(f"p_full{t}", 4) for t in range(ntiles)]
    pv = [Bar(f"pv_done{t}", 1) for t in range(ntiles)]
    events, now, use = [], [0.0], {}
    filled = {}   # (block, part) -> filled

    def later(dt, fn):
        events.append((now[0] + dt, rnd.random(), fn))

    def begin(region, who, kind):
        pa = region.split(".")
        for (r2, w2), k in use.items():
            pb = r2.split(".")
            same_thread_mma = who[:2] in ("qk", "pv") and w2[:2] in ("qk", "pv") and who[2] == w2[2]
            n = min(len(pa), len(pb))
            if not same_thread_mma and pa[:n] == pb[:n] and (k == "w" or kind == "w"):
                raise Violation(f"{region}: {who}/{kind} overlaps {r2} {w2}/{k}")
        use[(region, who)] = kind

    def end(region, who):
        del use[(region, who)]

    def expect(bar, uses_done, what):
        if bar.phase < uses_done:
            raise Violation(f"{what}: {bar.name} passed at phase {bar.phase}, needs {uses_done}")

    mma_done_at = {t: now[0] for t in range(ntiles)}

    def tma(region, bar, tag):
        begin(region, tag, "w")

        def done():
            end(region, tag)
            bar.complete_tx(1)
        later(heavy(1, 20), done)

    def mma(t, reads, writes, tag):
        for r in reads:
            begin(r, tag, "r")
        for w in writes:
            begin(w, tag, "w")
        t_done = max(mma_done_at[t], now[0]) + heavy(0.5, 5)
        mma_done_at[t] = t_done

        def done():
            for r in reads:
                end(r, tag)
            for w in writes:
                end(w, tag)
        events.append((t_done, rnd.random(), done))

    def commit(t, bar):
        events.append((mma_done_at[t] + 1e-9, rnd.random(), bar.arrive))

    def sleep(lo, hi):
        t_end = now[0] + heavy(lo, hi)
        later(t_end - now[0], lambda: None)
        return lambda: now[0] >= t_end

    def producer():
        own = npb if (fp8 and not old_ring) else nb
        for j in range(own):
            if fp8 and j < npb:
                s8 = j % S8
                if j >= 1:
                    yield lambda: f8e[s8].passed(((j // S8) & 1) ^ 1)
                    expect(f8e[s8], j // S8, f"producer, code stage for block {j}")
                f8f[s8].arrive(tx=8)
                for c in range(8):
                    tma(f"f8_{s8}.c{c}", f8f[s8], f"tma{j}.{c}")
            else:
                st = j % S16
                if j >= 1:
                    yield lambda: kve[st].passed(((j // S16) & 1) ^ 1)
                    expect(kve[st], j // S16, f"producer, bf16 stage for block {j}")
                kvf[st].arrive(tx=4)
                for _ in range(kvf[st].count - 1):
                    kvf[st].arrive()
                for c in range(4):
                    tma(f"bf_{st}.t{c}", kvf[st], f"tmab{j}.{c}")
                filled[(j, "all")] = True

    def converter(w):
        for j in range(npb if old_ring else nb):
            st = j % S16
            if j >= S16:
                yield lambda: kve[st].passed(((j // S16) & 1) ^ 1)
                expect(kve[st], j // S16, f"converter {w}, bf16 stage for block {j}")
            if j < npb:
                s8 = j % S8
                yield lambda: f8f[s8].passed((j // S8) & 1)
                expect(f8f[s8], j // S8 + 1, f"converter {w}, codes of block {j}")
                begin(f"f8_{s8}", f"cvt{w}.{j}", "r")
                begin(f"bf_{st}.q{w}", f"cvt{w}.{j}", "w")
                yield sleep(0.5, 4)
                end(f"f8_{s8}", f"cvt{w}.{j}")
                end(f"bf_{st}.q{w}", f"cvt{w}.{j}")
                filled[(j, w)] = True
                kvf[st].arrive()
                f8e[s8].arrive()
            else:
                if w == 0:
                    kvf[st].arrive(tx=4)
                    for c in range(4):
                        tma(f"bf_{st}.t{c}", kvf[st], f"tmat{j}.{c}")
                else:
                    kvf[st].arrive()
                filled[(j, w)] = True

    def is_filled(j):
        return filled.get((j, "all")) or all(filled.get((j, w)) for w in range(4))

    def mma_thread(t):
        def qk(j):
            st = j % S16
            if not is_filled(j):
                raise Violation(f"QK of tile {t} on block {j} before its stage was filled")
            mma(t, [f"bf_{st}"], [f"s{t}{j & 1}"], f"qk{t}.{j}")
            commit(t, sf[t][j & 1])
        yield lambda: kvf[0].passed(0)
        expect(kvf[0], 1, f"MMA {t}, block 0")
        qk(0)
        for j in range(nb):
            if j + 1 < nb:
                st = (j + 1) % S16
                yield lambda: kvf[st].passed(((j + 1) // S16) & 1)
                expect(kvf[st], (j + 1) // S16 + 1, f"MMA {t}, block {j + 1}")
                qk(j + 1)
            yield lambda: pf[t].passed(j & 1)
            expect(pf[t], j + 1, f"MMA {t}, P of block {j}")
            mma(t, [f"bf_{j % S16}", f"s{t}{j & 1}"], [f"o{t}"], f"pv{t}.{j}")
            commit(t, pv[t])
            commit(t, kve[j % S16])

    def softmax(t, w):
        for j in range(nb):
            yield lambda: sf[t][j & 1].passed((j >> 1) & 1)
            expect(sf[t][j & 1], (j >> 1) + 1, f"softmax {t}.{w}, S of block {j}")
            begin(f"s{t}{j & 1}.q{w}", f"sm{t}{w}.{j}", "w")
            if j >= 1 and not skip_pv_wait:
                yield lambda: pv[t].passed((j - 1) & 1)
                expect(pv[t], j, f"softmax {t}.{w}, PV of block {j - 1}")
            begin(f"o{t}.q{w}", f"sm{t}{w}.{j}", "w")    # a possible rescale of its O rows
            yield sleep(0.5, 3)
            end(f"o{t}.q{w}", f"sm{t}{w}.{j}")
            end(f"s{t}{j & 1}.q{w}", f"sm{t}{w}.{j}")
            pf[t].arrive()
        yield sleep(0, 10)
        yield lambda: pv[t].passed((nb - 1) & 1)
        expect(pv[t], nb, f"softmax {t}.{w}, last PV")

    actors = [producer()] + ([converter(w) for w in range(4)] if fp8 else []) + \
        [mma_thread(t) for t in range(ntiles)] + [softmax(t, w) for t in range(ntiles) for w in range(4)]
    waits = [None] * len(actors)
    alive = list(range(len(actors)))

    def step(i):
        try:
            waits[i] = next(actors[i])
        except StopIteration:
            alive.remove(i)

    for i in list(alive):
        step(i)
    while alive:
        progressed = False
        for i in list(alive):
            while i in alive and waits[i]():
                step(i)
                progressed = True
        if not progressed:
            if not events:
                raise Violation(f"deadlock: actors {alive} wait")
            events.sort()
            t, _, fn = events.pop(0)
            now[0] = max(now[0], t)
            fn()
    while events:
        events.sort()
        t, _, fn = events.pop(0)
        now[0] = max(now[0], t)
        fn()


SHAPES = [(1, 1), (3, 1), (4, 1), (5, 2), (9, 1), (40, 2), (0, 3), (7, 0)]


@pytest.mark.parametrize("fp8", [False, True])
def test_committed_protocol_holds(fp8):
    for seed in range(60):
        for npb, ntree in SHAPES:
            if npb + ntree:
                run_cta(npb, ntree, fp8, seed * 1000 + npb * 10 + ntree)


def _caught(**kw):
    bad = 0
    for seed in range(40):
        for npb, ntree in SHAPES:
            if npb + ntree:
                try:
                    run_cta(npb, ntree, True, seed * 1000 + npb * 10 + ntree, **kw)
                except Violation:
                    bad += 1
    return bad


def test_model_catches_the_first_fp8_ring_ownership():
    # the producer also loaded the tree blocks: its wait could pass one phase early
    assert _caught(old_ring=True) > 0


def test_model_catches_a_missing_pv_wait():
    assert _caught(skip_pv_wait=True) > 0
