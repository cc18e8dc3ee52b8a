"""The mbarrier protocol of the tensor-core phase 1 (phase1_tc.cu), simulated on the CPU.

Agents: the copy warp, the MMA warp and 16 compute warps.  Sweep 1 streams the tile through a
ring of SB slots; the two halves of the compute warps take alternate stages and wait only on
their own stages' "full" barriers, the MMA warp takes every stage.  Sweep 2 has its own ring
of SB2 slots over the same memory (MMA warp only) and two accumulators handed between the MMA
warp and all 16 compute warps (dfull / dempty).  Copies and MMA commits complete after random
delays (MMA commits in issue order, as a commit covers every earlier MMA of its thread).

Each barrier is modelled as the hardware counts it: a phase completes when its pending
arrivals reach zero, and a parity wait passes once the phase of that parity is done — so a
wait two phases behind passes on the older completion.  The checks: no slot is refilled while
a reader still uses it, every wait is satisfied by the phase it was meant for, no accumulator
is overwritten while read, sweep 2 never reuses memory a sweep-1 reader still holds, and every
run ends.  An odd sweep-1 slot count breaks them (a half a ring ahead takes the completion two
phases back for its own stage); even counts never do, which is why the kernel's plan rounds
the slot count down to even."""
import random

import pytest


class _Bar:
    def __init__(self, count):
        self.count, self.pending, self.phase = count, count, 0

    def arrive(self, n=1):
        assert n <= self.pending, "more arrivals than the phase expects"
        self.pending -= n
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def passed(self, parity):
        return (self.phase & 1) != parity


class _Violation(AssertionError):
    pass


def _check(cond, what):
    if not cond:
        raise _Violation(what)


def simulate(SB, SB2, nch, nch2, seed):
    rng = random.Random(seed)
    full = [_Bar(1) for _ in range(SB)]
    empty = [_Bar(9) for _ in range(SB)]           # a half's 8 warps + the stage's MMAs
    full2 = [_Bar(1) for _ in range(SB2)]
    empty2 = [_Bar(1) for _ in range(SB2)]         # the stage's MMAs
    dready, aready = _Bar(1), _Bar(16)
    dfull, dempty = [_Bar(1), _Bar(1)], [_Bar(16), _Bar(16)]
    slot, readers = [None] * SB, [set() for _ in range(SB)]
    slot2, readers2 = [None] * SB2, [set() for _ in range(SB2)]
    acc, acc_readers = [None, None], [set(), set()]
    events, now, mma_t, seq = [], [0], [0], [0]

    def later(dt, fn):
        events.append((now[0] + dt, rng.random(), fn))

    def later_mma(dt, fn):
        mma_t[0] = max(mma_t[0], now[0] + dt)
        seq[0] += 1
        events.append((mma_t[0], seq[0] * 1e-9, fn))

    def copy_warp():
        for ib in range(nch):
            bs = ib % SB
            if ib >= SB:
                yield (empty[bs], ((ib // SB) & 1) ^ 1)
                _check(empty[bs].phase == ib // SB, "refill waited on the wrong phase")
            _check(not readers[bs], "slot refilled while read")
            slot[bs] = ib
            later(rng.randint(1, 50), lambda bs=bs: full[bs].arrive())
            yield None
        for s in range(min(SB, nch)):          # drain: every sweep-1 stage consumed
            last = nch - 1 - ((nch - 1 - s) % SB)
            yield (empty[s], (last // SB) & 1)
        for q in range(nch2):
            bs = q % SB2
            if q >= SB2:
                yield (empty2[bs], ((q // SB2) & 1) ^ 1)
            _check(all(not r for r in readers), "sweep 2 reused memory still read")
            _check(not readers2[bs], "sweep-2 slot refilled while read")
            slot2[bs] = q
            later(rng.randint(1, 50), lambda bs=bs: full2[bs].arrive())
            yield None

    def mma_warp():
        for c in range(nch):
            bs = c % SB
            yield (full[bs], (c // SB) & 1)
            _check(slot[bs] == c, "MMA read a slot before its stage landed")
            readers[bs].add("mma")

            def done(bs=bs, c=c):
                readers[bs].discard("mma")
                empty[bs].arrive()
                if c == nch - 1:
                    dready.arrive()
            later_mma(rng.randint(1, 20), done)
            yield None
        yield (aready, 0)
        for q in range(nch2):
            bs, b, use = q % SB2, q & 1, q >> 1
            yield (full2[bs], (q // SB2) & 1)
            _check(slot2[bs] == q, "sweep-2 MMA read a slot before its stage landed")
            if use > 0:
                yield (dempty[b], (use - 1) & 1)
            _check(not acc_readers[b], "accumulator overwritten while read")
            readers2[bs].add("mma")
            acc[b] = q

            def done2(bs=bs, b=b):
                readers2[bs].discard("mma")
                empty2[bs].arrive()
                dfull[b].arrive()
            later_mma(rng.randint(1, 40), done2)
            yield None

    def compute_warp(w):
        for c in range(w >> 3, nch, 2):
            bs = c % SB
            yield (full[bs], (c // SB) & 1)
            _check(slot[bs] == c, "a half read a slot before its stage landed")
            readers[bs].add(w)
            yield ("sleep", rng.randint(0, 10))
            readers[bs].discard(w)
            empty[bs].arrive()
        yield ("barrier", 0)
        yield (dready, 0)
        yield ("barrier", 1)
        _check(all(not r for r in readers), "weights zeroed while the sweep-1 ring is read")
        yield ("sleep", rng.randint(0, 30))
        aready.arrive()
        yield ("barrier", 2)
        for q in range(nch2):
            b = q & 1
            yield (dfull[b], (q >> 1) & 1)
            _check(acc[b] == q, "accumulator read before its stage was done")
            acc_readers[b].add(w)
            yield ("sleep", rng.randint(0, 15))
            acc_readers[b].discard(w)
            dempty[b].arrive()
            yield ("sleep", rng.randint(0, 25))

    agents = {"copy": copy_warp(), "mma": mma_warp()}
    agents.update({w: compute_warp(w) for w in range(16)})
    state = {k: None for k in agents}
    arrived = {}
    finished = set()
    while len(finished) < len(agents):
        progressed = False
        for name, gen in agents.items():
            if name in finished:
                continue
            st = state[name]
            if st is None:
                ready = True
            elif st[0] == "sleep":
                ready = now[0] >= st[1]
            elif st[0] == "barrier":
                ready = arrived.get(st[1], 0) >= 16
            else:
                ready = st[0].passed(st[1])
            if not ready:
                continue
            progressed = True
            try:
                nxt = next(gen)
            except StopIteration:
                finished.add(name)
                continue
            if nxt is not None and nxt[0] == "sleep":
                nxt = ("sleep", now[0] + nxt[1])
            elif nxt is not None and nxt[0] == "barrier":
                arrived[nxt[1]] = arrived.get(nxt[1], 0) + 1
            state[name] = nxt
        if progressed:
            continue
        wakes = [v[1] for k, v in state.items()
                 if k not in finished and v is not None and v[0] == "sleep"]
        _check(events or wakes, "deadlock")
        events.sort(key=lambda e: (e[0], e[1]))
        if events and (not wakes or events[0][0] <= min(wakes)):
            t, _, fn = events.pop(0)
            now[0] = max(now[0], t)
            fn()
        else:
            now[0] = max(now[0], min(wakes))


@pytest.mark.parametrize("SB", [2, 4, 6, 10, 12])
@pytest.mark.parametrize("SB2", [2, 3, 5])
@pytest.mark.parametrize("nch,nch2", [(112, 56), (14, 7), (3, 2), (1, 1)])
def test_even_rings_never_alias(SB, SB2, nch, nch2):
    for seed in range(3):
        simulate(SB, SB2, nch, nch2, seed)


def test_odd_ring_aliases():
    """The failure the even slot count rules out: with 5 sweep-1 slots some schedule lets a
    half take an older completion for its own stage."""
    failures = 0
    for seed in range(6):
        try:
            simulate(5, 5, 112, 56, seed)
        except _Violation:
            failures += 1
    assert failures > 0
