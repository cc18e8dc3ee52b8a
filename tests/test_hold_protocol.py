"""The slot protocols of the persistent row rings, simulated on the CPU: the register-held
final-aggregation kernel (full_hold_kernel in fullring.cu) and, further down, the per-sublayer
backward (backward_ring_kernel in backward.cu, which frees g_y's slot before the sources').

One copy thread streams the CTA's rows, source by source, into a ring of SB slots (each slot's
`full` barrier completes when its copy lands; a refill waits on its `empty` barrier). W compute
warps take every row in order: pass 1 waits on each source's slot and reads it; a source below
R (the sources held in registers) is released at once, the others keep their slot; a barrier
over the W warps ends pass 1; pass 2 reads the kept slots again and releases them.  Copy
landings and the warps' work take random times.

Checked: no slot is refilled while a warp still has to read it (the pass-2 re-read sees its own
source), every wait is satisfied by the phase it was meant for, and every run ends.  A variant
that also releases the kept slots in pass 1 is caught, which shows the checks can fail."""
import random

import pytest


class _Bar:
    def __init__(self, count):
        self.count, self.pending, self.phase = count, count, 0

    def arrive(self):
        assert self.pending > 0
        self.pending -= 1
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


def simulate(SB, n, R, rows, W, seed, release_kept_early=False):
    rng = random.Random(seed)
    full = [_Bar(1) for _ in range(SB)]
    empty = [_Bar(W) for _ in range(SB)]
    content = [None] * SB
    events, now = [], [0]

    def later(dt, fn):
        events.append((now[0] + dt, rng.random(), fn))

    def copy_thread():
        g = 0
        for r in range(rows):
            for j in range(n):
                s = g % SB
                if g >= SB:
                    yield ("wait", empty[s], ((g // SB) & 1) ^ 1)
                    _check(empty[s].phase == g // SB, "refill passed on the wrong phase")
                content[s] = (r, j)
                later(rng.randint(1, 60), lambda s=s: full[s].arrive())
                g += 1
                yield None

    def warp(w):
        g = 0
        for r in range(rows):
            kept = []
            for j in range(n):
                s = g % SB
                yield ("wait", full[s], (g // SB) & 1)
                _check(content[s] == (r, j), f"warp {w} read {content[s]} for {(r, j)}")
                yield ("sleep", rng.randint(0, 8))
                _check(content[s] == (r, j), "slot overwritten during its pass-1 read")
                if j < R or release_kept_early:
                    empty[s].arrive()
                if j >= R:
                    kept.append((s, j))
                g += 1
            yield ("barrier", r)
            yield ("sleep", rng.randint(0, 20))         # statistics
            for s, j in kept:                           # pass 2 over the kept slots
                _check(content[s] == (r, j), f"kept slot of {(r, j)} refilled before pass 2")
                yield ("sleep", rng.randint(0, 6))
                _check(content[s] == (r, j), "kept slot refilled during its pass-2 read")
                if not release_kept_early:
                    empty[s].arrive()
            yield ("sleep", rng.randint(0, 15))         # stores

    agents = {"copy": copy_thread()}
    agents.update({w: warp(w) for w in range(W)})
    state = {k: None for k in agents}
    arrived = {}
    done = set()
    while len(done) < len(agents):
        progressed = False
        for name, gen in agents.items():
            if name in done:
                continue
            st = state[name]
            if st is None:
                ready = True
            elif st[0] == "sleep":
                ready = now[0] >= st[1]
            elif st[0] == "barrier":
                ready = arrived.get(st[1], 0) >= W
            else:
                ready = st[1].passed(st[2])
            if not ready:
                continue
            progressed = True
            try:
                nxt = next(gen)
            except StopIteration:
                done.add(name)
                continue
            if nxt is not None and nxt[0] == "sleep":
                nxt = ("sleep", now[0] + nxt[1])
            elif nxt is not None and nxt[0] == "barrier":
                arrived[nxt[1]] = arrived.get(nxt[1], 0) + 1
            state[name] = nxt
        if progressed:
            continue
        wakes = [v[1] for k, v in state.items() if k not in done and v and v[0] == "sleep"]
        _check(events or wakes, "deadlock")
        events.sort(key=lambda e: (e[0], e[1]))
        if events and (not wakes or events[0][0] <= min(wakes)):
            t, _, fn = events.pop(0)
            now[0] = max(now[0], t)
            fn()
        else:
            now[0] = max(now[0], min(wakes))


@pytest.mark.parametrize("n", [1, 7, 8, 9, 10])
@pytest.mark.parametrize("extra", [2, 5])
def test_hold_ring_is_safe(n, extra):
    """The kernel's ring has at least n + 2 slots (15 at the final aggregation's n = 10)."""
    for seed in range(4):
        simulate(SB=n + extra, n=n, R=8, rows=12, W=4, seed=seed)


def test_hold_ring_final_aggregation_shape():
    for seed in range(3):
        simulate(SB=15, n=10, R=8, rows=20, W=14, seed=seed)


def test_releasing_kept_slots_early_is_caught():
    caught = 0
    for seed in range(8):
        try:
            simulate(SB=12, n=10, R=8, rows=12, W=4, seed=seed, release_kept_early=True)
        except _Violation:
            caught += 1
    assert caught > 0


def simulate_backward(SB, n, rows, W, seed, release_sources_early=False):
    """The ring of the per-sublayer backward (backward_ring_kernel in backward.cu): per row the
    copy thread streams the n sources and then g_y; the warps wait for the sources in pass 1,
    for g_y in pass 2 and release g_y there (out of ring order), re-read the sources in passes
    2 to 4 (a barrier between passes) and release each source in pass 4 after storing its
    gradient."""
    rng = random.Random(seed)
    full = [_Bar(1) for _ in range(SB)]
    empty = [_Bar(W) for _ in range(SB)]
    content = [None] * SB
    events, now = [], [0]

    def later(dt, fn):
        events.append((now[0] + dt, rng.random(), fn))

    def copy_thread():
        g = 0
        for r in range(rows):
            for j in range(n + 1):  # j == n: g_y
                s = g % SB
                if g >= SB:
                    yield ("wait", empty[s], ((g // SB) & 1) ^ 1)
                    _check(empty[s].phase == g // SB, "refill passed on the wrong phase")
                content[s] = (r, j)
                later(rng.randint(1, 60), lambda s=s: full[s].arrive())
                g += 1
                yield None

    def warp(w):
        g = 0
        for r in range(rows):
            b0 = g % SB
            slot = [(b0 + j) % SB for j in range(n + 1)]
            for j in range(n):                              # pass 1
                yield ("wait", full[slot[j]], ((g + j) // SB) & 1)
                _check(content[slot[j]] == (r, j), f"pass 1 read {content[slot[j]]}")
                yield ("sleep", rng.randint(0, 5))
                if release_sources_early:
                    empty[slot[j]].arrive()
            yield ("barrier", (r, 1))
            for j in range(n):                              # pass 2: h
                _check(content[slot[j]] == (r, j), "source refilled before pass 2")
            yield ("wait", full[slot[n]], ((g + n) // SB) & 1)
            _check(content[slot[n]] == (r, n), "g_y slot holds the wrong row")
            yield ("sleep", rng.randint(0, 5))
            empty[slot[n]].arrive()                         # g_y released in pass 2
            yield ("barrier", (r, 2))
            for j in range(n):                              # pass 3: g_h . v_j
                _check(content[slot[j]] == (r, j), "source refilled before pass 3")
                yield ("sleep", rng.randint(0, 3))
            yield ("barrier", (r, 3))
            for j in range(n):                              # pass 4: dv_j, release
                _check(content[slot[j]] == (r, j), "source refilled before pass 4")
                yield ("sleep", rng.randint(0, 4))
                if not release_sources_early:
                    empty[slot[j]].arrive()
            g += n + 1

    agents = {"copy": copy_thread()}
    agents.update({w: warp(w) for w in range(W)})
    state = {k: None for k in agents}
    arrived = {}
    done = set()
    while len(done) < len(agents):
        progressed = False
        for name, gen in agents.items():
            if name in done:
                continue
            st = state[name]
            if st is None:
                ready = True
            elif st[0] == "sleep":
                ready = now[0] >= st[1]
            elif st[0] == "barrier":
                ready = arrived.get(st[1], 0) >= W
            else:
                ready = st[1].passed(st[2])
            if not ready:
                continue
            progressed = True
            try:
                nxt = next(gen)
            except StopIteration:
                done.add(name)
                continue
            if nxt is not None and nxt[0] == "sleep":
                nxt = ("sleep", now[0] + nxt[1])
            elif nxt is not None and nxt[0] == "barrier":
                arrived[nxt[1]] = arrived.get(nxt[1], 0) + 1
            state[name] = nxt
        if progressed:
            continue
        wakes = [v[1] for k, v in state.items() if k not in done and v and v[0] == "sleep"]
        _check(events or wakes, "deadlock")
        events.sort(key=lambda e: (e[0], e[1]))
        if events and (not wakes or events[0][0] <= min(wakes)):
            t, _, fn = events.pop(0)
            now[0] = max(now[0], t)
            fn()
        else:
            now[0] = max(now[0], min(wakes))


@pytest.mark.parametrize("n", [1, 2, 9, 10])
@pytest.mark.parametrize("extra", [3, 5])
def test_backward_ring_is_safe(n, extra):
    """The backward's ring has at least n + 3 slots (15 at n = 10, d = 7168)."""
    for seed in range(4):
        simulate_backward(SB=n + extra, n=n, rows=10, W=4, seed=seed)


def test_backward_ring_final_shape():
    for seed in range(3):
        simulate_backward(SB=15, n=10, rows=12, W=14, seed=seed)


def test_backward_releasing_sources_before_pass_4_is_caught():
    caught = 0
    for seed in range(8):
        try:
            simulate_backward(SB=13, n=10, rows=10, W=4, seed=seed, release_sources_early=True)
        except _Violation:
            caught += 1
    assert caught > 0
