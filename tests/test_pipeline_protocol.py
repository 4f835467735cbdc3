"""A randomised model of the relocation kernel's mbarrier protocol.

The kernel's roles (one TMA producer, one MMA issuer, two epilogue groups of
four warps, one page-store warp per group) hand shared-memory stages, TMEM
accumulator slots and U buffers to each other through mbarriers whose waits
test only the parity of a phase.
Such a wait is correct only if the waiter never falls two phases behind the
barrier.  The kernel keeps that invariant by construction: stage s belongs to
epilogue group s % 2, each group owns one accumulator slot, and the MMA issuer
observes every stage use and takes part in its release.

This model replays the same protocol under random interleavings and random
copy latencies and fails if any wait succeeds on the wrong phase or the
pipeline deadlocks.  A variant of the older protocol (accumulator slots in one
global order, an MMA issuer that skips unpatched stages) is shown to fail, so
the model does catch the hazard."""
import random

import pytest


class Bar:
    def __init__(self, count):
        self.count, self.pending, self.tx, self.done = count, count, 0, 0

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.done += 1
            self.pending = self.count

    def arrive(self, tx=0):
        assert self.pending > 0, "arrival on a barrier with no pending arrivals"
        self.tx += tx
        self.pending -= 1
        self._maybe_complete()

    def complete_tx(self, n):
        self.tx -= n
        assert self.tx >= 0
        self._maybe_complete()

    def try_wait(self, phase):
        """Hardware semantics: true when the current phase's parity differs from
        the awaited phase's parity.  Checked against the true phase count."""
        ok = (self.done & 1) != (phase & 1)
        if ok and self.done <= phase:
            raise AssertionError(f"wait for phase {phase} passed with only {self.done} phases done")
        return ok


def simulate(seed, items, S, groups=2, n_u=2, old_protocol=False):
    rnd = random.Random(seed)
    tmem = any(m for m, _ in items)
    slots = 4 if old_protocol else groups
    full = [Bar(1) for _ in range(S)]
    # released by the group's store warp (old protocol: by the four epilogue warps) and the MMA issuer
    empty = [Bar((4 if old_protocol else 1) + (1 if (tmem and not old_protocol) else 0)) for _ in range(S)]
    computed = [Bar(4) for _ in range(S)]
    acc_full, acc_empty = [Bar(1) for _ in range(slots)], [Bar(4) for _ in range(slots)]
    u_full, u_empty = [Bar(1) for _ in range(n_u)], [Bar(1) for _ in range(n_u)]
    events, clock = [], [0]

    def later(fn):
        events.append((clock[0] + rnd.randint(1, 30), fn))

    def producer():
        it = uit = 0
        for m, nsub in items:
            if m:
                ub = uit % n_u
                while uit >= n_u and not u_empty[ub].try_wait(uit // n_u - 1):
                    yield
                u_full[ub].arrive(tx=1)
                later(lambda b=ub: u_full[b].complete_tx(1))
                uit += 1
            for _ in range(nsub):
                st = it % S
                while it >= S and not empty[st].try_wait(it // S - 1):
                    yield
                full[st].arrive(tx=1)
                later(lambda s_=st: full[s_].complete_tx(1))
                it += 1
                yield

    def mma():
        it = uit = ait = 0
        cnt = [0] * slots
        for m, nsub in items:
            if old_protocol and not m:
                it += nsub
                continue
            ub = uit % n_u
            if m:
                while not u_full[ub].try_wait(uit // n_u):
                    yield
            for _ in range(nsub):
                st = it % S
                while not full[st].try_wait(it // S):
                    yield
                if m:
                    a = ait % slots if old_protocol else it % groups
                    use = ait // slots if old_protocol else cnt[a]
                    while use >= 1 and not acc_empty[a].try_wait(use - 1):
                        yield
                    later(lambda a_=a: acc_full[a_].arrive())
                    cnt[a] += 1
                    ait += 1
                if not old_protocol:
                    empty[st].arrive()
                it += 1
                yield
            if m:
                later(lambda b=ub: u_empty[b].arrive())
                uit += 1

    def epilogue_warp(g):
        it = ait = gait = 0
        for m, nsub in items:
            for _ in range(nsub):
                mine = it % groups == g
                if not mine:
                    if m:
                        ait += 1
                    it += 1
                    continue
                st = it % S
                while not full[st].try_wait(it // S):
                    yield
                if m:
                    a, use = (ait % slots, ait // slots) if old_protocol else (g, gait)
                    while not acc_full[a].try_wait(use):
                        yield
                    for _ in range(rnd.randint(0, 3)):
                        yield
                    acc_empty[a].arrive()
                    ait += 1
                    gait += 1
                for _ in range(rnd.randint(0, 5)):
                    yield
                (empty if old_protocol else computed)[st].arrive()
                it += 1
                yield

    def store_warp(g):
        it = 0
        for m, nsub in items:
            for _ in range(nsub):
                if it % groups != g:
                    it += 1
                    continue
                st = it % S
                while not computed[st].try_wait(it // S):
                    yield
                for _ in range(rnd.randint(0, 5)):
                    yield
                empty[st].arrive()
                it += 1
                yield

    roles = [producer()] + ([mma()] if tmem else []) + [epilogue_warp(g) for g in range(groups) for _ in range(4)]
    if not old_protocol:
        roles += [store_warp(g) for g in range(groups)]
    live, steps = list(roles), 0
    while live or events:
        steps += 1
        if steps > 1_000_000:
            raise AssertionError("deadlock")
        events.sort(key=lambda e: e[0])
        if events and (not live or rnd.random() < 0.3):
            t, fn = events.pop(0)
            clock[0] = max(clock[0], t)
            fn()
            continue
        r = rnd.choice(live)
        clock[0] += 1
        try:
            next(r)
        except StopIteration:
            live.remove(r)


def random_items(rnd):
    return [(rnd.choice([0, 0, 0, 64]), rnd.choice([1, 2, 4])) for _ in range(rnd.randint(5, 30))]


def test_protocol_never_accepts_a_stale_phase():
    for seed in range(150):
        rnd = random.Random(seed)
        simulate(seed, random_items(rnd), S=rnd.choice([2, 4, 6]), n_u=rnd.choice([1, 2]))


def test_model_catches_the_old_protocol():
    failures = 0
    for seed in range(300):
        rnd = random.Random(seed)
        items = [(rnd.choice([0, 0, 0, 64]), 4) for _ in range(rnd.randint(5, 40))]
        try:
            simulate(seed, items, S=4, groups=3, old_protocol=True)
        except AssertionError:
            failures += 1
    assert failures > 0
