"""A randomised model of the decode-attention block kernel's stage ring
(`block_kernel` in the attention kernels).

One producer warp fills an S-stage ring (barrier full[s]: one expect-tx arrival
by lane 0 plus the copies' bytes); four consumer warps each read every stage and
release it (barrier empty[s], four arrivals).  Both sides keep a stage index s
and a lap parity `par` that flips when s wraps: the producer waits empty[s] for
parity par ^ 1 (on the first lap that is the phase before the barrier's first,
which counts as complete) and the consumers wait full[s] for parity par.  Before
the CTA exits, the producer walks back over the last min(S, issued) stages,
flipping the parity whenever it steps below stage 0, and waits for each of their
copies to land.

The model replays that bookkeeping literally under random interleavings and copy
latencies.  It fails if a consumer reads a stage holding anything but the stage
it expects, a barrier arrival finds no pending arrival, a copy is still in flight
when the CTA exits, or the pipeline deadlocks.  Variants with the drain walk's
parity flip left out, or with the producer not waiting for the consumers, fail."""
import random

import pytest

from test_pipeline_protocol import Bar


def parity_wait(bar, parity):
    """mbarrier try_wait.parity: true once the phase of that parity has completed,
    i.e. when the number of completed phases has the other parity."""
    return (bar.done & 1) != (parity & 1)


def simulate(seed, n_stages_total, S=3, consumers=4, flip_in_drain=True, producer_waits=True):
    rnd = random.Random(seed)
    full, empty = [Bar(1) for _ in range(S)], [Bar(consumers) for _ in range(S)]
    held = [None] * S          # which stage of the share each ring slot holds
    landed = [0]
    issued_total = [0]
    events, clock = [], [0]

    def later(fn):
        events.append((clock[0] + rnd.randint(1, 40), fn))

    def producer():
        s, par, n_issued = 0, 0, 0
        for f in range(n_stages_total):
            if producer_waits:
                while not parity_wait(empty[s], par ^ 1):
                    yield
            full[s].arrive(tx=2)                     # lane 0: expect-tx for the K/V and U copies
            for part in range(2):
                def land(s=s, f=f):
                    held[s] = f
                    landed[0] += 1
                    full[s].complete_tx(1)
                later(land)
            issued_total[0] += 2
            n_issued += 1
            s += 1
            if s == S:
                s, par = 0, par ^ 1
            yield
        # drain: the last min(S, n_issued) stages, newest first
        for _ in range(min(S, n_issued)):
            s -= 1
            if s < 0:
                s = S - 1
                if flip_in_drain:
                    par ^= 1
            while not parity_wait(full[s], par):
                yield

    def consumer():
        s, par = 0, 0
        for f in range(n_stages_total):
            while not parity_wait(full[s], par):
                yield
            for _ in range(rnd.randint(1, 4)):      # ldmatrix reads of the stage
                assert held[s] == f, f"slot {s} holds stage {held[s]}, a consumer expected {f}"
                yield
            empty[s].arrive()
            s += 1
            if s == S:
                s, par = 0, par ^ 1
            yield

    roles = [producer()] + [consumer() for _ in range(consumers)]
    live, steps = list(roles), 0
    while live:
        steps += 1
        if steps > 20_000 + 5_000 * n_stages_total:   # a wait loop keeps yielding: a deadlock shows as the limit
            raise AssertionError("deadlock")
        events.sort(key=lambda e: e[0])
        if events and rnd.random() < 0.3:
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
            if r is roles[0]:
                # the producer warp exits only after its drain: all its copies must have landed
                if landed[0] != issued_total[0]:
                    raise AssertionError(f"{issued_total[0] - landed[0]} copies in flight at the producer's exit")


@pytest.mark.parametrize("S", [1, 2, 3, 4])
def test_ring_and_drain(S):
    for seed in range(150):
        rnd = random.Random(seed * 13 + S)
        simulate(seed, rnd.randint(1, 40), S=S)


def test_short_shares():
    # shares shorter than the ring, equal to it, and one past it
    for S in (2, 3):
        for n in (1, S - 1, S, S + 1):
            if n >= 1:
                for seed in range(40):
                    simulate(seed, n, S=S)


def test_model_catches_a_drain_without_the_parity_flip():
    failures = 0
    for seed in range(60):
        rnd = random.Random(seed)
        try:
            # a share that ends mid-lap makes the walk back cross stage 0
            simulate(seed, rnd.randint(4, 20), S=3, flip_in_drain=False)
        except AssertionError:
            failures += 1
    assert failures > 10


def test_model_catches_a_producer_that_does_not_wait():
    failures = 0
    for seed in range(200):
        rnd = random.Random(seed)
        try:
            simulate(seed, rnd.randint(4, 20), S=2, producer_waits=False)
        except AssertionError:
            failures += 1
    assert failures > 20
