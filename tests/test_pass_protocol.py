"""A randomised model of the persistent pass kernel's mbarrier protocol
(`pass_kernel` in the patch-formation kernels).

Roles: one TMA producer, one MMA issuer, four epilogue warps.  A CTA takes a
sequence of items (a 128-row tile, a K slice and a layer); every item is a run of
K-blocks.  The producer streams all K-blocks of all items through an S-stage ring
(barriers full / empty); the MMA issuer accumulates item j into TMEM buffer j % 2
and commits it to acc_full[j % 2]; the epilogue warps drain buffer j % 2 and
release it on acc_empty[j % 2] (four arrivals), which the MMA issuer awaits before
item j + 2.  Every wait tests only the parity of a phase, with the phase index
the kernel computes: stage phase g / S for K-block g, buffer phase j / 2 for item j.

The model replays that protocol under random interleavings, random copy
latencies and in-order tensor-core completion, and fails if a wait passes on the
wrong phase, a stage or buffer is read holding anything but what the reader
expects, a copy or MMA is still in flight when the CTA would free TMEM, or the
pipeline deadlocks.  Two broken variants (no wait for the epilogue before reusing
a buffer; no wait for the MMA before reusing a stage) are shown to fail, so the
model does catch those hazards."""
import random

import pytest

from test_pipeline_protocol import Bar


def simulate(seed, nks, S=4, n_epi=4, skip_acc_wait=False, skip_empty_wait=False):
    rnd = random.Random(seed)
    full, empty = [Bar(1) for _ in range(S)], [Bar(1) for _ in range(S)]
    acc_full, acc_empty = [Bar(1), Bar(1)], [Bar(n_epi), Bar(n_epi)]
    stage = [None] * S      # K-block held by each stage
    acc = [None, None]      # item whose MMAs last wrote each TMEM buffer
    events, clock, tc_time = [], [0], [0]

    def later(fn):
        events.append((clock[0] + rnd.randint(1, 30), fn))

    def tensor_pipe(fn):
        # tcgen05.mma and tcgen05.commit complete in issue order
        tc_time[0] = max(tc_time[0], clock[0]) + rnd.randint(1, 12)
        events.append((tc_time[0], fn))

    def producer():
        g = 0
        for nk in nks:
            for _ in range(nk):
                st = g % S
                if g >= S and not skip_empty_wait:
                    while not empty[st].try_wait(g // S - 1):
                        yield
                full[st].arrive(tx=1)

                def land(st=st, g=g):
                    stage[st] = g
                    full[st].complete_tx(1)
                later(land)
                g += 1
                yield
        # every issued copy lands before the CTA may exit
        for q in range(max(0, g - S), g):
            while not full[q % S].try_wait(q // S):
                yield

    def mma():
        g = 0
        for j, nk in enumerate(nks):
            b = j & 1
            if j >= 2 and not skip_acc_wait:
                while not acc_empty[b].try_wait((j >> 1) - 1):
                    yield
            for _ in range(nk):
                st = g % S
                while not full[st].try_wait(g // S):
                    yield
                assert stage[st] == g, f"stage {st} holds K-block {stage[st]}, MMA expected {g}"

                def done(st=st, b=b, j=j, g=g):
                    assert stage[st] == g, "stage overwritten while its MMAs read it"
                    acc[b] = j
                    empty[st].arrive()
                tensor_pipe(done)
                g += 1
                yield

            def commit(b=b, j=j):
                acc[b] = j
                acc_full[b].arrive()
            tensor_pipe(commit)

    def epilogue():
        for j, nk in enumerate(nks):
            b = j & 1
            while not acc_full[b].try_wait(j >> 1):
                yield
            if nk > 0:
                for _ in range(rnd.randint(1, 4)):   # column chunks read from TMEM
                    assert acc[b] == j, f"buffer {b} holds item {acc[b]} while item {j} is drained"
                    yield
            acc_empty[b].arrive()
            yield

    roles = [producer(), mma()] + [epilogue() for _ in range(n_epi)]
    live, steps = list(roles), 0
    while live:
        steps += 1
        if steps > 1_000_000:   # a role's wait loop keeps yielding, so a deadlock shows as the step limit
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
        if not live and events:
            raise AssertionError(f"{len(events)} copies or MMAs still in flight when TMEM is freed")


def random_nks(rnd, zero_ok=True):
    lo = 0 if zero_ok else 1
    return [rnd.randint(lo, 10) for _ in range(rnd.randint(1, 12))]


@pytest.mark.parametrize("S", [2, 3, 4, 6])
def test_protocol_never_accepts_a_stale_phase(S):
    for seed in range(120):
        rnd = random.Random(seed * 7 + S)
        simulate(seed, random_nks(rnd), S=S)


def test_single_item_and_single_block():
    for seed in range(20):
        simulate(seed, [1])
        simulate(seed, [0])
        simulate(seed, [1, 1, 1])


def test_model_catches_a_buffer_reused_before_it_was_drained():
    failures = 0
    for seed in range(200):
        rnd = random.Random(seed)
        try:
            simulate(seed, [rnd.randint(1, 3) for _ in range(rnd.randint(4, 12))], skip_acc_wait=True)
        except AssertionError:
            failures += 1
    assert failures > 20


def test_model_catches_a_stage_reused_before_its_mmas_read_it():
    failures = 0
    for seed in range(200):
        rnd = random.Random(seed)
        try:
            simulate(seed, random_nks(rnd, zero_ok=False), S=2, skip_empty_wait=True)
        except AssertionError:
            failures += 1
    assert failures > 20
