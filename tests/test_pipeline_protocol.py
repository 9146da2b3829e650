"""Host-side model of the GQA tensor-core kernel's hand-over protocol
(score_heads_tc.cu): a copy thread, two groups of feature warps and an MMA
thread exchange ring stages, operand buffers and accumulators through
mbarriers waited by phase parity. The model runs the same schedule of waits
and arrivals under many random interleavings, with copies and MMAs that
complete at random later moments, and checks:

  * every parity wait targets the phase in progress or the one just
    completed (a parity cannot tell a phase from the one two later, so a
    wait further ahead passes at once, and one further behind never does);
  * every stage, operand buffer and accumulator holds the block its reader
    expects when it reads it, and nothing is overwritten while in use;
  * the run ends (no wait is left without its arrival).

A planted variant with three ring stages shared by the two groups (tile t in
stage t % 3) must be caught: a group a tile ahead waits on a phase two ahead
of the barrier.
"""
import random

import pytest


class Barrier:
    def __init__(self, name, count):
        self.name, self.count = name, count
        self.phase = 0  # index of the phase in progress; phases < phase are complete
        self.pending = count

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, f"{self.name}: more arrivals than expected"
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count


class Violation(Exception):
    pass


def run_protocol(ntiles, nst, rng, nbuf=3, a_free_wait=True):
    """One random interleaving of the kernel's protocol for a run of ntiles
    blocks, ring of nst stages (tile t in stage t % nst). a_free_wait=False
    plants a mistake: a group writes an operand buffer without waiting for
    the MMAs of the block before it there. Raises Violation on a broken
    invariant; returns the number of scheduler steps."""
    full = [Barrier(f"full[{s}]", 1) for s in range(nst)]
    empty = [Barrier(f"empty[{s}]", 1) for s in range(nst)]  # one arrival per group (its threads together)
    a_full = [Barrier(f"a_full[{b}]", 1) for b in range(nbuf)]
    mma_done = [Barrier(f"mma_done[{b}]", 1) for b in range(nbuf)]
    d_free = [Barrier(f"d_free[{b}]", 1) for b in range(nbuf)]
    stage = [None] * nst  # tile whose bytes a stage holds (None while a copy is in flight)
    stage_busy = [False] * nst  # a copy is writing the stage
    abuf = [None] * nbuf  # block whose features an operand buffer holds
    abuf_reading = [None] * nbuf  # block whose MMAs are reading the buffer
    acc = [None] * nbuf  # block whose scores an accumulator holds
    pending = []  # async completions: (kind, payload)

    def wait(bar, j):
        # the waiter asks for completion of phase j by its parity
        while True:
            k = bar.phase
            if not (k == j or k == j + 1):
                raise Violation(f"{bar.name}: wait for phase {j} while phase {k} is in progress")
            if k == j + 1:
                return
            yield

    def copy_thread():
        for u in range(ntiles):
            st = u % nst
            if u >= nst:
                yield from wait(empty[st], u // nst - 1)
            if stage_busy[st]:
                raise Violation(f"stage {st} refilled while a copy is in flight")
            stage[st] = None
            stage_busy[st] = True
            pending.append(("copy", (st, u)))
            yield

    def group(g):
        last = -1
        t = g
        while t < ntiles:
            st = t % nst
            yield from wait(full[st], t // nst)
            if stage[st] != t:
                raise Violation(f"group {g} read stage {st} for tile {t}, it holds {stage[st]}")
            yield  # the lanes load the tile's chunks
            if stage[st] != t:
                raise Violation(f"stage {st} overwritten while group {g} loaded tile {t}")
            empty[st].arrive()
            if t >= nbuf and a_free_wait:
                yield from wait(mma_done[t % nbuf], t // nbuf - 1)
            b = t % nbuf
            if abuf_reading[b] is not None:
                raise Violation(f"operand buffer {b} written while MMAs of block {abuf_reading[b]} read it")
            abuf[b] = t
            yield  # features formed
            a_full[b].arrive()
            if t >= 2:
                yield from readout(g, t - 2)
            last = t
            t += 2
        if last >= 0:
            yield from readout(g, last)

    def readout(g, blk):
        b = blk % nbuf
        yield from wait(mma_done[b], blk // nbuf)
        if acc[b] != blk:
            raise Violation(f"group {g} read accumulator {b} for block {blk}, it holds {acc[b]}")
        yield
        d_free[b].arrive()

    def mma_thread():
        for t in range(ntiles):
            b = t % nbuf
            yield from wait(a_full[b], t // nbuf)
            if t >= nbuf:
                yield from wait(d_free[b], t // nbuf - 1)
            if abuf[b] != t:
                raise Violation(f"MMAs of block {t} found buffer {b} holding {abuf[b]}")
            abuf_reading[b] = t
            acc[b] = None  # the accumulator is being overwritten
            pending.append(("mma", (b, t)))
            yield

    actors = [copy_thread(), group(0), group(1), mma_thread()]
    live = list(actors)
    steps = 0
    while live or pending:
        steps += 1
        if steps > 100000:
            raise Violation("no progress (deadlock)")
        # an async completion or an actor step, at random
        if pending and (not live or rng.random() < 0.35):
            kind, payload = pending.pop(rng.randrange(len(pending)))
            if kind == "copy":
                st, u = payload
                stage[st] = u
                stage_busy[st] = False
                full[st].arrive()
            else:
                b, t = payload
                abuf_reading[b] = None
                acc[b] = t
                mma_done[b].arrive()
            continue
        a = rng.choice(live)
        try:
            next(a)
        except StopIteration:
            live.remove(a)
    return steps


@pytest.mark.parametrize("ntiles", [1, 2, 3, 4, 5, 7, 12])
def test_kernel_protocol_holds_under_random_interleavings(ntiles):
    # the kernel's ring: one stage per group's tile (two stages, tile t in stage t % 2)
    rng = random.Random(ntiles)
    for _ in range(300):
        run_protocol(ntiles, nst=2, rng=rng)


def test_four_stage_ring_of_the_d64_case_holds():
    # head_dim 64: 16 KB tiles in a 64 KB ring, four stages, still one group per stage
    rng = random.Random(64)
    for _ in range(300):
        run_protocol(12, nst=4, rng=rng)


def test_planted_three_stage_ring_is_caught():
    # three stages shared by the two groups: a group a tile ahead waits two
    # phases ahead of a stage's barrier (the race found by reading the
    # earlier form of the kernel)
    rng = random.Random(3)
    caught = []
    for _ in range(2000):
        try:
            run_protocol(12, nst=3, rng=rng)
        except Violation as e:
            caught.append(str(e))
    assert caught and all(c.startswith("full[") and "in progress" in c for c in caught)


def test_planted_missing_operand_buffer_wait_is_caught():
    # forming block t in buffer t % 3 without waiting for block t - 3's MMAs
    rng = random.Random(5)
    caught = []
    for _ in range(300):
        try:
            run_protocol(12, nst=2, rng=rng, a_free_wait=False)
        except Violation as e:
            caught.append(str(e))
    assert caught and any("operand buffer" in c for c in caught)


def run_shared_ring(ntiles, nst, nw, rng):
    """The CUDA-core score kernels' ring (score_common.cuh): nw warps each
    take every tile in order (waiting on the stage's full barrier by parity),
    count themselves done on the stage, and the last one of tile t refills
    the stage with tile t + nst. Warps drift apart by up to the ring depth."""
    full = [Barrier(f"full[{s}]", 1) for s in range(nst)]
    consumed = [0] * nst
    stage = [None] * nst
    pending = []

    def wait(bar, j):
        while True:
            k = bar.phase
            if not (k == j or k == j + 1):
                raise Violation(f"{bar.name}: wait for phase {j} while phase {k} is in progress")
            if k == j + 1:
                return
            yield

    def issue(u):
        stage[u % nst] = None
        pending.append(u)

    def warp(w):
        for t in range(ntiles):
            st = t % nst
            yield from wait(full[st], t // nst)
            if stage[st] != t:
                raise Violation(f"warp {w} read stage {st} for tile {t}, it holds {stage[st]}")
            yield
            if stage[st] != t:
                raise Violation(f"stage {st} refilled while warp {w} read tile {t}")
            consumed[st] += 1
            if consumed[st] == nw:
                consumed[st] = 0
                if t + nst < ntiles:
                    issue(t + nst)

    for u in range(min(nst, ntiles)):
        issue(u)
    live = [warp(w) for w in range(nw)]
    steps = 0
    while live or pending:
        steps += 1
        if steps > 200000:
            raise Violation("no progress (deadlock)")
        if pending and (not live or rng.random() < 0.3):
            u = pending.pop(rng.randrange(len(pending)))
            stage[u % nst] = u
            full[u % nst].arrive()
            continue
        a = rng.choice(live)
        try:
            next(a)
        except StopIteration:
            live.remove(a)


def test_shared_ring_with_drifting_warps_holds():
    rng = random.Random(7)
    for ntiles in (1, 3, 4, 9, 17):
        for _ in range(200):
            run_shared_ring(ntiles, nst=4, nw=8, rng=rng)
