"""Host-side model of the GEMM pipeline's barrier protocol (no GPU).

One pipeline of k_gemm_tc (w12_gemm.cu): a producer fills a ring of S record stages, two
decode groups take alternate units, each decodes into A buffer j % AB, an x warp fills SX x
stages, and one MMA issuer consumes A buffer and x stage in unit order; MMAs complete in
issue order and free their A buffer and x stage.  Every wait is an mbarrier parity wait: a
wait for the k-th completion of a barrier passes as soon as the barrier's phase parity differs
from k's, so it is exact only if, when it starts, the barrier has completed k or k + 1 phases.
At k - 1 it passes at once on the previous phase: a stale record or buffer.

The simulation gives every copy, decode, load and MMA a random latency (with heavy tails, so
units overtake one another wherever the protocol allows) and checks every wait's start.  The
full-barrier wait of a decode group is the delicate one: its stage's previous unit, j - S, is
the other group's when S is odd, and it has surely been consumed only when S >= AB + 2 (the
group finished unit j - 2 after the MMA of unit j - 2 - AB, which followed the decode of
every unit up to it); otherwise the group first waits for that unit's release.  The plans below are the (S, AB, SX) of every k_gemm_tc
instantiation (TcPlan: 12-bit and 8-bit records, NT 16..256, all launch modes); the planted
cases drop the release wait where it is needed and must go stale.

The accumulator hand-off is modelled too: a segment (a row block's units in the range) ends
with its last MMA's commit to the accumulator barrier; the group that decoded the segment's
last unit waits until the earlier segments are drained (a counter), then for the
accumulator, drains it and releases it; the issuer waits for that release before the first
MMA of the segment that reuses the accumulator (one or two of them).
"""
import heapq
import random

import pytest

# (S, AB, SX) of the k_gemm_tc instantiations
SHIPPED = sorted({(5, 2, 4), (4, 3, 3), (6, 2, 4), (5, 2, 3), (5, 2, 2), (3, 2, 3), (10, 4, 3), (10, 4, 2),
                  (8, 4, 2), (7, 4, 2), (8, 2, 4), (6, 3, 3), (8, 2, 3), (7, 2, 2), (15, 4, 3), (14, 4, 2),
                  (13, 4, 2), (11, 4, 2)})


def kernel_release_wait(S, AB):
    """The kernel's rule: the decode group waits for unit j - S's release first."""
    return S % 2 == 1 and S < AB + 2


class Sim:
    def __init__(self, rng):
        self.rng, self.t, self.seq, self.heap = rng, 0.0, 0, []
        self.done = {}       # barrier -> completed phases
        self.waiters = {}    # barrier -> [(k, actor)]
        self.violations = 0

    def lat(self, lo, hi):
        d = self.rng.uniform(lo, hi)
        return d * 6 if self.rng.random() < 0.08 else d

    def at(self, t, fn):
        self.seq += 1
        heapq.heappush(self.heap, (t, self.seq, fn))

    def complete(self, b):
        self.done[b] = self.done.get(b, 0) + 1
        keep = []
        for k, actor in self.waiters.pop(b, []):
            if self.done[b] > k:
                self.at(self.t, lambda a=actor: self.step(a))
            else:
                keep.append((k, actor))
        if keep:
            self.waiters[b] = keep

    def step(self, actor):
        try:
            op = next(actor)
        except StopIteration:
            return
        if op[0] == "delay":
            self.at(self.t + op[1], lambda: self.step(actor))
        elif op[0] == "count":  # ("count", counter, n): wait until the counter reaches n
            _, b, n = op
            if self.done.get(b, 0) >= n:
                self.at(self.t, lambda: self.step(actor))
            else:
                self.waiters.setdefault(b, []).append((n - 1, actor))
        else:  # ("wait", barrier, k): wait for the k-th completion (0-based) by parity
            _, b, k = op
            c = self.done.get(b, 0)
            if c not in (k, k + 1):
                self.violations += 1
            if c % 2 != k % 2 or c > k:   # parity differs (stale pass at k - 1) or already done
                self.at(self.t, lambda: self.step(actor))
            else:
                self.waiters.setdefault(b, []).append((k, actor))

    def run(self, actors):
        for a in actors:
            self.at(0.0, lambda a=a: self.step(a))
        while self.heap:
            self.t, _, fn = heapq.heappop(self.heap)
            fn()


def simulate(S, AB, SX, release_wait, n_units, seed, KC=None, kc0=0, acc_bufs=1, drain_count=True):
    """KC: units per row block (None: one segment); kc0: the first unit's chunk; a segment
    (the units of one row block) ends with a drain of the accumulator by the group that
    decoded its last unit, after the drains of the earlier segments (drain_count)."""
    sim = Sim(random.Random(seed))
    mma_end = [0.0]
    KC = KC or n_units + kc0

    def seg_of(j):
        return (kc0 + j) // KC - kc0 // KC

    def last_of_seg(j):
        return (kc0 + j) % KC == KC - 1 or j == n_units - 1

    def producer():
        for j in range(n_units):
            s = j % S
            if j >= S:
                yield ("wait", ("rec_empty", s), j // S - 1)
            yield ("delay", 0.05)
            sim.at(sim.t + sim.lat(0.5, 6.0), lambda s=s: sim.complete(("rec_full", s)))

    def xloader():
        for j in range(n_units):
            s = j % SX
            if j >= SX:
                yield ("wait", ("x_empty", s), j // SX - 1)
            sim.at(sim.t + sim.lat(0.3, 4.0), lambda s=s: sim.complete(("x_full", s)))
            yield ("delay", 0.05)

    def group(g):
        for j in range(g, n_units, 2):
            s = j % S
            if release_wait and j >= S:
                yield ("wait", ("rec_empty", s), j // S - 1)
            yield ("wait", ("rec_full", s), j // S)
            yield ("delay", sim.lat(0.05, 0.4))          # records into registers
            sim.complete(("rec_empty", s))
            if j >= AB:
                yield ("wait", ("a_empty", j % AB), j // AB - 1)
            yield ("delay", sim.lat(0.5, 3.0))           # decode and store the A tile
            sim.complete(("a_full", j % AB))
            if last_of_seg(j):                           # drain the segment's accumulator
                seg = seg_of(j)
                if drain_count and seg > 0:
                    yield ("count", "drains", seg)
                yield ("wait", ("acc_full", seg % acc_bufs), seg // acc_bufs)
                yield ("delay", sim.lat(0.3, 2.0))
                sim.complete(("acc_empty", seg % acc_bufs))
                sim.complete("drains")

    def issuer():
        for j in range(n_units):
            seg = seg_of(j)
            if (j == 0 or (kc0 + j) % KC == 0) and seg >= acc_bufs:   # the accumulator drained
                yield ("wait", ("acc_empty", seg % acc_bufs), seg // acc_bufs - 1)
            yield ("wait", ("a_full", j % AB), j // AB)
            yield ("wait", ("x_full", j % SX), j // SX)
            end = max(mma_end[0], sim.t) + sim.lat(0.1, 1.5)   # MMAs finish in issue order
            mma_end[0] = end
            sim.at(end, lambda j=j: (sim.complete(("a_empty", j % AB)), sim.complete(("x_empty", j % SX))))
            if last_of_seg(j):
                sim.at(end, lambda seg=seg: sim.complete(("acc_full", seg % acc_bufs)))
            yield ("delay", 0.02)

    sim.run([producer(), xloader(), group(0), group(1), issuer()])
    # every unit went through: the protocol neither stalled nor skipped a phase
    assert sim.done.get(("a_full", (n_units - 1) % AB), 0) == (n_units - 1) // AB + 1
    return sim.violations


@pytest.mark.parametrize("S,AB,SX", SHIPPED)
def test_shipped_plans_wait_exactly(S, AB, SX):
    assert S % 2 == 0 or S >= AB + 2 or kernel_release_wait(S, AB)
    for seed in range(25):
        assert simulate(S, AB, SX, kernel_release_wait(S, AB), 160, seed) == 0, seed


@pytest.mark.parametrize("S,AB", [(3, 2), (3, 3), (5, 4)])
def test_planted_missing_release_wait_goes_stale(S, AB):
    """Odd rings shorter than AB + 2 without the release wait: some runs pass a full-barrier
    wait on the previous phase (the fault met with a three-stage ring); with the wait, none."""
    stale = sum(simulate(S, AB, 3, False, 160, seed) > 0 for seed in range(60))
    assert stale > 0
    assert all(simulate(S, AB, 3, True, 160, seed) == 0 for seed in range(25))


@pytest.mark.parametrize("S,AB", [(5, 2), (5, 3), (7, 4), (4, 4)])
def test_rings_at_the_bound_need_no_release_wait(S, AB):
    """Odd rings of AB + 2 stages or more, and even rings, stay exact without the wait."""
    assert all(simulate(S, AB, 3, False, 160, seed) == 0 for seed in range(40))


@pytest.mark.parametrize("S,AB,SX", [(5, 2, 4), (4, 3, 3), (3, 2, 3), (7, 4, 2), (8, 2, 3)])
@pytest.mark.parametrize("acc_bufs", [1, 2])
def test_accumulator_handoff_waits_exactly(S, AB, SX, acc_bufs):
    """Row blocks of 1 to 9 units starting anywhere in the range: the MMA issuer waits for
    the drain of the accumulator's previous segment, and the group ending a segment waits
    for the drains before it, then for the accumulator; every such wait is exact."""
    rng = random.Random(S * 100 + AB * 10 + acc_bufs)
    for seed in range(30):
        KC = rng.randint(1, 9)
        kc0 = rng.randrange(KC)
        assert simulate(S, AB, SX, kernel_release_wait(S, AB), 120, seed, KC, kc0, acc_bufs) == 0, seed


def test_planted_drains_out_of_order_go_stale():
    """Without the count of earlier drains, a group ending a short segment can wait for the
    accumulator a phase early (the segment before has not been committed yet)."""
    stale = 0
    for seed in range(60):
        stale += simulate(5, 2, 4, False, 120, seed, KC=2, kc0=1, acc_bufs=1, drain_count=False) > 0
    assert stale > 0
