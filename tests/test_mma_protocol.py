"""A model of the batched tensor-memory kernel's hand-off protocol, run on the CPU.

The kernel (csrc/gemv_i8_mma.cu) moves each pair of 128-weight groups through
four roles joined by mbarriers: a copy warp fills a ring of input stages, 8
producer warps expand a pair into an A/B slot, two MMA warps (even and odd
pairs) run the pair's MMAs into a D buffer, and 8 folder warps read the D
buffer back. This test replays exactly the waits, arrivals and commits each
role makes -- the same barrier counts and the same phase-parity formulas as
the kernel -- under many random interleavings, with copies and MMAs
completing at random later times, and checks that

  * every role finishes (no schedule deadlocks),
  * no wait is ever satisfied by the wrong phase (a barrier is never more than
    one phase past the phase a waiter asks for, which the hardware's parity
    test could not tell apart),
  * an MMA reads a slot that holds its own pair, unchanged until the MMA has
    completed; a folder reads a D buffer that holds its own pair, not yet
    overwritten by a later MMA; a copy refills a stage only after every
    producer has read it.

The kernel's wait bounds and abort path are not modelled.
"""

import os
import random
import re

import pytest

_SRC = os.path.join(os.path.dirname(__file__), "..", "bit_decode_gemv_gb300", "csrc", "gemv_i8_mma.cu")


def _kernel_constant(name):
    """The value of `constexpr int <name> = <n>;` in the kernel source, so that the
    model always replays the protocol of the kernel as it stands."""
    with open(_SRC) as f:
        m = re.search(r"constexpr\s+int\s+" + name + r"\s*=\s*(\d+)\s*;", f.read())
    assert m, f"{name} not found in the kernel source"
    return int(m.group(1))


N_PRODUCERS = _kernel_constant("kProducerWarps")
N_FOLDERS = _kernel_constant("kFolderWarps")
N_MMA = _kernel_constant("kMmaWarps")
STAGES = _kernel_constant("kStages")
SLOTS = _kernel_constant("kSlots")
PAIR = _kernel_constant("kPair")


class Barrier:
    """An mbarrier: `count` arrivals complete a phase."""

    def __init__(self, count):
        self.count = count
        self.pending = 0
        self.completed = 0   # phases completed so far

    def arrive(self):
        self.pending += 1
        assert self.pending <= self.count
        if self.pending == self.count:
            self.pending = 0
            self.completed += 1

    def ready(self, index, parity):
        """Whether a wait for phase `index` (passed to the hardware as `parity`) returns."""
        assert parity == index & 1, "the kernel's parity formula disagrees with the phase it means"
        # the hardware compares parities only: the barrier must never be two phases past
        assert self.completed <= index + 1, "a waiter would see its phase completed twice over"
        return self.completed > index


def run_schedule(G, rng, slot_wait=True):
    """One random interleaving of the whole protocol for G groups; raises
    AssertionError on a hazard or a deadlock. slot_wait=False leaves out the
    producers' wait for a slot's previous MMAs (a planted mistake)."""
    npairs = (G + PAIR - 1) // PAIR
    m_full = [Barrier(1) for _ in range(STAGES)]
    m_empty = [Barrier(N_PRODUCERS) for _ in range(STAGES)]
    ab_full = [Barrier(N_PRODUCERS) for _ in range(SLOTS)]
    ab_empty = [Barrier(1) for _ in range(SLOTS)]
    d_full = [Barrier(1) for _ in range(SLOTS)]
    d_empty = [Barrier(N_FOLDERS) for _ in range(SLOTS)]

    stage_tag = [None] * STAGES        # pair whose inputs a stage holds (None while a copy is in flight)
    stage_reads = [set() for _ in range(STAGES)]
    slot_tag = [[None] * N_PRODUCERS for _ in range(SLOTS)]   # pair each producer's part of a slot holds
    mma_reading = [None] * SLOTS       # pair whose MMAs are reading the slot
    d_tag = [None] * SLOTS             # pair whose sums a D buffer holds
    d_reads = [set() for _ in range(SLOTS)]
    pending = []                       # asynchronous completions (copies landing, MMAs completing)

    def copy_warp():
        def issue(P):
            st = P % STAGES
            assert stage_tag[st] is None or stage_reads[st] == set(range(N_PRODUCERS)), \
                "a stage refilled before every producer read it"
            stage_tag[st] = None
            stage_reads[st].clear()

            def land():
                stage_tag[st] = P
                m_full[st].arrive()
            pending.append(land)
        for P in range(min(npairs, STAGES)):
            issue(P)
            yield True
        for P in range(npairs - STAGES):
            st = P % STAGES
            while not m_empty[st].ready(P // STAGES, (P // STAGES) & 1):
                yield False
            issue(P + STAGES)
            yield True

    def producer(i):
        st, st_par = 0, 0
        for P in range(npairs):
            sl, sl_par = P & 1, (P >> 1) & 1
            if P >= SLOTS and slot_wait:
                while not ab_empty[sl].ready((P >> 1) - 1, sl_par ^ 1):
                    yield False
            while not m_full[st].ready(P // STAGES, st_par):
                yield False
            assert stage_tag[st] == P, "a producer read a stage holding another pair"
            assert mma_reading[sl] is None, "a producer overwrote a slot an MMA is reading"
            stage_reads[st].add(i)
            slot_tag[sl][i] = P
            m_empty[st].arrive()
            ab_full[sl].arrive()
            st += 1
            if st == STAGES:
                st, st_par = 0, st_par ^ 1
            yield True

    def mma_warp(w):
        for P in range(w, npairs, N_MMA):
            par = (P // N_MMA) & 1
            while not ab_full[w].ready(P // N_MMA, par):
                yield False
            while not d_empty[w].ready(P // N_MMA, par):
                yield False
            assert all(t == P for t in slot_tag[w]), "an MMA read a slot not filled with its pair"
            assert d_tag[w] is None or d_reads[w] == set(range(N_FOLDERS)), \
                "an MMA overwrote a D buffer before every folder read it"
            mma_reading[w] = P
            d_tag[w] = None
            d_reads[w].clear()

            def complete(w=w, P=P):
                assert all(t == P for t in slot_tag[w]), "a slot changed under its MMAs"
                mma_reading[w] = None
                d_tag[w] = P
                ab_empty[w].arrive()   # the two commits arrive when the MMAs complete
                d_full[w].arrive()
            pending.append(complete)
            yield True

    def folder(i):
        for db in range(SLOTS):
            d_empty[db].arrive()   # D buffers start free
        yield True
        for P in range(npairs):
            sl, par = P & 1, (P >> 1) & 1
            while not d_full[sl].ready(P >> 1, par):
                yield False
            assert d_tag[sl] == P, "a folder read a D buffer holding another pair"
            d_reads[sl].add(i)
            d_empty[sl].arrive()
            yield True

    live = [copy_warp()] + [producer(i) for i in range(N_PRODUCERS)] + \
           [mma_warp(w) for w in range(N_MMA)] + [folder(i) for i in range(N_FOLDERS)]
    idle = 0   # consecutive steps in which nothing moved
    while live or pending:
        k = rng.randrange(len(live) + len(pending))
        if k >= len(live):
            pending.pop(k - len(live))()
            idle = 0
            continue
        try:
            moved = next(live[k])
        except StopIteration:
            live.pop(k)
            moved = True
        idle = 0 if moved else idle + 1
        # with nothing in flight, every live role blocked for many picks in a row is a deadlock
        assert pending or idle < 50 * (len(live) + 1), "deadlock: every role waits and nothing is in flight"


@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 6, 7, 8, 9, 12, 20, 40, 41])
def test_protocol_random_interleavings(G):
    """No deadlock and no hazard over random schedules, for odd and even group
    counts, fewer pairs than stages and many more."""
    rng = random.Random(1000 + G)
    for _ in range(40):
        run_schedule(G, rng)


def test_model_catches_a_missing_slot_wait():
    """The model is not vacuous: producers that do not wait for a slot's previous
    MMAs are caught overwriting a slot under its MMAs (or running its barrier
    two phases ahead) in some schedule."""
    rng = random.Random(7)
    caught = 0
    for _ in range(100):
        try:
            run_schedule(12, rng, slot_wait=False)
        except AssertionError:
            caught += 1
    assert caught > 0
