"""The CPU model of the S-slot full/empty protocol (no GPU)."""
import os

import numpy as np
import pytest

from oracle import ring_model as rm
from pipelined_warp_specialized_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _operands(M, N, K, seed):
    A = inputs.ints(seed, 0, (M, K)).astype(np.int64)
    B = inputs.ints(seed, 1, (N, K)).astype(np.int64)
    return A, B, A @ B.T


@pytest.mark.parametrize("S", [1, 2, 3, 4, 5, 6])
@pytest.mark.parametrize("BK", [16, 32, 64])
def test_ring_equals_triple_loop_for_every_stage_count(S, BK):
    A, B, want = _operands(5, 7, 3 * BK + 5, seed=S * 10 + BK)   # ragged K tail
    for sched in range(3):
        got = rm.pipelined_nt(A, B, S, BK, schedule_seed=sched)
        assert np.array_equal(got, want)


def test_ring_threads_equal_triple_loop():
    A, B, want = _operands(4, 6, 200, seed=3)
    for S in (1, 2, 4, 6):
        assert np.array_equal(rm.pipelined_nt_threads(A, B, S, 16), want)


@pytest.mark.parametrize("S", [1, 2, 4])
def test_missing_empty_seed_deadlocks(S):
    # Croqtile ch.6: without the initial "trigger empty" the producer's first wait never ends
    A, B, _ = _operands(3, 3, 64, seed=1)
    with pytest.raises(rm.Deadlock):
        rm.pipelined_nt(A, B, S, 16, seed_empty=False)


def test_missing_empty_seed_times_out_with_threads():
    A, B, _ = _operands(3, 3, 64, seed=1)
    with pytest.raises(rm.Deadlock):
        rm.pipelined_nt_threads(A, B, 2, 16, seed_empty=False, timeout_s=0.2)


def test_early_release_is_caught():
    # Croqtile ch.6: releasing empty before the multiply is done lets the
    # producer overwrite operands still in use
    A, B, _ = _operands(3, 3, 16 * 12, seed=2)
    caught = 0
    for sched in range(20):
        try:
            rm.pipelined_nt(A, B, 1, 16, release_early=True, schedule_seed=sched)
        except rm.Hazard:
            caught += 1
    assert caught > 0


def test_parity_wait_never_ambiguous():
    ev = rm.Event("e")
    assert not ev.done(0)
    ev.trigger()
    assert ev.done(0) and not ev.done(1)
    ev.trigger()
    assert ev.done(1)
    ev.trigger()
    with pytest.raises(AssertionError):
        ev.done(1)            # waiter two laps behind: parity alone cannot tell


def _golden_schedule():
    facts = {}
    with open(os.path.join(GOLDEN, "s32_swap_schedule.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = [p.strip() for p in line.split("=")]
                facts[k] = int(v)
    return facts


def test_swap_schedule_matches_the_pages_three_phases():
    g = _golden_schedule()
    assert g["tiles"] * g["tile_k"] == g["K"]
    assert g["grid_blocks"] * g["threads_per_block"] == g["M"] * g["N"]
    tr = rm.swap_schedule(g["tiles"])
    rm.check_swap_schedule(tr, g["tiles"])
    count = lambda ph, act: sum(1 for p, a, *_ in tr if p == ph and a == act)  # noqa: E731
    assert count("prologue", "load") == g["prologue_loads"]
    assert count("prologue", "compute") == g["prologue_computes"]
    assert count("steady", "swap") == g["steady_iterations"]
    assert count("steady", "load") == g["steady_iterations"]
    assert count("steady", "compute") == g["steady_iterations"]
    assert count("epilogue", "load") == g["epilogue_loads"]
    assert count("epilogue", "compute") == g["epilogue_computes"]


def test_swap_schedule_planted_mistake_is_caught():
    tr = rm.swap_schedule(4)
    # swapping before computing: the compute reads the buffer just being loaded
    bad = list(tr)
    i = next(i for i, t in enumerate(bad) if t[1] == "compute")
    phase, act, tile, buf = bad[i]
    bad[i] = (phase, act, tile, 1 - buf)
    with pytest.raises(rm.Hazard):
        rm.check_swap_schedule(bad, 4)
    # loading tile t into the buffer still holding tile t-1
    bad2 = list(tr)
    j = next(i for i, t in enumerate(bad2) if t[0] == "steady" and t[1] == "load")
    phase, act, tile, buf = bad2[j]
    bad2[j] = (phase, act, tile, 1 - buf)
    with pytest.raises(rm.Hazard):
        rm.check_swap_schedule(bad2, 4)


@pytest.mark.parametrize("S", [2, 3, 4, 5, 6])
@pytest.mark.parametrize("one_barrier", [False, True])
def test_ring_slot_schedules_are_hazard_free(S, one_barrier):
    # both barrier orders of the S-slot rotate read every tile once, in order,
    # after its copies landed and a barrier followed, and refill a slot only
    # after a barrier followed the read of its previous tile
    for T in range(0, 3 * S + 4):
        rm.check_ring_slot_schedule(rm.ring_slot_schedule(T, S, one_barrier), T, S)


def test_ring_slot_schedule_keeps_s_minus_one_tiles_ahead():
    # the one-barrier order refills after the wait, so during the wait for
    # tile t only tiles t+1 .. t+S-2 can be in flight; the two-barrier order
    # has already issued t+S-1 -- which is why it is kept for S = 2, where the
    # one-barrier order would wait with nothing else in flight
    for S in (2, 3, 6):
        for one_barrier, ahead in ((True, S - 2), (False, S - 1)):
            tr = rm.ring_slot_schedule(4 * S, S, one_barrier)
            issued, t = 0, 0
            for ev in tr:
                if ev[0] == "issue":
                    issued = max(issued, ev[1] + 1)
                elif ev[0] == "wait" and t < 4 * S - S:      # steady waits, before the tail runs dry
                    assert issued - 1 - t == ahead, (S, one_barrier, t, issued)
                elif ev[0] == "read":
                    t = ev[1] + 1


def test_ring_slot_schedule_planted_mistakes_are_caught():
    T, S = 10, 4
    one = rm.ring_slot_schedule(T, S, True)
    two = rm.ring_slot_schedule(T, S, False)
    # two-barrier order without its trailing barrier: a slot is refilled in
    # the interval in which its previous tile is still being read
    bad = [ev for i, ev in enumerate(two)
           if not (ev == ("barrier",) and i > 0 and two[i - 1][0] == "read")]
    with pytest.raises(rm.Hazard, match="no barrier after the read"):
        rm.check_ring_slot_schedule(bad, T, S)
    # one-barrier order with every refill moved before its barrier (from
    # iteration 1 on, the slot refilled still holds the tile read last)
    bad = list(one)
    for i in range(1, len(bad)):
        if bad[i][0] == "issue" and bad[i - 1] == ("barrier",):
            bad[i - 1], bad[i] = bad[i], bad[i - 1]
    with pytest.raises(rm.Hazard, match="no barrier after the read"):
        rm.check_ring_slot_schedule(bad, T, S)
    # one-barrier order waiting one group too few: the tile is read before it landed
    bad = [("wait", S - 1) if ev == ("wait", S - 2) else ev for ev in one]
    with pytest.raises(rm.Hazard, match="before its copy group was waited for"):
        rm.check_ring_slot_schedule(bad, T, S)
    # reading the slot the refill targets
    bad = list(one)
    j = next(j for j, ev in enumerate(bad) if ev[0] == "read" and ev[1] == 2)
    bad[j] = ("read", 2, (bad[j][2] + S - 1) % S)
    with pytest.raises(rm.Hazard):
        rm.check_ring_slot_schedule(bad, T, S)
