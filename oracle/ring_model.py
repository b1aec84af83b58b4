"""CPU model of the S-slot full/empty credit protocol -- TEST INFRASTRUCTURE ONLY.

It plays the two roles of the pipelined K loop on the CPU and checks what the
pages state about them:

* Croqtile tutorial ch.6, "带 event 的 1P1C 内核": one ``full[s]``/``empty[s]``
  pair per physical slot; ``stage = k % S``; the producer waits ``empty``,
  fills the slot, triggers ``full``; the consumer seeds every ``empty`` once
  before its loop, then waits ``full``, multiplies, commits, triggers
  ``empty``.  Without the seeding the producer's first wait never completes
  (a deadlock, which the model reports instead of hanging); releasing
  ``empty`` before the multiply has finished lets the producer overwrite an
  operand still in use (which the model's hazard detector reports).
* TileLang tutorial ch.22, section 3.2 (barrier versioning): a reused event
  is waited with the parity of its lap, ``(k // S) % 2``; the model waits by
  parity only, like an mbarrier, and separately asserts that no waiter is ever
  two laps behind (where parity alone would be ambiguous).
* Croqtile tutorial ch.6, "三阶段" and "swap": the double-buffer schedule of
  the s32 kernel -- a prologue load of tile 0, steady iterations that load
  tile t while computing tile t-1 and then swap the buffer names, and an
  epilogue that computes the last tile.
* The same chapter's rotate over S buffers, with asynchronous copies: as the
  TileLang tutorial ch.22 section 4.3 notes, a block barrier does not wait
  for them, so a tile may be read only after the copy group holding it has
  been waited for and a barrier has followed, and a buffer may be refilled
  only after a barrier has followed every read of its previous tile.
  ``ring_slot_schedule`` and ``check_ring_slot_schedule`` model that
  S-slot schedule, with the refill either before the wait (two barriers per
  tile) or after the barrier that publishes the tile (one barrier per tile).

The multiply step uses numpy's matmul on one K slice of integer-valued
operands, so the model's sum is exact and is compared for equality.
"""
from __future__ import annotations

import random
import threading

import numpy as np


class Event:
    """A phase-counting event with mbarrier-like parity waits.

    ``trigger()`` completes the current phase.  ``done(parity)`` is true when
    the most recently completed phase has that parity, i.e. a waiter for lap
    ``p`` passes once ``p + 1`` phases are complete.
    """

    def __init__(self, name: str):
        self.name = name
        self.completed = 0

    def trigger(self) -> None:
        self.completed += 1

    def done(self, lap: int) -> bool:
        parity = lap & 1
        # hardware view: only the parity of the phase is visible
        passed = self.completed > 0 and ((self.completed - 1) & 1) == parity
        # exact view, to check the parity wait is never ambiguous
        exact = self.completed >= lap + 1
        if passed != exact and self.completed > lap + 1:
            raise AssertionError(f"{self.name}: waiter for lap {lap} is two or more laps behind "
                                 f"({self.completed} phases complete); parity is ambiguous")
        return passed


class ProtocolError(Exception):
    pass


class Deadlock(ProtocolError):
    pass


class Hazard(ProtocolError):
    pass


def _tiles(K: int, BK: int) -> int:
    return -(-K // BK)


def pipelined_nt(A: np.ndarray, B: np.ndarray, S: int, BK: int, *, seed_empty: bool = True,
                 release_early: bool = False, sub_steps: int = 4, schedule_seed: int = 0,
                 max_steps: int = 10_000_000) -> np.ndarray:
    """C = A . B^T through an S-slot ring driven by a seeded adversarial interleaver.

    The producer and consumer are generators that yield after every visible
    action; at each step the interleaver picks one runnable role at random
    (seeded), so every run explores a different legal interleaving.  A state
    where no role can run raises ``Deadlock`` (the CPU analogue of a bounded
    device wait that expires).  The consumer reads its slot in ``sub_steps``
    pieces (the MMA sub-steps of one K strip); a producer write into a slot
    that is being read raises ``Hazard``.
    """
    if S < 1:
        raise ValueError("S must be >= 1")
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    T = _tiles(K, BK)
    full = [Event(f"full[{s}]") for s in range(S)]
    empty = [Event(f"empty[{s}]") for s in range(S)]
    slot_a = [np.zeros((M, BK), dtype=A.dtype) for _ in range(S)]
    slot_b = [np.zeros((N, BK), dtype=B.dtype) for _ in range(S)]
    readers = [0] * S
    C = np.zeros((M, N), dtype=np.int64)
    state = {"wait": None}

    def producer():
        for k in range(T):
            s, lap = k % S, k // S
            while not empty[s].done(lap):
                yield ("blocked", empty[s], lap)
            if readers[s]:
                raise Hazard(f"producer overwrote slot {s} while the consumer was reading it (k={k})")
            lo, hi = k * BK, min(K, (k + 1) * BK)
            slot_a[s][:] = 0                      # zero fill past K
            slot_b[s][:] = 0
            slot_a[s][:, : hi - lo] = A[:, lo:hi]
            yield ("run",)
            if readers[s]:
                raise Hazard(f"producer overwrote slot {s} while the consumer was reading it (k={k})")
            slot_b[s][:, : hi - lo] = B[:, lo:hi]
            yield ("run",)
            full[s].trigger()
            yield ("run",)

    def consumer():
        if seed_empty:
            for s in range(S):
                empty[s].trigger()
                yield ("run",)
        per = -(-BK // sub_steps)
        for k in range(T):
            s, lap = k % S, k // S
            while not full[s].done(lap):
                yield ("blocked", full[s], lap)
            if release_early:
                empty[s].trigger()                # BUG under test: released before the MMA ran
            readers[s] += 1
            for j in range(0, BK, per):
                a = slot_a[s][:, j:j + per].astype(np.int64)
                yield ("run",)
                b = slot_b[s][:, j:j + per].astype(np.int64)
                C[...] += a @ b.T
                yield ("run",)
            readers[s] -= 1                       # "mma.commit": the strip's reads are done
            if not release_early:
                empty[s].trigger()
            yield ("run",)

    rng = random.Random(schedule_seed)
    roles = {"producer": producer(), "consumer": consumer()}
    status = {name: ("run",) for name in roles}
    steps = 0
    while roles:
        steps += 1
        if steps > max_steps:
            raise Deadlock("step limit reached")
        runnable = []
        for name, st in status.items():
            if st[0] == "run" or st[1].done(st[2]):
                runnable.append(name)
        if not runnable:
            waits = {n: f"{st[1].name} lap {st[2]}" for n, st in status.items()}
            raise Deadlock(f"no role can run: {waits}")
        name = rng.choice(runnable)
        try:
            status[name] = next(roles[name])
        except StopIteration:
            del roles[name]
            del status[name]
    state["wait"] = None
    return C


def pipelined_nt_threads(A: np.ndarray, B: np.ndarray, S: int, BK: int, *, seed_empty: bool = True,
                         timeout_s: float = 2.0) -> np.ndarray:
    """The same protocol with two real threads and bounded waits.

    Each wait gives up after ``timeout_s`` and raises ``Deadlock`` in the
    caller, the host analogue of the kernel's bounded mbarrier waits.
    """
    M, K = A.shape
    N = B.shape[0]
    T = _tiles(K, BK)
    cv = threading.Condition()
    full = [0] * S        # completed phases per event
    empty = [0] * S
    slot_a = [np.zeros((M, BK), dtype=np.int64) for _ in range(S)]
    slot_b = [np.zeros((N, BK), dtype=np.int64) for _ in range(S)]
    C = np.zeros((M, N), dtype=np.int64)
    errors = []

    def wait(arr, s, lap):
        with cv:
            ok = cv.wait_for(lambda: arr[s] > 0 and ((arr[s] - 1) & 1) == (lap & 1) or errors,
                             timeout=timeout_s)
            if errors:
                raise Deadlock("peer failed")
            if not ok:
                raise Deadlock(f"wait timed out (slot {s}, lap {lap})")

    def trigger(arr, s):
        with cv:
            arr[s] += 1
            cv.notify_all()

    def producer():
        try:
            for k in range(T):
                s = k % S
                wait(empty, s, k // S)
                lo, hi = k * BK, min(K, (k + 1) * BK)
                slot_a[s][:] = 0
                slot_b[s][:] = 0
                slot_a[s][:, : hi - lo] = A[:, lo:hi]
                slot_b[s][:, : hi - lo] = B[:, lo:hi]
                trigger(full, s)
        except Exception as e:  # noqa: BLE001 -- reported to the caller below
            with cv:
                errors.append(e)
                cv.notify_all()

    def consumer():
        try:
            if seed_empty:
                for s in range(S):
                    trigger(empty, s)
            for k in range(T):
                s = k % S
                wait(full, s, k // S)
                C[...] += slot_a[s] @ slot_b[s].T
                trigger(empty, s)
        except Exception as e:  # noqa: BLE001
            with cv:
                errors.append(e)
                cv.notify_all()

    threads = [threading.Thread(target=producer), threading.Thread(target=consumer)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout_s * 4)
    if errors:
        raise errors[0]
    return C


def swap_schedule(T: int) -> list:
    """Trace of the two-buffer swap schedule over T K tiles.

    Returns (phase, action, tile, buffer) tuples, where ``buffer`` is the
    physical buffer (0 or 1) that the name ``cur``/``nxt`` denoted at that
    moment.  The swap exchanges the two names, never the data.
    """
    if T < 1:
        return []
    trace = []
    cur, nxt = 0, 1
    trace.append(("prologue", "load", 0, cur))
    for t in range(1, T):
        trace.append(("steady", "load", t, nxt))
        trace.append(("steady", "compute", t - 1, cur))
        cur, nxt = nxt, cur                      # swap the handles
        trace.append(("steady", "swap", t, cur))
    trace.append(("epilogue", "compute", T - 1, cur))
    return trace


def check_swap_schedule(trace: list, T: int) -> None:
    """Checks the hazards of a swap trace: each tile loaded and computed once,
    a compute reads the buffer its tile was loaded into (read after write),
    and a load never targets a buffer whose tile is still waiting to be
    computed (write after read)."""
    loaded_into = {}
    holds = {0: None, 1: None}        # tile sitting in each buffer, not yet computed
    computed = []
    for phase, action, tile, buf in trace:
        if action == "load":
            if holds[buf] is not None:
                raise Hazard(f"tile {tile} loaded over uncomputed tile {holds[buf]} in buffer {buf}")
            if tile in loaded_into:
                raise Hazard(f"tile {tile} loaded twice")
            loaded_into[tile] = buf
            holds[buf] = tile
        elif action == "compute":
            if loaded_into.get(tile) != buf:
                raise Hazard(f"tile {tile} computed from buffer {buf}, loaded into {loaded_into.get(tile)}")
            holds[buf] = None
            computed.append(tile)
    if computed != list(range(T)):
        raise Hazard(f"tiles computed out of order or missing: {computed}")


def ring_slot_schedule(T: int, S: int, one_barrier: bool) -> list:
    """Trace of the S-slot rotate over T K tiles with asynchronous copies.

    The block's threads are taken to move together between barriers.  Events:
    ``("issue", tile, slot)`` starts the copies of a tile, ``("commit",)``
    closes a copy group, ``("wait", n)`` returns once at most the newest ``n``
    groups are still in flight, ``("barrier",)`` is a block barrier and
    ``("read", tile, slot)`` is the multiply over a tile.

    The prologue fills slots 0..S-2.  Iteration t refills the slot tile t-1
    used with tile t+S-1 and reads tile t.  With ``one_barrier`` the refill
    comes after the barrier that publishes tile t (wait S-2 groups, barrier,
    refill, commit, read); otherwise before the wait (refill, commit, wait
    S-1 groups, barrier, read, barrier).
    """
    trace = []
    for t in range(S - 1):
        if t < T:
            trace.append(("issue", t, t))
        trace.append(("commit",))
    cur, nxt = 0, S - 1
    for t in range(T):
        if one_barrier:
            trace += [("wait", S - 2), ("barrier",)]
            if t + S - 1 < T:
                trace.append(("issue", t + S - 1, nxt))
            trace.append(("commit",))
            trace.append(("read", t, cur))
        else:
            if t + S - 1 < T:
                trace.append(("issue", t + S - 1, nxt))
            trace += [("commit",), ("wait", S - 1), ("barrier",), ("read", t, cur), ("barrier",)]
        cur = (cur + 1) % S                      # rotate the slot names
        nxt = (nxt + 1) % S
    trace.append(("wait", 0))
    return trace


def check_ring_slot_schedule(trace: list, T: int, S: int) -> None:
    """Checks the hazards of a ring trace.  A tile is read from the slot it
    was copied into, after its copy group has been waited for and a barrier
    has followed (read after write); a slot is refilled only once its
    previous tile has been read and a barrier has followed that read (write
    after read); every tile is read once, in order."""
    groups = []                  # committed copy groups, oldest first: lists of tiles
    open_group = []
    landed = {}                  # tile -> barrier epoch in which its group was waited for
    holds = [None] * S           # tile last copied into each slot
    read_epoch = [None] * S      # epoch of the last read of each slot's tile
    unread = [False] * S
    epoch = 0
    reads = []
    for ev in trace:
        kind = ev[0]
        if kind == "issue":
            _, tile, slot = ev
            if unread[slot]:
                raise Hazard(f"tile {tile} copied over unread tile {holds[slot]} in slot {slot}")
            if read_epoch[slot] is not None and read_epoch[slot] >= epoch:
                raise Hazard(f"tile {tile} copied into slot {slot} with no barrier after the read of "
                             f"tile {holds[slot]}")
            holds[slot], unread[slot] = tile, True
            open_group.append(tile)
        elif kind == "commit":
            groups.append(open_group)
            open_group = []
        elif kind == "wait":
            n = ev[1]
            while len(groups) > n:
                for tile in groups.pop(0):
                    landed[tile] = epoch
        elif kind == "barrier":
            epoch += 1
        elif kind == "read":
            _, tile, slot = ev
            if holds[slot] != tile:
                raise Hazard(f"tile {tile} read from slot {slot}, which holds tile {holds[slot]}")
            if tile not in landed:
                raise Hazard(f"tile {tile} read before its copy group was waited for")
            if landed[tile] >= epoch:
                raise Hazard(f"tile {tile} read with no barrier after its copies landed")
            read_epoch[slot], unread[slot] = epoch, False
            reads.append(tile)
        else:
            raise ValueError(f"unknown event {ev!r}")
    if reads != list(range(T)):
        raise Hazard(f"tiles read out of order or missing: {reads}")
