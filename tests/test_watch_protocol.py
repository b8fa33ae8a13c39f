"""Randomised model of the dense attention kernel's K/V ring and P barriers
(csrc/attn_fwd.cu, attn_fwd_kernel): one producer issues each unit's loads
K_0, V_0, K_1, V_1, ... into a ring of 4 slots (load L to slot L % 4, one
full barrier per slot), the unit's Q only once the previous unit's MMAs have
completed; the MMA thread waits for K_0 itself and then, per K/V tile j, only
for each q-tile's P barrier before P V_j and Q K_{j+1}^T; each P barrier
completes a phase on two arrivals, the q-tile's softmax (after its S) and the
watcher (after V_j and K_{j+1} have landed).  Copies and MMAs complete in any
order and every thread runs at any relative speed.

The model checks the watcher's wait order: every parity wait succeeds only
on its own phase, every MMA finds its operands landed, each P phase completes
with one arrival of each kind, and nothing deadlocks.  Two other orders fail
it, which pins the reasons for the kernel's: waiting for V_j and K_{j+1}
before the previous P phase lets a wait on K_{j+1} pass on K_{j-1}'s pending
phase when copies land out of order, and also waiting for the unit's K_0 can
meet K_0's barrier two phases on (the MMA thread consumes K_0 on its own, so
K_2 can refill the slot and land first) and never return."""
import random

import pytest

SLOTS = 4


class Stop(Exception):
    pass


def simulate(units, order, seed, max_steps=200000):
    """Returns None when the run completes cleanly, else what went wrong."""
    rng = random.Random(seed)
    # the ring: load L is (unit, kind, j); units' loads back to back
    loads, ring_base, tile_base = [], [], []
    t = 0
    for u, n in enumerate(units):
        ring_base.append(len(loads))
        tile_base.append(t)
        for j in range(n):
            loads.append((u, "K", j))
            loads.append((u, "V", j))
        t += n
    n_loads, n_tiles = len(loads), t
    complete = [False] * n_loads
    full_done = [0] * SLOTS            # completed phases per full barrier
    empty_done = [0] * SLOTS           # consumed uses per slot
    pf_done = [0, 0]                   # completed phases per P barrier
    pf_arrivals = [[], []]             # arrivals in the current phase
    s_ready = [set(), set()]           # tiles whose S_k is computed
    unit_mmas_done = [False] * len(units)
    async_events = []                  # pending completions: callables
    err = []

    def fail(msg):
        err.append(msg)
        raise Stop()

    def load_idx(u, kind, j):
        return ring_base[u] + 2 * j + (1 if kind == "V" else 0)

    def try_full(L):
        ok = (full_done[L % SLOTS] & 1) != ((L // SLOTS) & 1)
        if ok and not complete[L]:
            fail(f"parity wait on load {loads[L]} passed before it landed")
        return ok

    def try_pf(k, tile):
        ok = (pf_done[k] & 1) != (tile & 1)
        if ok and pf_done[k] <= tile:
            fail(f"wait on P{k} phase {tile} passed on a stale phase")
        return ok

    def arrive_pf(k, who, tile):
        pf_arrivals[k].append((who, tile))
        if len(pf_arrivals[k]) == 2:
            whos = sorted(w for w, _ in pf_arrivals[k])
            if whos != ["softmax", "watcher"] or any(tt != pf_done[k] for _, tt in pf_arrivals[k]):
                fail(f"P{k} phase {pf_done[k]} completed on {pf_arrivals[k]}")
            pf_arrivals[k] = []
            pf_done[k] += 1

    def consume(L):
        def done():
            assert empty_done[L % SLOTS] == L // SLOTS
            empty_done[L % SLOTS] += 1
        async_events.append(done)

    def need(L, what):
        if not complete[L]:
            fail(f"{what} issued before {loads[L]} landed")

    # ---- the producer
    def producer():
        for u, n in enumerate(units):
            while u > 0 and not unit_mmas_done[u - 1]:   # QEmpty of the previous unit
                yield
            for L in range(ring_base[u], ring_base[u] + 2 * n):
                while L >= SLOTS and empty_done[L % SLOTS] < L // SLOTS:
                    yield
                def land(L=L):
                    complete[L] = True
                    full_done[L % SLOTS] += 1
                async_events.append(land)
                yield

    # ---- the MMA thread
    def mma():
        for u, n in enumerate(units):
            k0 = load_idx(u, "K", 0)
            while not try_full(k0):
                yield
            need(k0, "Q K_0^T")
            for k in (0, 1):
                def s_done(k=k, tt=tile_base[u]):
                    s_ready[k].add(tt)
                async_events.append(s_done)
            consume(k0)
            for j in range(n):
                tt = tile_base[u] + j
                more = j + 1 < n
                for k in (0, 1):
                    while not try_pf(k, tt):
                        yield
                    need(load_idx(u, "V", j), "P V_j")
                    if more:
                        need(load_idx(u, "K", j + 1), "Q K_j+1^T")
                        def s_next(k=k, tt=tt + 1):
                            s_ready[k].add(tt)
                        async_events.append(s_next)
                    yield
                consume(load_idx(u, "V", j))
                if more:
                    consume(load_idx(u, "K", j + 1))
            def unit_done(u=u):
                unit_mmas_done[u] = True
            async_events.append(unit_done)
            yield

    # ---- the softmax of q-tile k
    def softmax(k):
        for tt in range(n_tiles):
            while tt not in s_ready[k]:
                yield
            yield
            arrive_pf(k, "softmax", tt)

    # ---- the watcher, in one of three orders
    def watcher():
        for u, n in enumerate(units):
            if order == "k0_too":
                while not try_full(load_idx(u, "K", 0)):
                    yield
            for j in range(n):
                tt = tile_base[u] + j
                more = j + 1 < n
                if order == "kernel" and tt > 0:
                    while not try_pf(0, tt - 1):
                        yield
                for L in [load_idx(u, "V", j)] + ([load_idx(u, "K", j + 1)] if more else []):
                    while not try_full(L):
                        yield
                for k in (0, 1):
                    if tt > 0 and not (order == "kernel" and k == 0):
                        while not try_pf(k, tt - 1):
                            yield
                    arrive_pf(k, "watcher", tt)
                    yield

    threads = [producer(), mma(), softmax(0), softmax(1), watcher()]
    finished = [False] * len(threads)
    try:
        for step in range(max_steps):
            if all(finished) and not async_events:
                return None
            choice = rng.randrange(len(threads) + 2)
            if choice >= len(threads):                # an asynchronous completion
                if async_events:
                    async_events.pop(rng.randrange(len(async_events)))()
                continue
            if not finished[choice]:
                try:
                    next(threads[choice])
                except StopIteration:
                    finished[choice] = True
        return "no progress (deadlock)"
    except Stop:
        return err[0]


UNIT_MIXES = [[1, 1, 1, 1, 1, 1], [2, 2, 2, 2], [3, 1, 2, 5, 1, 3], [6, 6, 6], [1, 4, 1, 4, 2]]


@pytest.mark.parametrize("units", UNIT_MIXES)
def test_kernel_order_is_safe(units):
    for seed in range(150):
        assert simulate(units, "kernel", seed) is None, (units, seed)


def test_data_waits_before_the_previous_p_phase_can_pass_on_a_stale_phase():
    found = [simulate(units, "data_first", seed) for units in UNIT_MIXES for seed in range(400)]
    assert any(r is not None and "passed" in r for r in found), "expected a stale parity wait"


def test_watcher_also_waiting_for_k0_can_stall_or_pass_stale():
    found = [simulate(units, "k0_too", seed) for units in UNIT_MIXES for seed in range(400)]
    assert any(r is not None for r in found), "expected a stale wait or a deadlock"
