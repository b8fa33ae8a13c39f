"""Randomised model of the K/V ring of the VSA fine kernel (csrc/vsa_attn.cu,
vsa_fine_kernel): one producer issues the loads of each unit in the order
K_0, K_1, then V_j, K_{j+2} for j = 0, 1, ...; two MMA threads take the loads
of alternate K/V tiles (tile j belongs to thread j % 2); load L goes to slot
L % S and completes on full barrier L % B.  Copies complete in any order and
the threads run at any relative speed.  The kernel relies on B = 2 S: a
thread's parity wait on load L can then only succeed on L's own completion,
never on the barrier's previous phase.  The model checks that claim, and
that with B = S the same schedules do hit a stale phase."""
import random

import pytest


def loads_of_unit(nkv):
    seq = [0, 1]                       # owners (tile j -> thread j % 2) of K_0, K_1
    for j in range(nkv):
        seq.append(j % 2)              # V_j
        if j + 2 < nkv:
            seq.append(j % 2)          # K_{j+2}
    return seq


def run(units, slots, bars, seed):
    """Returns None, or a description of the first stale-phase wait."""
    rng = random.Random(seed)
    owner = [t for nkv in units for t in loads_of_unit(nkv)]
    n = len(owner)
    full_done = [0] * bars             # completed phases per full barrier
    empty_done = [0] * slots           # completed phases per empty barrier
    issued, inflight, complete = 0, [], [False] * n
    mine = [[i for i in range(n) if owner[i] == g] for g in (0, 1)]
    nxt, pending, consumed = [0, 0], [], 0
    steps = 0
    while consumed < n:
        steps += 1
        assert steps < 10 ** 6, "no progress"
        act = rng.randrange(5)
        if act == 0 and issued < n:                   # producer: slot's previous use consumed
            if issued < slots or empty_done[issued % slots] >= issued // slots:
                inflight.append(issued)
                issued += 1
        elif act == 1 and inflight:                   # a copy completes
            x = inflight.pop(rng.randrange(len(inflight)))
            complete[x] = True
            full_done[x % bars] += 1
        elif act in (2, 3):                           # MMA thread g waits on its next load
            g = act - 2
            if nxt[g] < len(mine[g]):
                x = mine[g][nxt[g]]
                if (full_done[x % bars] & 1) != ((x // bars) & 1):   # try_wait.parity succeeds
                    if not complete[x]:
                        return f"thread {g} passed load {x} before it completed"
                    pending.append(x)
                    nxt[g] += 1
        elif act == 4 and pending:                    # an MMA completes, its slot is freed
            x = pending.pop(rng.randrange(len(pending)))
            assert empty_done[x % slots] == x // slots
            empty_done[x % slots] += 1
            consumed += 1
    return None


def schedules(count):
    for t in range(count):
        rng = random.Random(t)
        yield t, [rng.choice([2, 2, 3, 4, 5, 7, 10, 40]) for _ in range(rng.randrange(1, 6))]


def test_twice_the_slots_never_passes_a_stale_phase():
    for seed, units in schedules(400):
        assert run(units, slots=4, bars=8, seed=seed) is None, units


def test_as_many_barriers_as_slots_does_pass_a_stale_phase():
    # the negative control: the model can fail
    assert any(run(units, slots=4, bars=4, seed=seed) for seed, units in schedules(400))
