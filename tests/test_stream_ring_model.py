"""A CPU model of the ring protocol of the streamed single-token GEMV kernels: one producer
fills items in order into S shared-memory stages, G groups of compute warps take the items in
turn, copies land in any order, and every wait is an mbarrier parity wait as the hardware does
it (a wait for parity P passes as soon as the number of completed phases is odd when P = 0, even
when P = 1, so it cannot tell the phase it wants from one two phases earlier).

The kernels give each group stages of its own: item j goes to group g = j % G as its q-th item
(q = j // G), into stage g + G * (q % (S // G)) as that stage's (q // (S // G))-th fill. The model
checks, over random schedules, that no group then reads a stage before the fill it waits for has
landed, that the producer never refills a stage whose last fill is unconsumed, and that nothing
deadlocks; and that the simpler scheme (item j into stage j % S, one ring for all groups) does
read early, which is the fault the per-group stages remove."""
import random

import pytest


def _slots(scheme, G, S):
    if scheme == "shared":
        return (lambda j: (j % S, j // S)), (lambda g, q: (g + q * G, (g + q * G) % S, (g + q * G) // S))
    SG = S // G
    prod = lambda j: ((j % G) + G * ((j // G) % SG), (j // G) // SG)
    cons = lambda g, q: (g + q * G, g + G * (q % SG), q // SG)
    return prod, cons


def run(scheme, G, S, N, seed):
    rng = random.Random(seed)
    prod_slot, cons_slot = _slots(scheme, G, S)
    full_done, empty_done = [0] * S, [0] * S
    stage_item = [None] * S
    landed, consumed, inflight = set(), set(), []
    next_item, next_q = 0, [0] * G
    for _ in range(100000):
        if len(consumed) == N:
            return "ok"
        acts = []
        if next_item < N:
            st, n = prod_slot(next_item)
            if empty_done[st] % 2 != (n % 2) ^ 1:  # wait(empty, parity of fill n - 1)
                acts.append(("fill", st))
        for g in range(G):
            j, st, n = cons_slot(g, next_q[g])
            if j < N and full_done[st] % 2 != n % 2:  # wait(full, parity of fill n)
                acts.append(("read", g, j, st))
        if inflight:
            acts.append(("land",))
        if not acts:
            return "deadlock"
        a = rng.choice(acts)
        if a[0] == "fill":
            st = a[1]
            if stage_item[st] is not None and stage_item[st] not in consumed:
                return "overwrite"
            stage_item[st] = next_item
            inflight.append((next_item, st))
            next_item += 1
        elif a[0] == "land":
            j, st = inflight.pop(rng.randrange(len(inflight)))
            landed.add(j)
            full_done[st] += 1
        else:
            _, g, j, st = a
            if j not in landed or stage_item[st] != j:
                return "early read"
            consumed.add(j)
            next_q[g] += 1
            empty_done[st] += 1
    return "deadlock"


@pytest.mark.parametrize("G,S", [(2, 2), (2, 4), (2, 6), (3, 3), (3, 6)])
def test_per_group_stages_never_read_early(G, S):
    for seed in range(150):
        assert run("group", G, S, 29, seed) == "ok", seed


@pytest.mark.parametrize("G,S", [(3, 2), (2, 5)])
def test_one_ring_for_all_groups_can_read_early(G, S):
    results = {run("shared", G, S, 29, seed) for seed in range(150)}
    assert "early read" in results
