"""Pins of the oracle's adaptive expert-cache policy against what the
"Project Maya" page states: a route adds one to its expert's count, capped at
2^24; every 32,768 route events all counts are halved; a missing expert takes
a free slot of its layer and is resident from then on; between forwards each
layer evicts its least-used resident (recency breaks ties) until it has its
spares again; victims come only from the layer's own slots.  Plus invariants
of any such cache (slots conserved, never two experts in one slot) and the
LFU outcome on a stationary routing distribution."""
import numpy as np
import pytest

import oracle


def _counts(E, routed):
    c = np.zeros(E, np.int32)
    for e, n in routed.items():
        c[e] = n
    return c


def test_miss_is_promoted_into_a_free_slot_and_then_hits():
    # layer 0 owns slots 0..3; experts 0, 1 resident; slots 2, 3 free
    p = oracle.CachePolicy(1, 16, 4, [0, 4], 2, [0, 1] + [-1] * 14)
    prom = p.step(0, _counts(16, {5: 1}))
    assert list(prom) == [2]          # the lowest free slot
    assert p.table[0, 5] == 2         # resident from this forward on
    # the refill restored two free slots by evicting the least-used resident
    assert p.free[:4].sum() == 2
    prom = p.step(0, _counts(16, {5: 1}))
    assert list(prom) == []           # a hit now: no miss


def test_misses_beyond_the_free_slots_are_staged():
    p = oracle.CachePolicy(1, 16, 3, [0, 3], 1, [-1] * 16)
    prom = p.step(0, _counts(16, {2: 1, 7: 1, 9: 1, 11: 1}))
    # ascending ids take the free slots in ascending order, the rest staged
    assert list(prom) == [0, 1, 2, -1]
    assert p.table[0, 2] < 0 or p.table[0, 7] < 0 or p.table[0, 9] < 0  # one evicted (K = 1)


def test_count_is_capped_at_2_pow_24():
    p = oracle.CachePolicy(1, 4, 2, [0, 2], 0, [0, 1, -1, -1])
    big = (1 << 24) - 3
    p.step(0, _counts(4, {0: big}))
    # the forward's 16,777,213 routes crossed 32,768 events: halved once
    assert p.cnt[0, 0] == big >> 1
    p2 = oracle.CachePolicy(1, 4, 2, [0, 2], 0, [0, 1, -1, -1])
    p2.events[0] = 0
    # many small forwards without reaching a halving cannot exceed the cap:
    # set a count near the cap and add below the event threshold
    p2.cnt[0, 1] = (1 << 24) - 2
    p2.step(0, _counts(4, {1: 100}))
    assert p2.cnt[0, 1] == 1 << 24


def test_halving_every_32768_events_over_all_layers():
    p = oracle.CachePolicy(2, 4, 4, [0, 2, 4], 0, [0, 1, -1, -1, 2, 3, -1, -1])
    p.step(1, _counts(4, {0: 8}))              # layer 1: count 8
    p.step(0, _counts(4, {1: 32768 - 8 - 1}))  # 32,767 events in all: no halving
    assert p.cnt[1, 0] == 8 and p.cnt[0, 1] == 32768 - 9
    p.step(0, _counts(4, {1: 1}))              # the 32,768th event
    assert p.cnt[1, 0] == 4                    # the other layer's count halved too
    assert p.cnt[0, 1] == (32768 - 8) >> 1
    assert p.events[0] == 0


def test_boundary_evicts_least_used_with_recency_tie_break():
    # slots 0..3 all resident (experts 0..3), K = 1: one must go each forward
    p = oracle.CachePolicy(1, 8, 4, [0, 4], 0, [0, 1, 2, 3, -1, -1, -1, -1])
    p.K = 1
    p.step(0, _counts(8, {0: 3, 1: 1, 2: 1, 3: 2}))   # all counts set at forward 1
    # least used: experts 1 and 2 (count 1, same last): the lower id goes
    assert p.table[0, 1] < 0 and p.table[0, 2] >= 0
    # forward 2: expert 5 misses and takes the free slot; the boundary then
    # evicts between 2 (count 1, forward 1) and 5 (count 1, forward 2): 2
    p.step(0, _counts(8, {5: 1}))
    assert p.table[0, 5] >= 0 and p.table[0, 2] < 0
    # recency: equal counts, the one routed earlier goes first
    q = oracle.CachePolicy(1, 8, 4, [0, 4], 0, [0, 1, 2, 3, -1, -1, -1, -1])
    q.step(0, _counts(8, {0: 5, 1: 5, 2: 5, 3: 2}))   # K = 0: nothing evicted
    q.step(0, _counts(8, {3: 3}))                      # 3 reaches 5 at forward 2
    q.K = 1
    q.step(0, _counts(8, {0: 0}))                      # no routes; boundary: counts all 5
    assert q.table[0, 0] < 0       # 0, 1, 2 tie on (5, forward 1): the lowest id goes
    assert q.table[0, 3] >= 0      # 3 was routed last


def test_victims_only_from_the_layers_own_slots():
    p = oracle.CachePolicy(2, 8, 6, [0, 3, 6], 1, [0, 1, 2, -1, -1, -1, -1, -1,
                                                   -1, -1, -1, 3, 4, 5, -1, -1])
    t1 = p.table[1].copy()
    p.step(0, _counts(8, {6: 1}))
    assert (p.table[1] == t1).all()
    assert p.free[3:6].sum() == 0 and p.free[:3].sum() == 1


@pytest.mark.parametrize("K", [0, 1, 3])
def test_invariants_under_random_routing(K):
    rng = np.random.default_rng(7)
    L, E, per = 3, 40, 10
    ls = [0, per, 2 * per, 3 * per]
    table = -np.ones((L, E), np.int32)
    for l in range(L):
        for i in range(per - K):
            table[l, i] = ls[l] + i
    p = oracle.CachePolicy(L, E, 3 * per, ls, K, table)
    for step in range(300):
        l = step % L
        ids = rng.choice(E, size=6, replace=False)
        c = np.zeros(E, np.int32)
        c[ids] = rng.integers(1, 4, size=6)
        missing = [int(e) for e in np.flatnonzero(c) if p.table[l, e] < 0]
        free_before = [s for s in range(ls[l], ls[l + 1]) if p.free[s]]
        prom = p.step(l, c)
        # misses in ascending id, the first ones into the free slots in order
        assert len(prom) == len(missing)
        n_prom = min(len(missing), len(free_before))
        assert list(prom[:n_prom]) == free_before[:n_prom]
        assert all(v == -1 for v in prom[n_prom:])
        for ll in range(L):
            slots = [int(s) for s in p.table[ll] if s >= 0]
            assert len(slots) == len(set(slots))                       # one expert per slot
            assert all(ls[ll] <= s < ls[ll + 1] for s in slots)          # own partition
            free = [s for s in range(ls[ll], ls[ll + 1]) if p.free[s]]
            assert set(free).isdisjoint(slots)
            assert len(free) + len(slots) == per                        # slots conserved
            assert len(free) >= min(K, per)                              # spares refilled


def test_lfu_keeps_the_most_routed_experts():
    # stationary Zipf routing over 32 experts, 8 slots with 1 spare: after a
    # warm-up the 7 resident experts are (nearly) the 7 most routed
    rng = np.random.default_rng(3)
    E, n = 32, 8
    prob = 1.0 / np.arange(1, E + 1) ** 1.2
    prob /= prob.sum()
    p = oracle.CachePolicy(1, E, n, [0, n], 1, [-1] * E)
    hits = tot = 0
    for step in range(3000):
        ids = rng.choice(E, size=4, replace=False, p=prob)
        c = np.zeros(E, np.int32)
        c[ids] = 1
        resident_before = set(np.flatnonzero(p.table[0] >= 0))
        p.step(0, c)
        if step >= 1000:
            hits += sum(1 for e in ids if e in resident_before)
            tot += len(ids)
    res = set(np.flatnonzero(p.table[0] >= 0))
    assert len(res & set(range(7))) >= 6
    # the hit rate approaches the top-7 share of the routing mass (sampling
    # without replacement makes the share a little lower than prob[:7].sum())
    assert hits / tot > 0.8 * prob[:7].sum()
