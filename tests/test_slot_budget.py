"""Pins of the oracle's greedy per-layer slot budget ("Project Maya" page,
section "VRAM: one partition per layer, sized by what the layer routes"):
hand-worked cases, the tie rules, saturation, argument errors, and - on
every small case - optimality: because each layer's next expert serves a
non-increasing share, the greedy split maximises the summed share of lookups
served over all splits that give every layer at least the floor.  The
library's device planner (expcache_plan_slots) is checked against the oracle
on the GPU."""
import itertools
from fractions import Fraction

import numpy as np
import pytest

import oracle


def test_hand_worked_split():
    # layer 0 routes 8,4,2,2 (16 lookups), layer 1 routes 10,1,1,0 (12).
    # floor 1: expert 0 of each.  Then shares 4/16 vs 1/12 -> layer 0; 2/16
    # (expert 2, the lower id of the two 2s) vs 1/12 -> layer 0; 2/16 vs 1/12
    # -> layer 0.
    ls, order = oracle.slot_budget([[8, 4, 2, 2], [10, 1, 1, 0]], 5, 1)
    assert ls.tolist() == [0, 4, 5]
    assert order.tolist() == [[0, 1, 2, 3], [0, 1, 2, 3]]
    # order: count descending, ties to the lower id
    ls, order = oracle.slot_budget([[1, 5, 5, 0, 2]], 2, 0)
    assert order.tolist() == [[1, 2, 4, 0, 3]] and ls.tolist() == [0, 2]


def test_wide_layer_gets_more_slots():
    """A layer that spreads its routes wide (flat counts) takes more of the
    budget than one whose routes concentrate on a few experts."""
    E = 64
    skewed = (1000.0 / np.arange(1, E + 1) ** 1.5).astype(np.uint32) + 1
    flat = np.full(E, 40, np.uint32)
    ls, _ = oracle.slot_budget(np.stack([skewed, flat]), 64, 8)
    n = np.diff(ls)
    assert n.sum() == 64 and n[1] > n[0] >= 8


def test_ties_go_to_the_lower_layer_and_zero_route_layers():
    # 3 floors, then 4 slots over equal shares: every one is a tie, so the
    # lowest layer that still has room takes it
    ls, _ = oracle.slot_budget([[3, 3, 3, 3]] * 3, 7, 1)
    assert np.diff(ls).tolist() == [4, 2, 1]
    # a layer without routes (share 0) takes slots only once the others are full
    ls, _ = oracle.slot_budget([[0, 0, 0], [5, 4, 1]], 5, 1)
    assert np.diff(ls).tolist() == [2, 3]
    ls, _ = oracle.slot_budget([[0, 0, 0], [5, 4, 1]], 4, 1)
    assert np.diff(ls).tolist() == [1, 3]


def test_saturation_and_errors():
    ls, _ = oracle.slot_budget([[1, 2], [3, 4]], 10, 0)
    assert ls.tolist() == [0, 2, 4]  # every layer full, the rest unassigned
    assert oracle.slot_budget([[1, 2], [3, 4]], 3, 2) is None  # floors do not fit
    assert oracle.slot_budget([[1, 2], [3, 4]], 10, 3) is None  # floor > E


def _served(c, order, n):
    S = sum(int(v) for v in c)
    return Fraction(sum(int(c[e]) for e in order[:n]), S) if S else Fraction(0)


def test_greedy_split_is_optimal_on_small_cases():
    rng = np.random.default_rng(17)
    for trial in range(300):
        L, E = int(rng.integers(1, 4)), int(rng.integers(1, 6))
        c = rng.integers(0, 6, (L, E)).astype(np.uint32)
        if rng.random() < 0.2:
            c[rng.integers(L)] = 0
        floor = int(rng.integers(0, E + 1))
        total = int(rng.integers(L * floor, L * E + 3))
        ls, order = oracle.slot_budget(c, total, floor)
        n = np.diff(ls)
        assert n.sum() == min(total, L * E) and np.all(n >= floor) and np.all(n <= E)
        for l in range(L):  # the order is the definition's
            assert order[l].tolist() == sorted(range(E), key=lambda e: (-int(c[l, e]), e))
        got = sum(_served(c[l], order[l], n[l]) for l in range(L))
        best = max(sum(_served(c[l], order[l], m[l]) for l in range(L))
                   for m in itertools.product(range(floor, E + 1), repeat=L)
                   if sum(m) == min(total, L * E))
        assert got == best, (c, floor, total, n)
