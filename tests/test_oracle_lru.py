"""Pins of the LRU simulator: a second, list-based LRU, closed-form counts and invariants."""
from collections import OrderedDict

import numpy as np
import pytest

from oracle.lru import LRUSim
import synth


def ordered_dict_lru(keys, capacity):
    """Textbook LRU: an OrderedDict in recency order; miss evicts the front entry."""
    od = OrderedDict()
    events = []
    for key in keys:
        if key in od:
            od.move_to_end(key)
            events.append(("hit", key))
        else:
            ev = -1
            if len(od) >= capacity:
                ev, _ = od.popitem(last=False)
            od[key] = True
            events.append(("fill", key, ev))
    return events


@pytest.mark.parametrize("N,E,L,seed", [(1, 4, 1, 0), (3, 8, 2, 1), (6, 16, 1, 2), (10, 32, 3, 3), (64, 64, 4, 4)])
def test_single_access_steps_match_ordered_dict_lru(N, E, L, seed):
    keys = synth.lru_trace_keys(L * E, 600, seed)
    sim = LRUSim(N, E)
    got = []
    for key in keys:
        layer, e = divmod(int(key), E)
        ev, _ = sim.step(layer, [e])
        (kind, *rest), = ev
        if kind == "hit":
            got.append(("hit", int(key)))
        else:
            got.append(("fill", int(key), rest[2]))
    assert got == ordered_dict_lru([int(k) for k in keys], N)


def test_capacity_at_least_keys_misses_equal_distinct():
    E, L = 16, 3
    rng = np.random.default_rng(0)
    sim = LRUSim(L * E, E)
    seen = set()
    fills = 0
    for _ in range(200):
        layer = int(rng.integers(0, L))
        ex = rng.integers(0, E, size=5)
        ev, _ = sim.step(layer, ex)
        fills += sum(1 for x in ev if x[0] == "fill")
        seen |= {layer * E + int(e) for e in ex}
    assert fills == len(seen)


def test_mattson_inclusion_single_accesses():
    keys = synth.lru_trace_keys(40, 800, 5)
    prev = None
    for N in range(1, 41):
        sim = LRUSim(N, 40)
        for key in keys:
            sim.step(0, [int(key)])
        if prev is not None:
            assert sim.fills <= prev
        prev = sim.fills


def test_ratio_one_never_external_ratio_zero_fills_one_per_wave():
    E, N = 32, 12
    rng = np.random.default_rng(1)
    a, b = LRUSim(N, E), LRUSim(N, E)
    for step in range(100):
        ex = rng.integers(0, E, size=int(rng.integers(1, 10)))
        ev_a, _ = a.step(step % 3, ex, ratio=1.0)
        assert all(x[0] != "ext" for x in ev_a)
        ev_b, _ = b.step(step % 3, ex, ratio=1e-9)
        m = sum(1 for x in ev_b if x[0] != "hit")
        f = sum(1 for x in ev_b if x[0] == "fill")
        assert f == (1 if m else 0)


def test_external_experts_do_not_change_state():
    E, N = 16, 8
    s1 = LRUSim(N, E)
    s1.step(0, [1, 2, 3])
    before = (list(s1.key), list(s1.stamp))
    # ratio small: one fill, the rest external; compare with the same step restricted to the fill
    ev, so = s1.step(1, [4, 5, 6, 7], ratio=0.01)
    assert [x[0] for x in ev] == ["fill", "ext", "ext", "ext"]
    s2 = LRUSim(N, E)
    s2.step(0, [1, 2, 3])
    s2.step(1, [4])
    assert s1.key == s2.key and s1.stamp == s2.stamp
    assert so[0][5] == -2 and so[0][4] >= 0 and so[0][0] == -1


def test_waves_when_unique_exceeds_slots():
    E, N = 16, 6
    sim = LRUSim(N, E)
    ev, slot_of = sim.step(0, list(range(14)))
    assert len(slot_of) == 3                           # 6 + 6 + 2
    assert [x[1] for x in ev] == list(range(14))
    # the third wave evicts the least recently used: the first wave's slots
    assert all(x[0] == "fill" for x in ev)
    assert sorted(slot_of[2][e] for e in (12, 13)) == [0, 1]
    assert sim.clock == 3


def test_victims_are_empty_then_oldest_then_lowest_slot():
    sim = LRUSim(4, 8)
    sim.step(0, [0, 1])          # slots 0, 1 at stamp 1
    sim.step(0, [2])             # slot 2 at stamp 2
    ev, _ = sim.step(0, [3])     # empty slot 3 first
    assert ev == [("fill", 3, 3, -1)]
    ev, _ = sim.step(0, [0, 4])  # 0 hit (stamp 4); victim: oldest untouched = slot 1 (stamp 1)
    assert ev == [("hit", 0, 0), ("fill", 4, 1, 1)]
    ev, _ = sim.step(0, [5, 6])  # oldest: slot 2 (stamp 2), slot 3 (stamp 3)
    assert ev == [("fill", 5, 2, 2), ("fill", 6, 3, 3)]


def test_resize_keeps_most_recent_and_moves_minimally():
    E = 8
    sim = LRUSim(6, E)
    for e in range(6):
        sim.step(0, [e])         # slot s holds expert s with stamp s+1
    moves = sim.resize(3)
    # keep experts 5, 4, 3 (most recent); they sat in slots 5, 4, 3 and move to 0, 1, 2
    assert moves == [(3, 0), (4, 1), (5, 2)]
    assert sim.key == [3, 4, 5] and sim.stamp == [4, 5, 6]
    sim.resize(5)
    assert sim.key == [3, 4, 5, -1, -1]
    ev, _ = sim.step(0, [0, 3])
    assert ev == [("fill", 0, 3, -1), ("hit", 3, 0)]


def test_stream_carve_and_adopt():
    E = 4
    sim = LRUSim(12, E)
    sim.step(1, [0, 1])                      # keys 4, 5 in slots 0, 1
    base, moves = sim.stream_begin()
    assert base == 4 and moves == []
    # layers 0..2 streamed; layer 1 sat in buffer 1, layer 2 in buffer 0
    sim.stream_end([(1, 1), (2, 0)])
    assert sim.N == 12
    # layer 1 experts 0, 1 were resident: refreshed in place, their buffer slots stay empty
    assert sim.key[0] == 4 and sim.key[1] == 5 and sim.stamp[0] == 2
    assert sim.key[8:12] == [-1, -1, 6, 7]
    assert sim.key[4:8] == [8, 9, 10, 11] and sim.stamp[4] == 3
    ev, _ = sim.step(2, [3])
    assert ev == [("hit", 3, 7)]
