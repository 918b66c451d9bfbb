"""Pins of the placement-policy replay ([Review] §2.4), and the native replay against it.

The oracle's three policies are checked on a trace worked out by hand, against
a second LRU written with an ordered dictionary, and on invariants (full
capacity, nested fixed sets, inclusion for single accesses).  libft's
ft_placement_replay (host code, no GPU) must then give the oracle's counts
exactly on seeded random traces.
"""
from collections import OrderedDict

import numpy as np
import pytest

from oracle import placement

# L = 2 layers, E = 3 experts: key = layer * 3 + expert
HAND = [
    [[1, 1, 0], [2]],        # step 0: layer 0 routes {0, 1}, layer 1 routes {2}
    [[2], [0, 2]],           # step 1
    [[0], [1]],              # step 2
]
PREFILL = {0: 5, 3: 4, 5: 4, 1: 1, 2: 0, 4: 0}


def test_hand_worked_trace():
    # 8 accesses.  Static split of 3: layer 0 resident, the 4 layer-1 accesses miss.
    assert placement.static_set(2, 3, 3) == {0, 1, 2} and placement.static_set(2, 3, 4) == {0, 1, 2, 3}
    assert placement.fixed_set(HAND, 2, 3, placement.static_set(2, 3, 3)) == (8, 4)
    # Prefill hot set of 3: keys 0, 3, 5 (3 before 5 on the tie); misses are keys 1, 2 and 4.
    hot = placement.prefill_hot_set(PREFILL, 3)
    assert hot == {0, 3, 5}
    assert placement.fixed_set(HAND, 2, 3, hot) == (8, 3)
    # with 2 slots the tie between keys 3 and 5 decides: key 3 stays, and keys 1, 2, 4 and 5 miss
    assert placement.prefill_hot_set(PREFILL, 2) == {0, 3}
    assert placement.fixed_set(HAND, 2, 3, placement.prefill_hot_set(PREFILL, 2)) == (8, 5)
    # Shared LRU of 3 slots from empty: only key 5 at step 1 hits (key 0 was evicted
    # by key 2, key 1 by key 3, then key 2 by key 0 and key 3 by key 4).
    assert placement.global_lru(HAND, 2, 3, 3) == (8, 7)


def _od_lru(seq, capacity):
    lru, miss = OrderedDict(), 0
    for k in seq:
        if k in lru:
            lru.move_to_end(k)
        else:
            miss += 1
            if len(lru) == capacity:
                lru.popitem(last=False)
            lru[k] = True
    return miss


def _random_trace(rng, steps, L, E, width, skew=1.2):
    p = 1.0 / np.arange(1, E + 1) ** skew
    p /= p.sum()
    perm = [rng.permutation(E) for _ in range(L)]
    tr = np.full((steps, L, width), -1, dtype=np.int32)
    for t in range(steps):
        for l in range(L):
            n = rng.integers(1, width + 1)
            tr[t, l, :n] = perm[l][rng.choice(E, n, p=p)]
    return tr


def test_global_lru_single_accesses_match_an_ordered_dict_lru():
    rng = np.random.default_rng(3)
    L, E = 3, 5
    for cap in (5, 7, 11, 15):
        tr = _random_trace(rng, 60, L, E, 1)
        seq = [l * E + int(tr[t, l, 0]) for t in range(60) for l in range(L)]
        acc, miss = placement.global_lru(tr.tolist(), L, E, cap)
        assert acc == len(seq) and miss == _od_lru(seq, cap)


def test_invariants():
    rng = np.random.default_rng(4)
    L, E = 4, 8
    tr = _random_trace(rng, 40, L, E, 4).tolist()
    keys = {l * E + e for step in tr for l in range(L) for e in step[l] if e >= 0}
    acc, m_lru = placement.global_lru(tr, L, E, L * E)
    assert m_lru == len(keys)                                     # only cold misses at full capacity
    assert placement.fixed_set(tr, L, E, placement.static_set(L, E, L * E)) == (acc, 0)
    counts = {k: 1 for k in range(L * E)}
    assert placement.fixed_set(tr, L, E, placement.prefill_hot_set(counts, L * E)) == (acc, 0)
    # fixed sets grow with the capacity (prefixes of one ranking): misses never rise
    pc = {k: int(c) for k, c in enumerate(rng.integers(0, 9, size=L * E))}
    prev_s = prev_p = None
    for cap in range(1, L * E + 1):
        _, ms = placement.fixed_set(tr, L, E, placement.static_set(L, E, cap))
        _, mp = placement.fixed_set(tr, L, E, placement.prefill_hot_set(pc, cap))
        assert prev_s is None or ms <= prev_s
        assert prev_p is None or mp <= prev_p
        prev_s, prev_p = ms, mp
    # single accesses: the LRU's misses never rise with the capacity (inclusion)
    tr1 = _random_trace(rng, 50, L, E, 1).tolist()
    m = [placement.global_lru(tr1, L, E, cap)[1] for cap in range(E, L * E + 1)]
    assert all(a >= b for a, b in zip(m, m[1:]))


@pytest.mark.parametrize("seed,L,E,width,steps", [(0, 4, 16, 8, 50), (1, 6, 32, 4, 80), (2, 3, 64, 16, 30)])
def test_native_replay_matches_the_oracle(ftlib, seed, L, E, width, steps):
    rng = np.random.default_rng(seed)
    tr = _random_trace(rng, steps, L, E, width)
    pc = rng.integers(0, 20, size=L * E).astype(np.int32)
    pcd = {k: int(c) for k, c in enumerate(pc)}
    trl = tr.tolist()
    for cap in sorted({E, E + 3, (L * E) // 3, (L * E) // 2, L * E}):
        want = placement.global_lru(trl, L, E, cap)
        assert ftlib.ft_placement_replay(ftlib.FT_PLACE_GLOBAL_LRU, L, E, cap, tr) == want
        want = placement.fixed_set(trl, L, E, placement.prefill_hot_set(pcd, cap))
        assert ftlib.ft_placement_replay(ftlib.FT_PLACE_PREFILL_HOT, L, E, cap, tr, pc) == want
        want = placement.fixed_set(trl, L, E, placement.static_set(L, E, cap))
        assert ftlib.ft_placement_replay(ftlib.FT_PLACE_STATIC_SPLIT, L, E, cap, tr) == want
    hand = np.full((3, 2, 3), -1, dtype=np.int32)
    for t, step in enumerate(HAND):
        for l, ids in enumerate(step):
            hand[t, l, :len(ids)] = ids
    assert ftlib.ft_placement_replay(ftlib.FT_PLACE_GLOBAL_LRU, 2, 3, 3, hand) == (8, 7)
    pch = np.array([PREFILL.get(k, 0) for k in range(6)], dtype=np.int32)
    assert ftlib.ft_placement_replay(ftlib.FT_PLACE_PREFILL_HOT, 2, 3, 3, hand, pch) == (8, 3)
    assert ftlib.ft_placement_replay(ftlib.FT_PLACE_STATIC_SPLIT, 2, 3, 3, hand) == (8, 4)


def test_native_replay_rejects_bad_arguments(ftlib):
    tr = np.zeros((2, 2, 1), dtype=np.int32)
    for policy, cap in ((ftlib.FT_PLACE_GLOBAL_LRU, 2), (ftlib.FT_PLACE_STATIC_SPLIT, 0),
                        (ftlib.FT_PLACE_STATIC_SPLIT, 13), (7, 4)):
        with pytest.raises(ftlib.FTError):
            ftlib.ft_placement_replay(policy, 2, 6, cap, tr)
    with pytest.raises(ftlib.FTError):
        ftlib.ft_placement_replay(ftlib.FT_PLACE_PREFILL_HOT, 2, 6, 4, tr, None)
