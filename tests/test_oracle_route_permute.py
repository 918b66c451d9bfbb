"""Pins of the oracle's gating and permutation against brute force and closed forms."""
import math

import numpy as np
import pytest

from oracle import moe


def brute_topk(z_row, k):
    """Selection by repeated scan: largest logit, lowest index on ties."""
    chosen = []
    for _ in range(k):
        best = None
        for e, v in enumerate(z_row):
            if e in chosen:
                continue
            if best is None or v > z_row[best]:
                best = e
        chosen.append(best)
    return chosen


@pytest.mark.parametrize("T,E,k,seed", [(7, 5, 2, 0), (9, 16, 2, 1), (5, 8, 8, 2), (6, 12, 1, 3), (33, 64, 6, 4)])
def test_route_matches_brute_force(T, E, k, seed):
    rng = np.random.default_rng(seed)
    # coarse values so that exact ties occur
    z = rng.integers(-3, 4, size=(T, E)).astype(np.float64) * 0.5
    idx, w = moe.route(z, k)
    for t in range(T):
        assert list(idx[t]) == brute_topk(list(z[t]), k)
        ez = [math.exp(z[t, e]) for e in idx[t]]
        s = sum(ez)
        for j in range(k):
            assert w[t, j] == pytest.approx(ez[j] / s, rel=1e-13)


def test_route_weights_sum_to_one_and_descend():
    rng = np.random.default_rng(5)
    z = rng.normal(size=(50, 32))
    idx, w = moe.route(z, 6)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-14)
    assert np.all(np.diff(w, axis=1) <= 0)


def test_route_k_equals_E_is_full_softmax():
    rng = np.random.default_rng(6)
    z = rng.normal(size=(4, 7))
    idx, w = moe.route(z, 7)
    for t in range(4):
        ez = np.exp(z[t] - z[t].max())
        p = ez / ez.sum()
        assert np.allclose(w[t], p[idx[t]], atol=1e-15)


def test_route_k1_weight_is_one():
    z = np.random.default_rng(7).normal(size=(10, 9))
    idx, w = moe.route(z, 1)
    assert np.all(w == 1.0)
    assert np.all(idx[:, 0] == np.argmax(z, axis=1))


def test_route_two_experts_closed_form():
    # E = 2, k = 2: the larger logit's weight is the logistic of the gap
    z = np.array([[0.3, -1.2], [2.0, 2.5], [0.0, 0.0]])
    idx, w = moe.route(z, 2)
    for t in range(3):
        gap = abs(z[t, 0] - z[t, 1])
        assert w[t, 0] == pytest.approx(1.0 / (1.0 + math.exp(-gap)), rel=1e-14)
    assert list(idx[2]) == [0, 1]          # exact tie: lower index first
    assert w[2, 0] == 0.5


def test_route_all_equal():
    z = np.zeros((3, 10))
    idx, w = moe.route(z, 4)
    assert (idx == np.arange(4)).all()
    assert np.all(w == 0.25)


def test_router_logits_hand_example():
    x = np.array([[1.0, 2.0, -1.0]])
    wr = np.array([[1.0, 0.0, 0.0], [0.5, 0.5, 0.5], [0.0, -1.0, 2.0]])  # stored [E, H]
    b = np.array([0.0, 1.0, -1.0])
    z = moe.router_logits(x, wr, b)
    assert z.tolist() == [[1.0, 2.0, -5.0]]


def brute_permute(idx, E):
    T, k = idx.shape
    counts = [0] * E
    for t in range(T):
        for j in range(k):
            counts[idx[t, j]] += 1
    offsets = [0]
    for e in range(E):
        offsets.append(offsets[-1] + counts[e])
    perm = []
    for e in range(E):
        for a in range(T * k):
            if idx.reshape(-1)[a] == e:
                perm.append(a)
    return counts, offsets, perm


@pytest.mark.parametrize("T,k,E,seed", [(1, 1, 3, 0), (5, 2, 4, 1), (16, 8, 32, 2), (64, 2, 16, 3), (3, 6, 256, 4)])
def test_permute_matches_brute_force(T, k, E, seed):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    counts, offsets, perm, inv = moe.permute(idx, E)
    bc, bo, bp = brute_permute(idx, E)
    assert counts.tolist() == bc
    assert offsets.tolist() == bo
    assert perm.tolist() == bp
    assert offsets[-1] == T * k
    assert sorted(perm.tolist()) == list(range(T * k))
    assert (perm[inv] == np.arange(T * k)).all()


def test_permute_empty_experts():
    idx = np.array([[2, 2], [2, 0]], dtype=np.int32)  # duplicate expert in a row is allowed here
    counts, offsets, perm, inv = moe.permute(idx, 4)
    assert counts.tolist() == [1, 0, 3, 0]
    assert offsets.tolist() == [0, 1, 1, 4, 4]
    assert perm.tolist() == [3, 0, 1, 2]


def test_near_ties_flags_only_close_gaps():
    z = np.array([[3.0, 2.0, 1.0, 0.9999999], [3.0, 2.0, 1.0, 0.0]])
    assert moe.near_ties(z, 3).tolist() == [True, False]
