"""Pins of the oracle's expert FFN, layer sum, combine and split against hand values and invariants."""
import numpy as np
import pytest

from oracle import moe

SIGMOID_1 = 0.7310585786300049   # 1 / (1 + e^-1)
SIGMOID_M2 = 0.11920292202211755  # 1 / (1 + e^2)


def test_ffn_hand_example():
    # H = 2, I = 1: G = x.gate = 0.5 + 0.5 = 1, U = x.up = 3, A = silu(1) * 3,
    # Y = A * [2, -1]
    x = np.array([[1.0, 2.0]])
    gate = np.array([[0.5, 0.25]])      # [I, H]
    up = np.array([[1.0, 1.0]])         # [I, H]
    down = np.array([[2.0], [-1.0]])    # [H, I]
    y = moe.expert_ffn(x, gate, up, down)
    a = 1.0 * SIGMOID_1 * 3.0
    assert y[0].tolist() == pytest.approx([2 * a, -a], rel=1e-15)


def test_ffn_gate_and_up_are_not_interchangeable():
    # silu is not symmetric: swapping gate and up changes the result (G = -2, U = 1 here)
    x = np.array([[1.0, -1.0]])
    gate = np.array([[-1.0, 1.0]])
    up = np.array([[0.5, -0.5]])
    down = np.array([[1.0]])
    y = moe.expert_ffn(x, gate, up, down)
    assert y[0, 0] == pytest.approx(-2.0 * SIGMOID_M2 * 1.0, rel=1e-14)
    y_sw = moe.expert_ffn(x, up, gate, down)
    assert y_sw[0, 0] == pytest.approx(1.0 * SIGMOID_1 * -2.0, rel=1e-14)


def scalar_ffn(x, gate, up, down):
    """Scalar triple loop over the stored layouts."""
    H = len(x)
    I = len(gate)
    A = []
    for n in range(I):
        g = sum(x[h] * gate[n][h] for h in range(H))
        u = sum(x[h] * up[n][h] for h in range(H))
        A.append(g / (1.0 + np.exp(-g)) * u)
    return [sum(A[n] * down[h][n] for n in range(I)) for h in range(H)]


def test_ffn_matches_scalar_loops_rectangular():
    rng = np.random.default_rng(0)
    H, I = 5, 3                       # rectangular: a transposed operand would not fit
    x = rng.normal(size=(2, H))
    gate, up, down = rng.normal(size=(I, H)), rng.normal(size=(I, H)), rng.normal(size=(H, I))
    y = moe.expert_ffn(x, gate, up, down)
    for r in range(2):
        assert y[r] == pytest.approx(scalar_ffn(x[r], gate, up, down), rel=1e-12)


def test_ffn_zero_input_and_linearity_in_down():
    rng = np.random.default_rng(1)
    gate, up, down = rng.normal(size=(4, 6)), rng.normal(size=(4, 6)), rng.normal(size=(6, 4))
    assert np.all(moe.expert_ffn(np.zeros((1, 6)), gate, up, down) == 0)
    x = rng.normal(size=(3, 6))
    assert np.allclose(moe.expert_ffn(x, gate, up, 2 * down), 2 * moe.expert_ffn(x, gate, up, down), rtol=1e-14)


def _random_experts(rng, E, H, I, scale=0.3):
    ex = [(rng.normal(size=(I, H)) * scale, rng.normal(size=(I, H)) * scale, rng.normal(size=(H, I)) * scale)
          for _ in range(E)]
    return lambda e: ex[e]


def test_identical_experts_reduce_to_one_dense_ffn():
    rng = np.random.default_rng(2)
    H, I, E, k, T = 8, 6, 5, 3, 7
    g, u, d = rng.normal(size=(I, H)), rng.normal(size=(I, H)), rng.normal(size=(H, I))
    x = rng.normal(size=(T, H))
    z = rng.normal(size=(T, E))
    idx, w = moe.route(z, k)
    out = moe.moe_layer(x, idx, w, lambda e: (g, u, d))
    assert np.allclose(out, moe.dense_swiglu(x, g, u, d), rtol=1e-12, atol=1e-14)


def test_grouped_evaluation_equals_token_loop():
    # evaluating expert by expert over permuted rows and combining gives the token-loop sum
    rng = np.random.default_rng(3)
    H, I, E, k, T = 6, 4, 7, 2, 11
    ex = _random_experts(rng, E, H, I)
    x = rng.normal(size=(T, H))
    idx, w = moe.route(rng.normal(size=(T, E)), k)
    counts, offsets, perm, inv = moe.permute(idx, E)
    Y = np.zeros((T * k, H))
    for e in range(E):
        rows = perm[offsets[e]:offsets[e + 1]]
        if len(rows):
            Y[offsets[e]:offsets[e + 1]] = moe.expert_ffn(x[rows // k], *ex(e))
    out = moe.combine(Y, inv, w, k)
    assert np.allclose(out, moe.moe_layer(x, idx, w, ex), rtol=1e-13, atol=1e-15)


def test_split_partials_add_up_exactly():
    # GPU part + external part = whole layer, for every split of the experts
    rng = np.random.default_rng(4)
    H, I, E, k, T = 6, 4, 8, 3, 9
    ex = _random_experts(rng, E, H, I)
    x = rng.normal(size=(T, H))
    idx, w = moe.route(rng.normal(size=(T, E)), k)
    full = moe.moe_layer(x, idx, w, ex)
    for mask in range(0, 1 << E, 37):
        C = [e for e in range(E) if mask >> e & 1]
        G = [e for e in range(E) if not mask >> e & 1]
        part = moe.moe_layer(x, idx, w, ex, only=C)
        gpu = moe.moe_layer(x, idx, w, ex, only=G)
        assert np.allclose(gpu + part, full, rtol=1e-13, atol=1e-15)
        # the same split through combine's skip + partial
        counts, offsets, perm, inv = moe.permute(idx, E)
        Y = np.zeros((T * k, H))
        for a in range(T * k):
            Y[inv[a]] = moe.expert_ffn(x[a // k:a // k + 1], *ex(idx.reshape(-1)[a]))[0]
        skip = np.isin(idx, C)
        out = moe.combine(Y, inv, w, k, skip=skip, partial=part)
        assert np.allclose(out, full, rtol=1e-13, atol=1e-15)


def test_single_token_single_expert_layer():
    x = np.array([[1.0, 2.0]])
    gate = np.array([[0.5, 0.25]])
    up = np.array([[1.0, 1.0]])
    down = np.array([[2.0], [-1.0]])
    idx = np.array([[0]], dtype=np.int32)
    out = moe.moe_layer(x, idx, np.array([[1.0]]), lambda e: (gate, up, down))
    a = SIGMOID_1 * 3.0
    assert out[0].tolist() == pytest.approx([2 * a, -a], rel=1e-15)
