"""The routed-expert MoE layer in fp64 -- plain definitions, no blocking or fusion.

What the layer computes is fixed by [Review] §2 opening and §2.5 "最后说结果为什么
是精确的": the cache, the miss split and streaming change only where experts are
evaluated; GPU and host partial sums are added and the MoE output is kept
exactly.  So the oracle evaluates the layer directly:

    out[t] = sum_{j<k} w[t,j] * FFN_{e[t,j]}(x[t])   (+ an external partial P[t])

with FFN_e(x) = W_d[e]^T (silu(W_g[e]^T x) * (W_u[e]^T x)), silu(g) = g / (1 + e^-g).
Each expert is an independent set of FFN weights ([Review] §1, "专家 ... 本质是
一组独立的前馈网络权重").  Gating: softmax over all E experts, the k most
probable kept (lowest index on ties), their probabilities renormalised.

Weights arrive in stored K-major layout: gate [I, H], up [I, H], down [H, I],
router [E, H].  Matrix products use numpy (a library primitive) in fp64.
"""
from __future__ import annotations

from typing import Callable, Dict, Iterable, Optional, Tuple

import numpy as np

from . import formats


def router_logits(x: np.ndarray, w_router: np.ndarray, bias: Optional[np.ndarray] = None) -> np.ndarray:
    """z[t, e] = sum_h x[t, h] W_r[h, e] + b[e], in fp64 from the stored values."""
    z = np.asarray(x, np.float64) @ np.asarray(w_router, np.float64).T
    if bias is not None:
        z = z + np.asarray(bias, np.float64)[None, :]
    return z


def softmax(z: np.ndarray) -> np.ndarray:
    """Row softmax over all experts, fp64."""
    z = np.asarray(z, np.float64)
    ez = np.exp(z - z.max(axis=-1, keepdims=True))
    return ez / ez.sum(axis=-1, keepdims=True)


def route(z: np.ndarray, k: int) -> Tuple[np.ndarray, np.ndarray]:
    """Top-k gating: (idx [T, k] int32, w [T, k] fp64).

    Experts are ranked by descending softmax probability, ties to the lower
    index; softmax is strictly increasing in the logit, so the ranking is taken
    on the logits themselves (a stable sort of -z keeps equal logits in index
    order).  The chosen probabilities are renormalised to sum to one, which is
    the same as a softmax over the k chosen logits.
    """
    z = np.asarray(z, np.float64)
    order = np.argsort(-z, axis=1, kind="stable")[:, :k]
    p = softmax(z)
    sel = np.take_along_axis(p, order, axis=1)
    w = sel / sel.sum(axis=1, keepdims=True)
    return order.astype(np.int32), w


def permute(idx: np.ndarray, n_experts: int):
    """Group the T*k assignments a = t*k + j by expert.

    Returns counts [E], offsets [E+1] (exclusive prefix sum, offsets[E] = T*k),
    perm [T*k] (perm[offsets[e] + r] = the r-th assignment routed to e, in
    ascending a) and inv [T*k] (inv[perm[p]] = p).
    """
    a = np.asarray(idx).reshape(-1).astype(np.int64)
    counts = np.bincount(a, minlength=n_experts).astype(np.int32)
    offsets = np.zeros(n_experts + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    perm = np.argsort(a, kind="stable").astype(np.int32)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size, dtype=np.int32)
    return counts, offsets, perm, inv


def silu(g: np.ndarray) -> np.ndarray:
    return g / (1.0 + np.exp(-g))


def expert_ffn(X: np.ndarray, gate: np.ndarray, up: np.ndarray, down: np.ndarray,
               act_round: Optional[Callable[[np.ndarray], np.ndarray]] = None,
               x_round: Optional[Callable[[np.ndarray], np.ndarray]] = None) -> np.ndarray:
    """SwiGLU expert on rows X [m, H]: Y = (silu(X gate^T) * (X up^T)) down^T, fp64.

    ``x_round`` and ``act_round`` apply the rounding the evaluated kernel
    declares for its token rows X and for the intermediate A = silu(G) * U
    (None: not rounded), e.g. the FP4 activation rules of ``formats``.
    """
    X = np.asarray(X, np.float64)
    if x_round is not None:
        X = x_round(X)
    G = X @ gate.T
    U = X @ up.T
    A = silu(G) * U
    if act_round is not None:
        A = act_round(A)
    return A @ down.T


class ExpertSource:
    """fp64 (gate, up, down) of an expert, decoded from synth's stored components once."""

    def __init__(self, fetch: Callable[[int], Dict[str, dict]], wtype: int):
        self.fetch, self.wtype, self.cache = fetch, wtype, {}

    def __call__(self, e: int):
        if e not in self.cache:
            c = self.fetch(e)
            self.cache[e] = tuple(formats.dequant(c[m], self.wtype) for m in ("gate", "up", "down"))
        return self.cache[e]


def combine(Y: np.ndarray, inv: np.ndarray, w: np.ndarray, k: int,
            skip: Optional[np.ndarray] = None, partial: Optional[np.ndarray] = None) -> np.ndarray:
    """out[t] = sum_j w[t,j] Y[inv[t k + j]] (+ P[t]); assignments with skip[t,j] add nothing."""
    T = w.shape[0]
    out = np.zeros((T, Y.shape[1]), dtype=np.float64)
    for t in range(T):
        for j in range(k):
            if skip is not None and skip[t, j]:
                continue
            out[t] += w[t, j] * Y[inv[t * k + j]]
    if partial is not None:
        out += np.asarray(partial, np.float64)
    return out


def moe_layer(x: np.ndarray, idx: np.ndarray, w: np.ndarray, experts: Callable[[int], tuple],
              act_round=None, only: Optional[Iterable[int]] = None, x_round=None) -> np.ndarray:
    """The layer output for given routing, token by token.

    out[t] = sum_j w[t,j] FFN_{idx[t,j]}(x[t]).  With ``only`` given, the sum is
    restricted to experts in that set (the partial output of a subset, as the
    external part of a split).
    """
    x = np.asarray(x, np.float64)
    T, k = idx.shape
    keep = None if only is None else set(int(e) for e in only)
    out = np.zeros((T, experts(int(idx[0, 0]))[2].shape[0]), dtype=np.float64)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            if keep is not None and e not in keep:
                continue
            g, u, d = experts(e)
            out[t] += w[t, j] * expert_ffn(x[t:t + 1], g, u, d, act_round, x_round)[0]
    return out


def dense_swiglu(x: np.ndarray, gate: np.ndarray, up: np.ndarray, down: np.ndarray) -> np.ndarray:
    """One dense SwiGLU FFN (what a layer of identical experts must reduce to)."""
    return expert_ffn(x, gate, up, down)


def near_ties(z: np.ndarray, k: int, rel: float = 1e-5) -> np.ndarray:
    """Tokens whose k-th and (k+1)-th logits are closer than rel * max|z| (routing may flip)."""
    z = np.asarray(z, np.float64)
    if k >= z.shape[1]:
        return np.zeros(z.shape[0], dtype=bool)
    s = -np.sort(-z, axis=1)
    scale = np.maximum(np.abs(z).max(axis=1), 1e-30)
    return (s[:, k - 1] - s[:, k]) < rel * scale
