"""Seeded synthetic inputs for the expert-cache MoE layer.

This module is the only code that both the CUDA path (through its Python
binding and ``bench.py``) and the fp64 oracle consume.  It holds none of the
layer's arithmetic: it draws weights, activations, router biases and decode
traces, and quantises weights into the stored formats (BF16, FP8 e4m3,
NVFP4, MXFP4).  Both sides read exactly the bytes produced here.

Draws use ``torch.Generator`` on the requested device, seeded per tensor from
``seed_for(...)`` (SplitMix64 mixing of the integer coordinates), so any one
(layer, expert, matrix) can be regenerated on its own.  The same seed gives
different numbers on CPU and CUDA; every consumer therefore takes the bytes
from one generation, never from two.

Weights are stored K-major (the contraction index contiguous):
  gate[n][h] = W_g[h][n]   shape [I, H]
  up[n][h]   = W_u[h][n]   shape [I, H]
  down[h][n] = W_d[n][h]   shape [H, I]
  router[e][h] = W_r[h][e] shape [E, H]
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import numpy as np
import torch

MASK64 = (1 << 64) - 1

# Stored weight formats (values match the C enum ft_wtype).
W_F32, W_BF16, W_FP8, W_NVFP4, W_MXFP4 = 0, 1, 2, 3, 4
WTYPE_NAMES = {W_F32: "f32", W_BF16: "bf16", W_FP8: "fp8e4m3", W_NVFP4: "nvfp4", W_MXFP4: "mxfp4"}

# tensor ids for seed derivation
_T_ROUTER, _T_BIAS, _T_GATE, _T_UP, _T_DOWN, _T_X, _T_PERM = 1, 2, 3, 4, 5, 6, 7


def _splitmix64(z: int) -> int:
    """SplitMix64 finaliser (Steele, Lea, Flood 2014)."""
    z = (z + 0x9E3779B97F4A7C15) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def seed_for(*coords: int) -> int:
    """Deterministic 63-bit seed from integer coordinates (seed, tensor, layer, ...)."""
    h = 0x243F6A8885A308D3
    for c in coords:
        h = _splitmix64(h ^ (int(c) & MASK64))
    return h & ((1 << 63) - 1)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    """fp32 N(0, std^2) draw from a generator seeded with ``seed``."""
    g = _gen(device, seed)
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    return t.mul_(std)


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    """Shape of a stacked MoE layer workload."""
    name: str
    hidden: int          # H
    n_experts: int       # E
    top_k: int           # k
    inter: int           # I
    n_layers: int        # L (logical)
    wtype: int           # stored expert weight format
    x_dtype: str = "bf16"  # activations / router weight dtype ("bf16" or "f32")
    seed: int = 0
    zipf_s: float = 0.0  # router bias exponent (0 = no bias)
    std: float = 0.02


# The workloads; sizes follow the problem statement.
TINY_F32 = MoEConfig("tiny_f32", 256, 16, 2, 128, 1, W_F32, "f32", seed=0)
DECODE_BF16 = MoEConfig("decode_bf16_40L", 2048, 256, 8, 512, 40, W_BF16, "bf16", seed=1, zipf_s=1.1)
PREFILL_BF16 = MoEConfig("prefill_bf16_40L", 2048, 256, 8, 512, 40, W_BF16, "bf16", seed=2, zipf_s=0.0)
NVFP4_43L = MoEConfig("nvfp4_43L", 4096, 256, 6, 2048, 43, W_NVFP4, "bf16", seed=3, zipf_s=1.1)
MXFP4_MIXED = MoEConfig("mxfp4_mixed_4L", 6144, 256, 8, 2048, 4, W_MXFP4, "bf16", seed=4, zipf_s=1.1)
CONFIGS = {c.name: c for c in (TINY_F32, DECODE_BF16, PREFILL_BF16, NVFP4_43L, MXFP4_MIXED)}


# ---------------------------------------------------------------- quantisers
# (data generation only: they decide which bytes are stored)

_E2M1_MAG = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1_encode(v: torch.Tensor) -> torch.Tensor:
    """fp32 -> 4-bit e2m1 code (uint8 in 0..15), round to nearest even, saturating at 6."""
    mag = _E2M1_MAG.to(v.device)
    a = v.abs().clamp(max=6.0)
    # index of the largest magnitude <= a
    lo = torch.bucketize(a, mag, right=True) - 1
    lo = lo.clamp(0, 7)
    hi = (lo + 1).clamp(max=7)
    dlo = a - mag[lo]
    dhi = mag[hi] - a
    up = (dhi < dlo) | ((dhi == dlo) & (lo % 2 == 1))
    code = torch.where(up & (hi != lo), hi, lo).to(torch.uint8)
    sign = ((v < 0) & (code != 0)).to(torch.uint8) << 3
    return code | sign


def _pack_nibbles(codes: torch.Tensor) -> torch.Tensor:
    """[..., K] 4-bit codes -> [..., K/2] bytes, element 2i in the low nibble."""
    c = codes.reshape(*codes.shape[:-1], codes.shape[-1] // 2, 2)
    return (c[..., 0] | (c[..., 1] << 4)).contiguous()


def e4m3_encode(v: torch.Tensor) -> torch.Tensor:
    """fp32 -> e4m3 (fn) byte, RNE, saturating at +-448."""
    return v.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)


def quant_nvfp4(w: torch.Tensor):
    """NVFP4: blocks of 16 along K; e4m3 block scale; fp32 tensor scale.

    Returns (codes [R, K/2] u8, scales [R, K/16] u8, global_scale float).
    """
    R, K = w.shape
    amax = w.abs().max().item()
    s_g = amax / (6.0 * 448.0) if amax > 0 else 1.0
    blk = w.reshape(R, K // 16, 16)
    bamax = blk.abs().amax(dim=-1)
    sc = e4m3_encode(bamax / (6.0 * s_g))
    sc_val = sc.view(torch.float8_e4m3fn).to(torch.float32)
    denom = (sc_val * s_g).unsqueeze(-1)
    q = torch.where(denom > 0, blk / torch.where(denom > 0, denom, torch.ones_like(denom)), torch.zeros_like(blk))
    codes = e2m1_encode(q.reshape(R, K))
    return _pack_nibbles(codes), sc.contiguous(), float(np.float32(s_g))


def quant_mxfp4(w: torch.Tensor):
    """MXFP4 (OCP MX v1.0): blocks of 32 along K; E8M0 scale 2^(floor(log2 amax) - 2).

    Returns (codes [R, K/2] u8, scales [R, K/32] u8).
    """
    R, K = w.shape
    blk = w.reshape(R, K // 32, 32)
    bamax = blk.abs().amax(dim=-1)
    safe = torch.where(bamax > 0, bamax, torch.ones_like(bamax))
    x = torch.floor(torch.log2(safe)) - 2.0
    x = torch.where(bamax > 0, x, torch.full_like(x, -127.0)).clamp(-127.0, 127.0)
    sbyte = (x + 127.0).to(torch.uint8)
    q = blk / torch.exp2(x).unsqueeze(-1)
    codes = e2m1_encode(q.reshape(R, K))
    return _pack_nibbles(codes), sbyte.contiguous()


def quant_fp8_rows128(w: torch.Tensor):
    """FP8 e4m3 with one fp32 scale per 128 consecutive K elements of a row.

    Returns (codes [R, K] u8, scales [R, K/128] f32).
    """
    R, K = w.shape
    blk = w.reshape(R, K // 128, 128)
    amax = blk.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    codes = e4m3_encode((blk / scale.unsqueeze(-1)).reshape(R, K))
    return codes.contiguous(), scale.to(torch.float32).contiguous()


# ---------------------------------------------------------------- weights

def _matrix(cfg: MoEConfig, tid: int, layer: int, expert: int, rows: int, cols: int, device):
    return normal((rows, cols), cfg.std, seed_for(cfg.seed, tid, layer, expert), device)


def _store(cfg: MoEConfig, w: torch.Tensor) -> Dict[str, object]:
    if cfg.wtype == W_F32:
        return {"w": w.contiguous()}
    if cfg.wtype == W_BF16:
        return {"w": w.to(torch.bfloat16).contiguous()}
    if cfg.wtype == W_FP8:
        c, s = quant_fp8_rows128(w)
        return {"codes": c, "scales": s}
    if cfg.wtype == W_NVFP4:
        c, s, g = quant_nvfp4(w)
        return {"codes": c, "scales": s, "gscale": g}
    if cfg.wtype == W_MXFP4:
        c, s = quant_mxfp4(w)
        return {"codes": c, "scales": s}
    raise ValueError(cfg.wtype)


def expert_weights(cfg: MoEConfig, layer: int, expert: int, device="cpu") -> Dict[str, Dict[str, object]]:
    """Stored components of one expert of physical layer ``layer``.

    {"gate": {...}, "up": {...}, "down": {...}} with each entry as produced by
    the format's quantiser (``{"w": tensor}`` for f32/bf16).
    """
    H, I = cfg.hidden, cfg.inter
    if cfg.name == TINY_F32.name:
        g, u, d = tiny_f32_draws()["experts"][expert]
        return {"gate": {"w": g.to(device)}, "up": {"w": u.to(device)}, "down": {"w": d.to(device)}}
    return {
        "gate": _store(cfg, _matrix(cfg, _T_GATE, layer, expert, I, H, device)),
        "up": _store(cfg, _matrix(cfg, _T_UP, layer, expert, I, H, device)),
        "down": _store(cfg, _matrix(cfg, _T_DOWN, layer, expert, H, I, device)),
    }


def router_weights(cfg: MoEConfig, layer: int, device="cpu"):
    """(W_r stored [E, H] in the activation dtype, bias [E] fp32)."""
    if cfg.name == TINY_F32.name:
        d = tiny_f32_draws()
        return d["router"].to(device), torch.zeros(cfg.n_experts, dtype=torch.float32, device=device)
    w = _matrix(cfg, _T_ROUTER, layer, 0, cfg.n_experts, cfg.hidden, device)
    w = w.to(torch.bfloat16) if cfg.x_dtype == "bf16" else w
    return w.contiguous(), zipf_bias(cfg, layer).to(device)


def zipf_bias(cfg: MoEConfig, layer: int) -> torch.Tensor:
    """Additive log-prior b_e = -s * ln(rank_l(e)), ranks a seeded permutation per layer.

    Adding b to the logits multiplies the softmax by a Zipf(s) prior over experts.
    """
    E = cfg.n_experts
    if cfg.zipf_s == 0.0:
        return torch.zeros(E, dtype=torch.float32)
    rng = np.random.default_rng(seed_for(cfg.seed, _T_PERM, layer))
    rank = rng.permutation(E) + 1
    return torch.from_numpy((-cfg.zipf_s * np.log(rank.astype(np.float64))).astype(np.float32))


def tiny_f32_draws():
    """The single tiny fp32 layer: numpy default_rng(0) draws in fp64, rounded to fp32.

    Draw order: W_r [H, E]; per expert W_g [H, I], W_u [H, I], W_d [I, H]; x [64, H].
    Returned in stored (K-major) layout.
    """
    global _TINY
    try:
        return _TINY
    except NameError:
        pass
    c = TINY_F32
    rng = np.random.default_rng(0)
    H, E, I = c.hidden, c.n_experts, c.inter
    wr = rng.normal(0.0, c.std, size=(H, E))
    experts = []
    for _ in range(E):
        wg = rng.normal(0.0, c.std, size=(H, I))
        wu = rng.normal(0.0, c.std, size=(H, I))
        wd = rng.normal(0.0, c.std, size=(I, H))
        experts.append(tuple(torch.from_numpy(np.ascontiguousarray(m.T).astype(np.float32)) for m in (wg, wu, wd)))
    x = rng.normal(0.0, 1.0, size=(64, H))
    _TINY = {
        "router": torch.from_numpy(np.ascontiguousarray(wr.T).astype(np.float32)),
        "experts": experts,
        "x": torch.from_numpy(x.astype(np.float32)),
    }
    return _TINY


# ---------------------------------------------------------------- activations

def activations(cfg: MoEConfig, T: int, tag: int = 0, device="cpu") -> torch.Tensor:
    """x [T, H] ~ N(0, 1) in the activation dtype (prefill chunks, single batches)."""
    if cfg.name == TINY_F32.name and T == 64 and tag == 0:
        return tiny_f32_draws()["x"].to(device)
    x = normal((T, cfg.hidden), 1.0, seed_for(cfg.seed, _T_X, tag), device)
    return x.to(torch.bfloat16) if cfg.x_dtype == "bf16" else x


class AR1Trace:
    """Decode trace of T independent chains h_t = 0.9 h_{t-1} + 0.436 N(0, 1), h_0 ~ N(0, 1).

    ``step(t)`` returns the hidden states of step t as [T, H] in the activation
    dtype; state is advanced in fp32 on ``device``.  Every layer of a step
    sees the same hidden state.
    """

    RHO, SIGMA = 0.9, 0.436

    def __init__(self, cfg: MoEConfig, T: int, device="cpu", tag: int = 0):
        self.cfg, self.T, self.device, self.tag = cfg, T, device, tag
        self.t = 0
        self.h = normal((T, cfg.hidden), 1.0, seed_for(cfg.seed, _T_X, 1000 + tag, T, 0), device)

    def next(self) -> torch.Tensor:
        if self.t > 0:
            eps = normal((self.T, self.cfg.hidden), 1.0, seed_for(self.cfg.seed, _T_X, 1000 + self.tag, self.T, self.t), self.device)
            self.h = self.h.mul_(self.RHO).add_(eps, alpha=self.SIGMA)
        self.t += 1
        h = self.h
        return h.to(torch.bfloat16) if self.cfg.x_dtype == "bf16" else h.clone()


def lru_trace_keys(n_keys: int, length: int, seed: int, locality: float = 0.8) -> np.ndarray:
    """A key sequence with temporal locality (for LRU simulator checks)."""
    rng = np.random.default_rng(seed)
    out = np.empty(length, dtype=np.int64)
    recent = []
    for i in range(length):
        if recent and rng.random() < locality:
            out[i] = recent[int(rng.integers(0, len(recent)))]
        else:
            out[i] = int(rng.integers(0, n_keys))
        recent.append(int(out[i]))
        recent = recent[-8:]
    return out
