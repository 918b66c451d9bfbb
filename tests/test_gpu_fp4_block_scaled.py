"""The block-scaled FP4 tensor-core path of NVFP4 / MXFP4 experts (small and large batches).

The weights go to tcgen05.mma kind::mxf4nvf4 packed, with their block scales;
the token rows and the intermediate silu(G)*U are quantised to the weights'
format by the rule stated in oracle/formats.py (quant_act_nvfp4 /
quant_act_mxfp4).  The quantiser decides integers (codes and scale bytes)
from floating point, so it must agree with the oracle's rule exactly on the
same fp32 inputs, ties included; the layer then matches the oracle evaluated
on quantised token rows and intermediate, at the bar for quantised
activations (relative Frobenius <= 1e-2, max |err| <= 2e-2 * max |ref|).
"""
import numpy as np
import pytest
import torch

import synth
from conftest import assert_close_layer, rel_fro
from oracle import formats, moe

pytestmark = pytest.mark.gpu
DEV = "cuda"
QUANT = {synth.W_NVFP4: formats.quant_act_nvfp4, synth.W_MXFP4: formats.quant_act_mxfp4}


@pytest.fixture(scope="module")
def ft(ftlib):
    assert torch.cuda.is_available()
    ftlib.ft_expert_set_fp4_path(ftlib.FT_FP4_BLOCK_SCALED)
    yield ftlib
    ftlib.ft_expert_set_fp4_path(ftlib.FT_FP4_BLOCK_SCALED)


def _decode(codes: np.ndarray, scales: np.ndarray, wtype) -> np.ndarray:
    if wtype == synth.W_NVFP4:
        return formats.dequant_nvfp4(codes, scales, 1.0)
    return formats.dequant_mxfp4(codes, scales)


@pytest.mark.parametrize("wtype", [synth.W_NVFP4, synth.W_MXFP4])
@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_quantiser_agrees_with_the_oracle_rule(ft, wtype, dt):
    rng = np.random.default_rng(5)
    K = 512
    x = rng.normal(size=(48, K)) * 10.0 ** rng.integers(-3, 3, size=(48, 1))
    # rows whose blocks put values exactly on e2m1 midpoints (scale 1: amax 6 / amax 4..7.99)
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, -0.25, -2.5, -5.0, 0.0, 1.0, 3.0, -6.0, 4.0])
    x[0] = np.tile(ties, K // 16)
    x[1] = np.tile(ties * 0.5, K // 16)
    x[2] = 0.0                                     # all-zero blocks
    x[3, :] = 1e-30                                # tiny values (scale underflow)
    xt = torch.from_numpy(x.astype(np.float32)).to(DEV)
    if dt == "bf16":
        xt = xt.to(torch.bfloat16)
    blk = 16 if wtype == synth.W_NVFP4 else 32
    q = torch.empty(48, K // 2, dtype=torch.uint8, device=DEV)
    s = torch.empty(48, K // blk, dtype=torch.uint8, device=DEV)
    ft.ft_debug_quant_fp4(xt, wtype, q, s)
    torch.cuda.synchronize()
    got = _decode(q.cpu().numpy(), s.cpu().numpy(), wtype)
    want = QUANT[wtype](formats.to_f64(xt).astype(np.float32))
    assert np.array_equal(got, want), np.argwhere(got != want)[:5]


def _setup(ft, wtype, H, I, E, k, T, seed, skewed=False):
    assert k <= E, "each token routes to k distinct experts"
    cfg = synth.MoEConfig(f"bs{wtype}_{H}_{I}", H, E, k, I, 1, wtype, "bf16", seed=seed)
    L = ft.ft_expert_layout_get(wtype, H, I)
    S = int(L.bytes)
    n_slots = E + 3
    pool = torch.zeros(n_slots * S, dtype=torch.uint8, device=DEV)
    rng = np.random.default_rng(seed)
    slot_perm = rng.permutation(n_slots)[:E]
    comps = {}
    for e in range(E):
        comps[e] = synth.expert_weights(cfg, 0, e, DEV)
        ft.pack_expert(comps[e], wtype, L, pool[slot_perm[e] * S:(slot_perm[e] + 1) * S])
    x = synth.activations(cfg, T, tag=5, device=DEV)
    if skewed:
        p = 1.0 / np.arange(1, E + 1) ** 1.2
        p /= p.sum()
        idx = np.stack([rng.choice(E, k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    else:
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    return cfg, S, n_slots, pool, slot_perm, comps, x, idx


def _run(ft, x, k, I, E, wtype, perm, offsets, slot_of, pool, S, n_slots):
    T, H = x.shape
    y = torch.full((T * k, H), float("nan"), dtype=torch.float32, device=DEV)
    ws = torch.empty(ft.ft_expert_grouped_workspace(T, k, H, I), dtype=torch.uint8, device=DEV)
    ft.ft_expert_grouped(x, k, I, E, wtype, torch.from_numpy(perm).to(DEV), torch.from_numpy(offsets).to(DEV),
                         torch.from_numpy(slot_of).to(DEV), pool, S, n_slots, y, ws)
    torch.cuda.synchronize()
    assert ft.ft_get_device_error() == 0
    return y.cpu().numpy()


@pytest.mark.parametrize("wtype,H,I,E,k,T,seed,skewed", [
    (synth.W_NVFP4, 4096, 2048, 16, 6, 1, 0, False),     # one token: gate/up and down split along K
    (synth.W_NVFP4, 4096, 2048, 64, 6, 64, 1, True),     # the NVFP4 stack's decode shape, T = 64
    (synth.W_NVFP4, 1024, 512, 8, 4, 37, 2, False),      # ragged token chunks
    (synth.W_NVFP4, 512, 256, 4, 2, 200, 3, False),      # 100 rows per expert: two token chunks
    (synth.W_MXFP4, 6144, 2048, 16, 8, 1, 4, False),     # the MXFP4 trace's decode shape
    (synth.W_MXFP4, 6144, 2048, 32, 8, 16, 5, True),
    (synth.W_MXFP4, 1024, 768, 8, 3, 50, 6, False),
    (synth.W_MXFP4, 256, 256, 2, 2, 1, 7, False),        # one stage per product
    # large batches (T*k >= 2048): 128 token rows x 128 weight rows per tile
    (synth.W_NVFP4, 1024, 512, 16, 8, 300, 8, False),    # 150 rows per expert: a ragged second row tile
    (synth.W_NVFP4, 4096, 2048, 8, 6, 700, 9, True),     # the NVFP4 stack's shape, heavy and light experts
    (synth.W_MXFP4, 2048, 1024, 8, 4, 600, 10, False),
    (synth.W_MXFP4, 6144, 2048, 8, 8, 260, 13, False),   # the MXFP4 trace's shape, 260 rows per expert
])
def test_block_scaled_expert_parity(ft, wtype, H, I, E, k, T, seed, skewed):
    cfg, S, n_slots, pool, slot_perm, comps, x, idx = _setup(ft, wtype, H, I, E, k, T, seed, skewed)
    counts, offsets, perm, inv = moe.permute(idx, E)
    slot_of = slot_perm.astype(np.int32).copy()
    slot_of[E - 1] = -1                                   # not evaluated: rows untouched
    Y = _run(ft, x, k, I, E, wtype, perm, offsets, slot_of, pool, S, n_slots)
    xs = formats.to_f64(x)
    got, ref = [], []
    for e in range(E - 1):
        rows = np.arange(offsets[e], offsets[e + 1])
        if rows.size == 0:
            continue
        g, u, d = (formats.dequant(comps[e][m], wtype) for m in ("gate", "up", "down"))
        ref.append(moe.expert_ffn(xs[perm[rows] // k], g, u, d, act_round=QUANT[wtype], x_round=QUANT[wtype]))
        got.append(Y[rows])
    rows = np.arange(offsets[E - 1], offsets[E])
    assert np.isnan(Y[rows]).all()
    got, ref = np.concatenate(got), np.concatenate(ref)
    assert np.isfinite(got).all()
    assert_close_layer(got, ref, fro=1e-2)
    # the same arithmetic up to the fp32 accumulation order: far inside the bar
    assert rel_fro(got, ref) < 2e-3


def test_block_scaled_independent_of_slot_and_other_experts(ft):
    """An expert's rows are the same bit for bit whether it is evaluated alone or with others,
    and whatever slot holds it (fixed-order reductions, splits summed in split order)."""
    wtype, H, I, E, k, T = synth.W_NVFP4, 2048, 1024, 8, 4, 9
    cfg, S, n_slots, pool, slot_perm, comps, x, idx = _setup(ft, wtype, H, I, E, k, T, 11)
    counts, offsets, perm, inv = moe.permute(idx, E)
    full = _run(ft, x, k, I, E, wtype, perm, offsets, slot_perm.astype(np.int32), pool, S, n_slots)
    for e in range(E):
        so = np.full(E, -1, dtype=np.int32)
        so[e] = slot_perm[e]
        alone = _run(ft, x, k, I, E, wtype, perm, offsets, so, pool, S, n_slots)
        rows = np.arange(offsets[e], offsets[e + 1])
        assert np.array_equal(alone[rows], full[rows])
    # move expert 0 to another slot
    moved = pool.clone()
    spare = n_slots - 1 if (n_slots - 1) not in slot_perm else [s for s in range(n_slots) if s not in slot_perm][0]
    moved[spare * S:(spare + 1) * S] = pool[slot_perm[0] * S:(slot_perm[0] + 1) * S]
    so = slot_perm.astype(np.int32).copy()
    so[0] = spare
    again = _run(ft, x, k, I, E, wtype, perm, offsets, so, moved, S, n_slots)
    assert np.array_equal(again, full)


def test_expansion_path_still_available(ft):
    """FT_FP4_EXPAND_BF16 takes the exact expansion at small batches (x and the intermediate in bf16)."""
    wtype, H, I, E, k, T = synth.W_MXFP4, 1024, 512, 4, 2, 6
    cfg, S, n_slots, pool, slot_perm, comps, x, idx = _setup(ft, wtype, H, I, E, k, T, 12)
    counts, offsets, perm, inv = moe.permute(idx, E)
    ft.ft_expert_set_fp4_path(ft.FT_FP4_EXPAND_BF16)
    try:
        Y = _run(ft, x, k, I, E, wtype, perm, offsets, slot_perm.astype(np.int32), pool, S, n_slots)
    finally:
        ft.ft_expert_set_fp4_path(ft.FT_FP4_BLOCK_SCALED)
    xs = formats.to_f64(x)
    ref = np.concatenate([moe.expert_ffn(xs[perm[offsets[e]:offsets[e + 1]] // k],
                                         *(formats.dequant(comps[e][m], wtype) for m in ("gate", "up", "down")),
                                         act_round=formats.round_to_bf16) for e in range(E)])
    assert_close_layer(Y, ref, fro=1e-2)
    assert rel_fro(Y, ref) < 2e-3
