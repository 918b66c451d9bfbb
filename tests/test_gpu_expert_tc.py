"""Parity of the tensor-core (tcgen05) grouped expert path against the fp64 oracle, through the C ABI.

(bf16 experts of a single decode token, T*k <= FT_CC_MAX_ASSIGNMENTS, run on the CUDA
cores with an fp32 intermediate; those cases compare with the unrounded reference.)

bf16 weights run on the tensor cores at every batch size: x is rounded to
bf16 and the intermediate silu(G)*U is rounded to bf16 before the down
product.  The oracle applies the same two roundings (x is already bf16 here;
the intermediate goes through formats.round_to_bf16), and the bar is the
tensor-core one: relative Frobenius error <= 1e-2, max |err| <= 2e-2 * max |ref|.
Batches below FT_TC_WIDE_ASSIGNMENTS use the small-batch tiling (weights on
the MMA's M side, up to 64 token rows on N, K split when few experts are
routed), larger ones 256-column weight tiles against 128-row token tiles; both
are covered, including split and multi-chunk cases.
"""
import numpy as np
import pytest
import torch

import synth
from conftest import assert_close_layer, bf16_act_round, rel_fro
from oracle import formats, moe

pytestmark = pytest.mark.gpu
DEV = "cuda"
TC_WIDE = 2048  # FT_TC_WIDE_ASSIGNMENTS in include/ft.h


@pytest.fixture(scope="module")
def ft(ftlib):
    assert torch.cuda.is_available()
    return ftlib


def _setup(ft, H, I, E, k, T, seed, skewed=False, wtype=synth.W_BF16, xdt="bf16"):
    cfg = synth.MoEConfig(f"tc_{H}_{I}_{E}", H, E, k, I, 1, wtype, xdt, seed=seed)
    L = ft.ft_expert_layout_get(wtype, H, I)
    S = int(L.bytes)
    n_slots = E + 5
    pool = torch.zeros(n_slots * S, dtype=torch.uint8, device=DEV)
    rng = np.random.default_rng(seed)
    slot_perm = rng.permutation(n_slots)[:E]
    comps = {}
    for e in range(E):
        comps[e] = synth.expert_weights(cfg, 0, e, DEV)
        ft.pack_expert(comps[e], wtype, L, pool[slot_perm[e] * S:(slot_perm[e] + 1) * S])
    x = synth.activations(cfg, T, tag=5, device=DEV)
    if skewed:
        # a few heavy experts (several 128-row tiles) and a tail of light ones
        p = 1.0 / np.arange(1, E + 1) ** 1.2
        p /= p.sum()
        idx = np.stack([rng.choice(E, k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    else:
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    return cfg, L, S, n_slots, pool, slot_perm, comps, x, idx


def _run(ft, x, k, I, E, perm, offsets, slot_of, pool, S, n_slots, wtype=synth.W_BF16):
    T, H = x.shape
    y = torch.full((T * k, H), float("nan"), dtype=torch.float32, device=DEV)
    ws = torch.empty(ft.ft_expert_grouped_workspace(T, k, H, I), dtype=torch.uint8, device=DEV)
    ft.ft_expert_grouped(x, k, I, E, wtype, torch.from_numpy(perm).to(DEV),
                         torch.from_numpy(offsets).to(DEV), torch.from_numpy(slot_of).to(DEV), pool, S, n_slots, y, ws)
    torch.cuda.synchronize()
    assert ft.ft_get_device_error() == 0
    return y.cpu().numpy()


@pytest.mark.parametrize("H,I,E,k,T,seed,skewed", [
    (256, 128, 8, 8, 300, 0, False),      # 300 rows per expert: 3 row tiles, ragged tail; one n-tile
    (512, 256, 4, 2, 1100, 1, False),     # ~550 rows per expert, 5 row tiles
    (2048, 512, 32, 8, 512, 2, False),    # the decode/prefill expert shape, ~128 rows per expert
    (1024, 384, 16, 4, 700, 3, True),     # skewed counts: heavy and light experts, I = 3 x 128
    (768, 256, 64, 8, 256, 4, False),     # exactly 2048 assignments; ~32 rows per expert (mostly-empty tiles)
    (2048, 512, 32, 8, 1, 5, False),      # one decode token: 8 experts of one row, 128-column tiles
    (2048, 512, 64, 8, 16, 6, True),      # decode batch of 16, skewed
    (256, 128, 8, 2, 3, 7, False),        # tiny: H = 256, I = 128
    (4096, 256, 16, 6, 40, 8, False),     # wide hidden, narrow intermediate
    (4096, 512, 16, 4, 1, 10, False),     # one token, 4 experts: gate/up K split 4 ways
    (256, 2048, 8, 2, 1, 11, False),      # one token, 2 experts: down K split 4 ways
    (512, 256, 2, 2, 100, 12, False),     # 100 rows per expert: two token chunks on the small-batch tiling
    (256, 128, 64, 8, 250, 13, True),     # 2000 assignments over 64 experts, heavy and light
    (512, 256, 8, 8, 255, 14, False),     # 255 rows per expert: four 64-row chunks each
])
def test_tc_expert_grouped_parity(ft, H, I, E, k, T, seed, skewed):
    cfg, L, S, n_slots, pool, slot_perm, comps, x, idx = _setup(ft, H, I, E, k, T, seed, skewed)
    counts, offsets, perm, inv = moe.permute(idx, E)
    slot_of = slot_perm.astype(np.int32).copy()
    skipped = {E - 1, 1}
    slot_of[E - 1] = -1                      # not evaluated
    slot_of[1] = -2                          # evaluated elsewhere
    Y = _run(ft, x, k, I, E, perm, offsets, slot_of, pool, S, n_slots)
    xs = formats.to_f64(x)
    got, ref = [], []
    for e in range(E):
        rows = np.arange(offsets[e], offsets[e + 1])
        if e in skipped:
            assert np.isnan(Y[rows]).all(), "rows of skipped experts must be left untouched"
            continue
        g, u, d = (formats.dequant(comps[e][m], synth.W_BF16) for m in ("gate", "up", "down"))
        ref.append(moe.expert_ffn(xs[perm[rows] // k], g, u, d, act_round=bf16_act_round(T, k)))
        got.append(Y[rows])
    got, ref = np.concatenate(got), np.concatenate(ref)
    assert np.isfinite(got).all()
    assert_close_layer(got, ref, fro=1e-2)
    # both sides round the same intermediate (bf16 on the tensor cores, fp32 on the CUDA cores
    # for one-token batches): they differ only by fp32 sums and bf16 rounding-boundary cases
    assert rel_fro(got, ref) < 2e-3


def test_tc_both_tilings(ft):
    """T*k just below FT_TC_WIDE_ASSIGNMENTS (small-batch tiling) and at it (large-batch tiling)."""
    H, I, E, k = 512, 256, 8, 8
    T_narrow, T_wide = TC_WIDE // k - 1, TC_WIDE // k
    cfg, L, S, n_slots, pool, slot_perm, comps, x, idx = _setup(ft, H, I, E, k, T_wide, 9)
    experts = {e: tuple(formats.dequant(comps[e][m], synth.W_BF16) for m in ("gate", "up", "down")) for e in range(E)}
    slot_of = slot_perm.astype(np.int32)
    xs = formats.to_f64(x)
    for T in (T_narrow, T_wide):
        counts, offsets, perm, inv = moe.permute(idx[:T], E)
        Y = _run(ft, x[:T], k, I, E, perm, offsets, slot_of, pool, S, n_slots)
        ref = np.concatenate([moe.expert_ffn(xs[perm[offsets[e]:offsets[e + 1]] // k], *experts[e],
                                             act_round=formats.round_to_bf16) for e in range(E)])
        assert_close_layer(Y, ref, fro=1e-2)
        assert rel_fro(Y, ref) < 2e-3
        ref32 = np.concatenate([moe.expert_ffn(xs[perm[offsets[e]:offsets[e + 1]] // k], *experts[e])
                                for e in range(E)])
        assert rel_fro(Y, ref32) > 1e-5       # the intermediate is visibly rounded to bf16


def test_tc_independent_of_slot_and_other_experts(ft):
    """Same expert, same rows: bitwise equal output whatever the slot or the other experts in the call."""
    H, I, E, k, T = 512, 256, 6, 4, 600
    cfg, L, S, n_slots, pool, slot_perm, comps, x, idx = _setup(ft, H, I, E, k, T, 11)
    # second copy of expert 2 in a spare slot
    spare = int(np.setdiff1d(np.arange(n_slots), slot_perm)[0])
    ft.pack_expert(comps[2], synth.W_BF16, L, pool[spare * S:(spare + 1) * S])
    counts, offsets, perm, inv = moe.permute(idx, E)
    all_on = slot_perm.astype(np.int32)
    only2 = np.full(E, -1, dtype=np.int32)
    only2[2] = spare
    Y1 = _run(ft, x, k, I, E, perm, offsets, all_on, pool, S, n_slots)
    Y2 = _run(ft, x, k, I, E, perm, offsets, only2, pool, S, n_slots)
    r = slice(int(offsets[2]), int(offsets[3]))
    assert np.array_equal(Y1[r], Y2[r])


def test_tc_empty_experts_and_all_rows_on_one_expert(ft):
    """Every assignment routed to experts 0..k-1 (the rest empty): k experts of T rows each."""
    H, I, E, k, T = 256, 128, 16, 8, 260
    cfg, L, S, n_slots, pool, slot_perm, comps, x, _ = _setup(ft, H, I, E, k, T, 13)
    idx = np.tile(np.arange(k, dtype=np.int32), (T, 1))
    counts, offsets, perm, inv = moe.permute(idx, E)
    assert (counts[k:] == 0).all()
    Y = _run(ft, x, k, I, E, perm, offsets, slot_perm.astype(np.int32), pool, S, n_slots)
    xs = formats.to_f64(x)
    ref = np.concatenate([moe.expert_ffn(xs[perm[offsets[e]:offsets[e + 1]] // k],
                                         *(formats.dequant(comps[e][m], synth.W_BF16) for m in ("gate", "up", "down")),
                                         act_round=formats.round_to_bf16) for e in range(k)])
    assert_close_layer(Y, ref, fro=1e-2)
    assert rel_fro(Y, ref) < 2e-3


def test_tc_split_k_is_deterministic(ft):
    """A one-token step whose K is split: repeated calls give bitwise equal outputs."""
    H, I, E, k, T = 4096, 512, 16, 4, 1
    cfg, L, S, n_slots, pool, slot_perm, comps, x, idx = _setup(ft, H, I, E, k, T, 14)
    counts, offsets, perm, inv = moe.permute(idx, E)
    so = slot_perm.astype(np.int32)
    Y = [_run(ft, x, k, I, E, perm, offsets, so, pool, S, n_slots) for _ in range(3)]
    assert np.array_equal(Y[0], Y[1]) and np.array_equal(Y[0], Y[2])


@pytest.mark.parametrize("wtype,H,I,E,k,T,seed", [
    (synth.W_NVFP4, 4096, 2048, 16, 6, 1, 20),    # the NVFP4 stack's shape, one decode token
    (synth.W_NVFP4, 1024, 512, 8, 2, 1, 21),      # NVFP4 with the gate/up K split
    (synth.W_NVFP4, 4096, 2048, 32, 6, 64, 22),   # NVFP4 decode batch of 64
    (synth.W_MXFP4, 6144, 2048, 16, 8, 1, 23),    # the MXFP4 layer's shape, one decode token
    (synth.W_MXFP4, 2048, 512, 32, 8, 16, 24),
    (synth.W_MXFP4, 256, 128, 8, 2, 3, 25),       # tiny: one 64-element scale pair per row
    (synth.W_NVFP4, 1024, 512, 16, 8, 300, 26),   # 2400 assignments: large-batch tiling with FP4 expansion
    (synth.W_MXFP4, 2048, 1024, 8, 4, 600, 27),
    (synth.W_NVFP4, 4096, 2048, 4, 2, 1100, 28),  # the NVFP4 stack's expert shape, ~550 rows per expert
])
def test_tc_fp4_expert_parity(ft, wtype, H, I, E, k, T, seed):
    """NVFP4 / MXFP4 weights expanded to bf16 in shared memory (exact), then the same tensor-core path
    (the expansion is asked for explicitly: small batches otherwise take the block-scaled FP4 MMA)."""
    cfg, L, S, n_slots, pool, slot_perm, comps, x, idx = _setup(ft, H, I, E, k, T, seed, wtype=wtype)
    counts, offsets, perm, inv = moe.permute(idx, E)
    slot_of = slot_perm.astype(np.int32).copy()
    slot_of[E - 1] = -1
    ft.ft_expert_set_fp4_path(ft.FT_FP4_EXPAND_BF16)
    try:
        Y = _run(ft, x, k, I, E, perm, offsets, slot_of, pool, S, n_slots, wtype)
    finally:
        ft.ft_expert_set_fp4_path(ft.FT_FP4_BLOCK_SCALED)
    xs = formats.to_f64(x)
    got, ref = [], []
    for e in range(E - 1):
        rows = np.arange(offsets[e], offsets[e + 1])
        if rows.size == 0:
            continue
        g, u, d = (formats.dequant(comps[e][m], wtype) for m in ("gate", "up", "down"))
        ref.append(moe.expert_ffn(xs[perm[rows] // k], g, u, d, act_round=formats.round_to_bf16))
        got.append(Y[rows])
    rows = np.arange(offsets[E - 1], offsets[E])
    assert np.isnan(Y[rows]).all()
    got, ref = np.concatenate(got), np.concatenate(ref)
    assert np.isfinite(got).all()
    assert_close_layer(got, ref, fro=1e-2)
    assert rel_fro(got, ref) < 2e-3


@pytest.mark.parametrize("T,k", [(300, 8), (20, 4)])
def test_tc_fp32_activations_are_rounded_to_bf16(ft, T, k):
    """fp32 x with bf16 weights: the rows are rounded to bf16 (RNE) on their way to the tensor cores."""
    H, I, E = 512, 256, 8
    cfg, L, S, n_slots, pool, slot_perm, comps, x, idx = _setup(ft, H, I, E, k, T, 31, xdt="f32")
    assert x.dtype == torch.float32
    counts, offsets, perm, inv = moe.permute(idx, E)
    Y = _run(ft, x, k, I, E, perm, offsets, slot_perm.astype(np.int32), pool, S, n_slots)
    xs = formats.round_to_bf16(formats.to_f64(x))
    ref = np.concatenate([moe.expert_ffn(xs[perm[offsets[e]:offsets[e + 1]] // k],
                                         *(formats.dequant(comps[e][m], synth.W_BF16) for m in ("gate", "up", "down")),
                                         act_round=formats.round_to_bf16) for e in range(E)])
    assert_close_layer(Y, ref, fro=1e-2)
    assert rel_fro(Y, ref) < 2e-3
