"""The allocation-free grouped-expert entry point agrees with the workspace one.

ft_expert_grouped_noalloc serves callers that cannot call cudaMalloc (a host
application that owns all device memory through its own allocator, or a
latency-critical path that cannot afford cudaMalloc's implicit device
synchronisation).  Its intermediate lives in a fixed 4 MiB array inside the
library instead of a caller workspace, and it always runs the CUDA-core
kernels (fp32 intermediate).  These tests call it through the C ABI twice in a
row and compare each result with the fp64 oracle and with ft_expert_grouped's
on the same inputs, within the tolerances the other parity tests use, and
check the size limit on both sides of it.  This file is named so that pytest
collects it after every other test file.
"""
import numpy as np
import pytest
import torch

import synth
from conftest import assert_close_layer
from oracle import formats, moe

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _setup(ft, wtype, H, I, E, seed):
    cfg = synth.MoEConfig(f"noalloc{wtype}_{H}_{I}", H, E, 8, I, 1, wtype, "bf16", seed=seed)
    L = ft.ft_expert_layout_get(wtype, H, I)
    S = int(L.bytes)
    n_slots = E + 2
    pool = torch.zeros(n_slots * S, dtype=torch.uint8, device=DEV)
    for e in range(E):
        ft.pack_expert(synth.expert_weights(cfg, 0, e, DEV), wtype, L, pool[(e + 1) * S:(e + 2) * S])
    return cfg, pool, S, n_slots


def _oracle_rows(cfg, x, perm, offsets, k, experts):
    """The oracle's Y rows (permuted order) for the given experts; others stay NaN."""
    xs = formats.to_f64(x)
    Y = np.full((perm.size, cfg.hidden), np.nan)
    for e in experts:
        rows = np.arange(offsets[e], offsets[e + 1])
        if rows.size == 0:
            continue
        c = synth.expert_weights(cfg, 0, e, DEV)
        g, u, d = (formats.dequant(c[m], cfg.wtype) for m in ("gate", "up", "down"))
        Y[rows] = moe.expert_ffn(xs[perm[rows] // k], g, u, d)
    return Y


def _one_call(ft, cfg, pool, S, n_slots, T, k, tag):
    E, H, I = cfg.n_experts, cfg.hidden, cfg.inter
    rng = np.random.default_rng(tag)
    idx = np.array([rng.permutation(E)[:k] for _ in range(T)], dtype=np.int32).reshape(T, k)
    _, offsets, perm, _ = moe.permute(idx, E)
    slot_of = (np.arange(E) + 1).astype(np.int32)
    slot_of[0] = -1                                   # one expert not evaluated: its rows stay untouched
    x = synth.activations(cfg, T, tag=tag, device=DEV)
    d_perm, d_off = torch.from_numpy(perm).to(DEV), torch.from_numpy(offsets).to(DEV)
    d_slot = torch.from_numpy(slot_of).to(DEV)
    y_ref = torch.full((T * k, H), float("nan"), device=DEV)
    ws = torch.empty(ft.ft_expert_grouped_workspace(T, k, H, I), dtype=torch.uint8, device=DEV)
    # the workspace entry point with the FP4 weights expanded exactly (bf16 products), not the
    # block-scaled FP4 MMA, whose quantised activations sit outside this comparison's tolerance
    ft.ft_expert_set_fp4_path(ft.FT_FP4_EXPAND_BF16)
    try:
        ft.ft_expert_grouped(x, k, I, E, cfg.wtype, d_perm, d_off, d_slot, pool, S, n_slots, y_ref, ws)
    finally:
        ft.ft_expert_set_fp4_path(ft.FT_FP4_BLOCK_SCALED)
    y_na = torch.full((T * k, H), float("nan"), device=DEV)
    ft.ft_expert_grouped_noalloc(x, k, I, E, cfg.wtype, d_perm, d_off, d_slot, pool, S, n_slots, y_na)
    torch.cuda.synchronize()
    assert ft.ft_get_device_error() == 0
    a, b = y_na.cpu().numpy(), y_ref.cpu().numpy()
    skipped = np.arange(offsets[0], offsets[1])
    assert np.isnan(a[skipped]).all()
    keep = np.setdiff1d(np.arange(T * k), skipped)
    # against the oracle (fp32 intermediate on this path: the plain bar, and far inside it)
    ref = _oracle_rows(cfg, x, perm, offsets, k, range(1, E))
    assert_close_layer(a[keep], ref[keep])
    assert np.linalg.norm(a[keep] - ref[keep]) / np.linalg.norm(ref[keep]) < 2e-5
    # against the workspace entry point (tensor cores for bf16 / FP4: bf16 intermediate)
    assert_close_layer(a[keep], b[keep], fro=1e-2)


def test_noalloc_matches_workspace_entry_point_twice(ftlib):
    ft = ftlib
    cfg, pool, S, n_slots = _setup(ft, ft.FT_W_BF16, 2048, 512, 32, seed=21)
    # two calls in a row sharing the library's array: a large batch, then a small one
    _one_call(ft, cfg, pool, S, n_slots, T=64, k=8, tag=1)
    _one_call(ft, cfg, pool, S, n_slots, T=5, k=8, tag=2)


def test_noalloc_matches_for_a_block_scaled_format(ftlib):
    ft = ftlib
    cfg, pool, S, n_slots = _setup(ft, ft.FT_W_MXFP4, 1024, 512, 16, seed=22)
    _one_call(ft, cfg, pool, S, n_slots, T=33, k=8, tag=3)
    _one_call(ft, cfg, pool, S, n_slots, T=33, k=8, tag=4)


def test_noalloc_accepts_a_call_exactly_at_the_limit(ftlib):
    ft = ftlib
    k, I = 8, 2048
    T = ft.FT_NOALLOC_MAX_ELEMS // (k * I)             # T*k*I == FT_NOALLOC_MAX_ELEMS (T = 64)
    assert T * k * I == ft.FT_NOALLOC_MAX_ELEMS
    cfg, pool, S, n_slots = _setup(ft, ft.FT_W_BF16, 512, I, 16, seed=23)
    _one_call(ft, cfg, pool, S, n_slots, T=T, k=k, tag=5)


def test_noalloc_refuses_sizes_beyond_its_array(ftlib):
    ft = ftlib
    H, I, k = 2048, 2048, 8
    T = ft.FT_NOALLOC_MAX_ELEMS // (k * I) + 1          # T*k*I just over the limit
    x = torch.zeros(T, H, dtype=torch.bfloat16, device=DEV)
    z32 = torch.zeros(T * k, dtype=torch.int32, device=DEV)
    L = ft.ft_expert_layout_get(ft.FT_W_BF16, H, I)
    with pytest.raises(ft.FTError) as ei:
        ft.ft_expert_grouped_noalloc(x, k, I, 4, ft.FT_W_BF16, z32, z32, z32, x, int(L.bytes), 1,
                                     torch.zeros(1, device=DEV))
    assert ei.value.status == ft.FT_EINVAL
