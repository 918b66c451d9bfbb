"""Parity of the CUDA-core grouped expert kernels against the fp64 oracle.

ft_expert_grouped sends bf16 weights above one decode token, NVFP4 and MXFP4
weights to the tensor cores, so the CUDA-core kernels (gate/up and down,
weights dequantised in registers, fp32 intermediate) run there for fp32 and
FP8 weights and for one token of bf16 weights (a form that keeps more weight
loads in flight, one row per expert at a time).  The
no-allocation entry point ft_expert_grouped_noalloc runs the CUDA-core kernels
for every format; these tests call it through the C ABI for all five formats
and compare each evaluated row with the oracle's SwiGLU on the same stored
weights (x is not rounded, nor is the intermediate, on this path), at sizes
that span several 8-row chunks with ragged tails, with skipped experts (rows
left untouched) and fp32 or bf16 activations.
"""
import numpy as np
import pytest
import torch

import synth
from conftest import assert_close_layer, rel_fro
from oracle import formats, moe

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def ft(ftlib):
    assert torch.cuda.is_available()
    return ftlib


CASES = [
    # wtype, H, I, E, k, T, x dtype
    (synth.W_F32, 256, 128, 8, 2, 29, "f32"),
    (synth.W_BF16, 512, 256, 12, 4, 37, "bf16"),
    (synth.W_BF16, 2048, 512, 32, 8, 64, "bf16"),       # the decode layer shape, 512 assignments
    (synth.W_BF16, 384, 128, 6, 2, 1, "f32"),           # one token, fp32 activations
    (synth.W_FP8, 512, 384, 10, 3, 41, "bf16"),
    (synth.W_FP8, 256, 128, 4, 4, 5, "f32"),
    (synth.W_NVFP4, 1024, 512, 16, 6, 23, "bf16"),
    (synth.W_NVFP4, 4096, 256, 8, 6, 3, "bf16"),        # wide hidden
    (synth.W_MXFP4, 1024, 512, 16, 8, 33, "bf16"),
    (synth.W_MXFP4, 768, 256, 6, 2, 17, "f32"),
    # one token: the one-row form of the kernels
    (synth.W_BF16, 2048, 512, 32, 8, 1, "bf16"),        # the decode layer shape
    (synth.W_FP8, 512, 384, 10, 3, 1, "bf16"),
    (synth.W_NVFP4, 1024, 512, 16, 6, 1, "bf16"),
    (synth.W_MXFP4, 1024, 512, 16, 8, 1, "f32"),
]


@pytest.mark.parametrize("wtype,H,I,E,k,T,xdt", CASES)
def test_cuda_core_kernels_match_oracle(ft, wtype, H, I, E, k, T, xdt):
    cfg = synth.MoEConfig(f"cc{wtype}_{H}_{I}", H, E, k, I, 1, wtype, xdt, seed=40 + wtype)
    L = ft.ft_expert_layout_get(wtype, H, I)
    S = int(L.bytes)
    n_slots = E + 3
    pool = torch.zeros(n_slots * S, dtype=torch.uint8, device=DEV)
    rng = np.random.default_rng(H + I + wtype + T)
    slot_perm = rng.permutation(n_slots)[:E]
    comps = {}
    for e in range(E):
        comps[e] = synth.expert_weights(cfg, 0, e, DEV)
        ft.pack_expert(comps[e], wtype, L, pool[slot_perm[e] * S:(slot_perm[e] + 1) * S])
    x = synth.activations(cfg, T, tag=9, device=DEV)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    counts, offsets, perm, inv = moe.permute(idx, E)
    slot_of = slot_perm.astype(np.int32).copy()
    skipped = {E - 1}
    slot_of[E - 1] = -1
    if E > 4:
        slot_of[2] = -2
        skipped.add(2)
    y = torch.full((T * k, H), float("nan"), dtype=torch.float32, device=DEV)
    ft.ft_expert_grouped_noalloc(x, k, I, E, wtype, torch.from_numpy(perm).to(DEV),
                                 torch.from_numpy(offsets).to(DEV), torch.from_numpy(slot_of).to(DEV), pool, S,
                                 n_slots, y)
    torch.cuda.synchronize()
    assert ft.ft_get_device_error() == 0
    Y = y.cpu().numpy()
    xs = formats.to_f64(x)
    got, ref = [], []
    for e in range(E):
        rows = np.arange(offsets[e], offsets[e + 1])
        if e in skipped:
            assert np.isnan(Y[rows]).all(), "rows of skipped experts must be left untouched"
            continue
        g, u, d = (formats.dequant(comps[e][m], wtype) for m in ("gate", "up", "down"))
        ref.append(moe.expert_ffn(xs[perm[rows] // k], g, u, d))
        got.append(Y[rows])
    got, ref = np.concatenate(got), np.concatenate(ref)
    assert_close_layer(got, ref)
    # fp32 products of exact inputs: far inside the bar
    assert rel_fro(got, ref) < 2e-5


def test_one_token_with_a_repeated_expert(ft):
    """One token whose routing names an expert three times (the one-row form then takes that
    expert's rows one at a time): every row matches the oracle, through both entry points
    (ft_expert_grouped takes the CUDA-core kernels for one bf16 token too)."""
    wtype, H, I, E, k, T = synth.W_BF16, 512, 256, 8, 4, 1
    cfg = synth.MoEConfig("cc_repeat", H, E, k, I, 1, wtype, "bf16", seed=77)
    L = ft.ft_expert_layout_get(wtype, H, I)
    S = int(L.bytes)
    pool = torch.zeros(E * S, dtype=torch.uint8, device=DEV)
    comps = {e: synth.expert_weights(cfg, 0, e, DEV) for e in range(E)}
    for e in range(E):
        ft.pack_expert(comps[e], wtype, L, pool[e * S:(e + 1) * S])
    x = synth.activations(cfg, T, tag=3, device=DEV)
    idx = np.array([[3, 5, 3, 3]], dtype=np.int32)
    counts, offsets, perm, inv = moe.permute(idx, E)
    args = (torch.from_numpy(perm).to(DEV), torch.from_numpy(offsets).to(DEV),
            torch.arange(E, dtype=torch.int32, device=DEV), pool, S, E)
    y1 = torch.full((T * k, H), float("nan"), dtype=torch.float32, device=DEV)
    ft.ft_expert_grouped_noalloc(x, k, I, E, wtype, *args, y1)
    y2 = torch.full((T * k, H), float("nan"), dtype=torch.float32, device=DEV)
    ws = torch.empty(ft.ft_expert_grouped_workspace(T, k, H, I), dtype=torch.uint8, device=DEV)
    ft.ft_expert_grouped(x, k, I, E, wtype, *args, y2, ws)
    torch.cuda.synchronize()
    assert ft.ft_get_device_error() == 0
    xs = formats.to_f64(x)
    ref = np.concatenate([moe.expert_ffn(xs[perm[offsets[e]:offsets[e + 1]] // k],
                                         *(formats.dequant(comps[e][m], wtype) for m in ("gate", "up", "down")))
                          for e in range(E) if counts[e]])
    for y in (y1, y2):
        got = y.cpu().numpy()
        assert_close_layer(got, ref)
        assert rel_fro(got, ref) < 2e-5
    assert torch.equal(y1, y2)
