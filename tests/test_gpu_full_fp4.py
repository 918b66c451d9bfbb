"""Full-size parity of the FP4 workloads: the 43-layer NVFP4 stack and the MXFP4 mixed trace.

Shapes are the workloads' own (NVFP4: H=4096, E=256, top-6, I=2048; MXFP4:
H=6144, E=256, top-8, I=2048).  Routing, the cache's decisions (against the
LRU simulator) and the miss split are compared exactly on every step; layer
outputs are compared with the fp64 oracle on sampled steps and tokens (the
oracle dequantises the same stored bytes).  Decode batches run both FP4
paths: the block-scaled FP4 MMA, which quantises the token rows and the
intermediate to the weights' format (the oracle applies the same rule), and
the exact expansion to bf16, which rounds the intermediate to bf16 (so does
the oracle); bar: relative Frobenius 1e-2.  Prefill chunks take the same path.
The host pool holds a window of physical layers (logical l reads l mod the
window), which changes neither keys nor outputs.
"""
import numpy as np
import pytest
import torch

import synth
from conftest import assert_close_layer
from oracle import formats, moe
from oracle.lru import LRUSim

pytestmark = pytest.mark.gpu
DEV = "cuda"
TC_ROUND = formats.round_to_bf16


@pytest.fixture(scope="module")
def ft(ftlib):
    assert torch.cuda.is_available()
    return ftlib


@pytest.fixture(params=["block_scaled", "expand"])
def fp4_path(request, ft):
    ft.ft_expert_set_fp4_path(ft.FT_FP4_BLOCK_SCALED if request.param == "block_scaled" else ft.FT_FP4_EXPAND_BF16)
    yield request.param
    ft.ft_expert_set_fp4_path(ft.FT_FP4_BLOCK_SCALED)


def decode_rounding(wtype, path):
    """(x_round, act_round) of a decode batch on the given FP4 path."""
    if path == "expand":
        return None, TC_ROUND
    q = formats.quant_act_nvfp4 if wtype == synth.W_NVFP4 else formats.quant_act_mxfp4
    return q, q


class Experts:
    """fp64 experts of a config, decoded on use per (physical layer, expert); a few kept (they are large)."""

    def __init__(self, cfg, n_phys, keep=16):
        self.cfg, self.n_phys, self.keep, self.cache = cfg, n_phys, keep, {}

    def __call__(self, layer):
        p = layer % self.n_phys

        def get(e):
            if (p, e) not in self.cache:
                if len(self.cache) >= self.keep:
                    self.cache.pop(next(iter(self.cache)))
                c = synth.expert_weights(self.cfg, p, e, DEV)
                self.cache[(p, e)] = tuple(formats.dequant(c[m], self.cfg.wtype) for m in ("gate", "up", "down"))
            return self.cache[(p, e)]
        return get


def _waves(ft, L, cache, layer, x, ratio, sim, S, pool_slots, fill_stream=None):
    """All waves of a layer step; with ``fill_stream`` in the split form (hits beside the fill)."""
    idx = L.idx[: x.shape[0]].cpu().numpy()
    ev, sim_slot_of = sim.step(layer, idx.reshape(-1), ratio)
    counts = np.zeros(4, dtype=np.int64)
    for w in range(cache.n_waves()):
        exp = sim_slot_of[w] if w < len(sim_slot_of) else [-1] * cache.E
        if fill_stream is None:
            cache.step(layer, L.counts, ratio, w, L.slot_of, L.ext, L.step_counts)
            assert L.slot_of.cpu().numpy().tolist() == list(exp), f"layer {layer} wave {w}"
            L.experts(x, L.slot_of, cache.slot_pool, S, pool_slots)
        else:
            cache.step_split(layer, L.counts, ratio, w, L.slot_of, L.slot_fill, L.ext, L.step_counts,
                             fill_stream=fill_stream)
            L.experts(x, L.slot_of, cache.slot_pool, S, pool_slots)
            cache.fill_join()
            L.experts(x, L.slot_fill, cache.slot_pool, S, pool_slots)
            got = torch.where(L.slot_fill >= 0, L.slot_fill, L.slot_of)
            assert got.cpu().numpy().tolist() == list(exp), f"layer {layer} wave {w}"
        counts += L.step_counts.cpu().numpy()
    return counts


def test_nvfp4_stack_decode_and_prefill(ft, fp4_path):
    cfg = synth.NVFP4_43L
    xr, ar = decode_rounding(cfg.wtype, fp4_path)
    n_phys, n_slots = 2, 600
    pool = ft.ExpertPool(cfg, n_phys)
    pool.fill(DEV)
    sp = torch.empty(n_slots * pool.S, dtype=torch.uint8, device=DEV)
    cache = ft.Cache(cfg.n_layers, cfg.n_experts, n_phys, n_slots, n_slots, pool.S, pool.ptr, sp)
    sim = LRUSim(n_slots, cfg.n_experts)
    experts = Experts(cfg, n_phys)
    layers = [0, 1, 2, 21, 42]                      # logical layers; physical l % 2
    routers = {l: synth.router_weights(cfg, l, DEV) for l in layers}
    T = 16
    lay = ft.MoELayer(cfg, T)
    tr = synth.AR1Trace(cfg, T, DEV)
    sample = [0, 7, 15]
    fs = torch.cuda.Stream()
    for step in range(4):
        x = tr.next()
        for l in layers:
            lay.route(x, *routers[l])
            z = lay.logits[:T].cpu().numpy().astype(np.float64)
            ri, rw = moe.route(z, cfg.top_k)
            assert np.array_equal(lay.idx[:T].cpu().numpy(), ri)
            # odd steps in the split form (the decode form used for FP4 weights)
            _waves(ft, lay, cache, l, x, 1.0, sim, pool.S, n_slots, fill_stream=fs if step % 2 else None)
            out = lay.combine(T, lay.ext, None).cpu().numpy()
            if (step, l) in ((0, 0), (3, 21), (3, 42)):
                xs = formats.to_f64(x[sample])
                ref = moe.moe_layer(xs, ri[sample], rw[sample], experts(l), act_round=ar, x_round=xr)
                assert_close_layer(out[sample], ref, fro=1e-2)
    st = cache.stats()
    assert (st.hits, st.fills) == (sim.hits, sim.fills)
    key, stamp, clock = cache.export()
    sk, ss = sim.state()
    assert key.tolist() == sk.tolist() and stamp.tolist() == ss.tolist() and clock == sim.clock

    # one 8192-token prefill chunk of physical layer 1 with every expert resident (large-batch tiling)
    fused = pool.host[1 * cfg.n_experts * pool.S:2 * cfg.n_experts * pool.S].to(DEV)
    lp = ft.MoELayer(cfg, 8192)
    wr, _ = synth.router_weights(cfg, 1, DEV)
    zero = torch.zeros(cfg.n_experts, dtype=torch.float32, device=DEV)
    xp = synth.activations(cfg, 8192, tag=4, device=DEV)
    so = torch.arange(cfg.n_experts, dtype=torch.int32, device=DEV)
    out = lp.forward_slots(xp, wr, zero, so, fused, pool.S, cfg.n_experts).cpu().numpy()
    z = lp.logits.cpu().numpy().astype(np.float64)
    ri, rw = moe.route(z, cfg.top_k)
    assert np.array_equal(lp.idx.cpu().numpy(), ri)
    rows = [5, 4000, 8191]
    ref = moe.moe_layer(formats.to_f64(xp[rows]), ri[rows], rw[rows], experts(1), act_round=ar, x_round=xr)
    assert_close_layer(out[rows], ref, fro=1e-2)
    assert ft.ft_get_device_error() == 0
    cache.destroy()
    pool.free()


def test_mxfp4_mixed_resizes_and_split(ft, fp4_path):
    """Decode steps with the 0.7 miss split and safe-point resizes 592 -> 410 -> 205 -> 592 slots
    (from step 3 in the split cache-step form).

    The external experts' partial output is supplied by the oracle (fp64 ->
    fp32): the layer output must match the oracle's full layer, whatever the
    cache size or split; between resizes every cache decision matches the
    simulator."""
    cfg = synth.MXFP4_MIXED
    xr, ar = decode_rounding(cfg.wtype, fp4_path)
    L_, E = cfg.n_layers, cfg.n_experts
    pool = ft.ExpertPool(cfg, L_)
    pool.fill(DEV)
    max_slots = 592
    sp = torch.empty(max_slots * pool.S, dtype=torch.uint8, device=DEV)
    cache = ft.Cache(L_, E, L_, max_slots, max_slots, pool.S, pool.ptr, sp)
    sim = LRUSim(max_slots, E)
    experts = Experts(cfg, L_)
    routers = [synth.router_weights(cfg, l, DEV) for l in range(L_)]
    lay = ft.MoELayer(cfg, 1)
    tr = synth.AR1Trace(cfg, 1, DEV, tag=3)
    schedule = {6: 410, 12: 205, 18: 592}
    n_ext = 0
    fs = torch.cuda.Stream()
    for step in range(22):
        if step in schedule:
            cache.resize(schedule[step])
            sim.resize(schedule[step])
        x = tr.next()
        for l in range(L_):
            lay.route(x, *routers[l])
            z = lay.logits[:1].cpu().numpy().astype(np.float64)
            ri, rw = moe.route(z, cfg.top_k)
            assert np.array_equal(lay.idx[:1].cpu().numpy(), ri)
            _waves(ft, lay, cache, l, x, 0.7, sim, pool.S, max_slots, fill_stream=fs if step >= 3 else None)
            ext = lay.ext.cpu().numpy()
            C = [e for e in range(E) if ext[e]]
            n_ext += len(C)
            check = (step in (0, 10, 21) and l in (0, 3)) or (C and n_ext <= 2)
            P = None
            if C and check:
                P = torch.from_numpy(moe.moe_layer(formats.to_f64(x), ri, rw, experts(l), only=C)
                                     .astype(np.float32)).to(DEV)
            elif C:
                P = torch.zeros(1, cfg.hidden, dtype=torch.float32, device=DEV)
            out = lay.combine(1, lay.ext, P).cpu().numpy()
            if check:
                # the GPU's experts with the path's rounding, plus the external part as supplied
                on_gpu = [e for e in set(ri.reshape(-1).tolist()) if e not in C]
                ref = moe.moe_layer(formats.to_f64(x), ri, rw, experts(l), act_round=ar, x_round=xr, only=on_gpu)
                if C:
                    ref = ref + P.cpu().numpy().astype(np.float64)
                assert_close_layer(out, ref, fro=1e-2)
    st = cache.stats()
    assert (st.hits, st.fills, st.externals) == (sim.hits, sim.fills, sim.externals)
    assert st.externals > 0 and cache.n_waves() == 1
    key, stamp, clock = cache.export()
    sk, ss = sim.state()
    assert key.tolist() == sk.tolist() and stamp.tolist() == ss.tolist() and clock == sim.clock
    assert ft.ft_get_device_error() == 0
    cache.destroy()
    pool.free()
