"""A whole decode step captured in one CUDA graph, replayed, and re-captured
after safe-point resizes ([Review] §2.6: the cache control runs on the device
with fixed-shape buffers and device-side counts, so the step can be put into
a CUDA graph; §2.7: a new cache configuration re-captures the execution
path).

The graph holds every layer of the step: router logits, routing,
permutation, every wave of the split cache step (hits evaluated while the
miss fill copies on a second stream, then the filled experts after the join)
and the combine.  After each replay the test compares every layer's output
with the fp64 oracle and the cache's residency tables and per-wave counts
with the LRU simulator; after each resize (which changes the wave count) it
captures a new graph and goes on.
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


@pytest.fixture(scope="module")
def ft(ftlib):
    assert torch.cuda.is_available()
    return ftlib


def test_captured_decode_step_with_resize_and_recapture(ft):
    cfg = synth.MoEConfig("graph", 256, 32, 4, 128, 3, synth.W_BF16, "bf16", seed=13, zipf_s=1.1)
    L, E, k, T = cfg.n_layers, cfg.n_experts, cfg.top_k, 8
    pool = ft.ExpertPool(cfg, L)
    pool.fill(DEV)
    S = pool.S
    max_slots = 16
    sp = torch.empty(max_slots * S, dtype=torch.uint8, device=DEV)
    cache = ft.Cache(L, E, L, 12, max_slots, S, pool.ptr, sp)
    box = {"sim": LRUSim(12, E)}
    lay = ft.MoELayer(cfg, T)
    routers = [synth.router_weights(cfg, l, DEV) for l in range(L)]
    src = [moe.ExpertSource(lambda e, l=l: synth.expert_weights(cfg, l, e, DEV), cfg.wtype) for l in range(L)]
    x_buf = torch.empty(T, cfg.hidden, dtype=torch.bfloat16, device=DEV)
    outs = torch.empty(L, T, cfg.hidden, dtype=torch.float32, device=DEV)
    counts = torch.zeros(L, 8, 4, dtype=torch.int32, device=DEV)     # per layer, per wave
    fs = torch.cuda.Stream(device=DEV)
    trace = synth.AR1Trace(cfg, T, DEV, tag=2)

    def decode_step(ratio):
        for l in range(L):
            lay.route(x_buf, *routers[l])
            for w in range(cache.n_waves()):
                lay.cached_wave(x_buf, l, cache, S, ratio, w, counts[l, w], fill_stream=fs)
            outs[l].copy_(lay.combine(T, lay.ext, None))

    def check(ratio):
        """Oracle outputs and simulator decisions for the step just run on x_buf."""
        sim = box["sim"]
        x64 = formats.to_f64(x_buf)
        got_out = outs.cpu().numpy()
        got_counts = counts.cpu().numpy()
        for l in range(L):
            wr, b = routers[l]
            z = moe.router_logits(x64, formats.to_f64(wr), formats.to_f64(b))
            assert not moe.near_ties(z, k).any()
            idx, w = moe.route(z, k)
            events, _ = sim.step(l, idx.reshape(-1), ratio)
            U = sorted(set(idx.reshape(-1).tolist()))
            nw = cache.n_waves()
            for wv in range(nw):
                wave = set(U[wv * sim.N:(wv + 1) * sim.N])
                ev = [e for e in events if e[1] in wave]
                want = [len(ev), sum(e[0] == "hit" for e in ev), sum(e[0] == "fill" for e in ev),
                        sum(e[0] == "ext" for e in ev)]
                assert got_counts[l, wv].tolist() == want, (l, wv)
            on_gpu = [e[1] for e in events if e[0] != "ext"]
            ref = moe.moe_layer(x64, idx, w, src[l], act_round=formats.round_to_bf16, only=on_gpu)
            assert_close_layer(got_out[l], ref, fro=1e-2)
        key, stamp, clock = cache.export()
        sk, ss = sim.state()
        assert key.tolist() == sk.tolist() and stamp.tolist() == ss.tolist() and clock == sim.clock

    schedule = [(12, 1.0, 4), (7, 0.7, 4), (12, 0.7, 3)]     # (slots, fill ratio, replays)
    sim = box["sim"]
    for phase, (N, ratio, reps) in enumerate(schedule):
        if phase:
            torch.cuda.synchronize()
            cache.resize(N)                                     # safe point: nothing in flight
            sim.resize(N)
            key, stamp, clock = cache.export()
            sk, ss = sim.state()
            assert key.tolist() == sk.tolist() and stamp.tolist() == ss.tolist()
        assert cache.n_waves() == -(-E // N)
        # one eager step (kernel attributes set outside capture), then the graph
        x_buf.copy_(trace.next())
        counts.zero_()
        decode_step(ratio)
        torch.cuda.synchronize()
        check(ratio)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            decode_step(ratio)
        for _ in range(reps):
            x_buf.copy_(trace.next())
            counts.zero_()
            g.replay()
            torch.cuda.synchronize()
            check(ratio)
        if phase < len(schedule) - 1:
            del g
    st = cache.stats()
    assert (st.hits, st.fills, st.externals) == (sim.hits, sim.fills, sim.externals)
    assert sim.externals > 0 and sim.fills > 0 and sim.hits > 0

    # a cold restart keeps the handle's tables in place: the last graph replays from an
    # empty cache, twice over the same inputs, with the same decisions as a fresh simulator
    xs = [trace.next() for _ in range(3)]
    for rnd in range(2):
        torch.cuda.synchronize()
        cache.reset()
        key, stamp, clock = cache.export()
        assert (key == -1).all() and (stamp == 0).all() and clock == 0
        s0 = cache.stats()
        assert (s0.steps, s0.hits, s0.fills, s0.externals, s0.bytes_h2d) == (0, 0, 0, 0, 0)
        box["sim"] = LRUSim(12, E)
        for xt in xs:
            x_buf.copy_(xt)
            counts.zero_()
            g.replay()
            torch.cuda.synchronize()
            check(0.7)
        if rnd == 0:
            first = cache.export()
        else:
            again = cache.export()
            assert all(np.array_equal(a, b) for a, b in zip(first[:2], again[:2])) and first[2] == again[2]
    del g
    assert ft.ft_get_device_error() == 0
    cache.destroy()
    pool.free()


def test_captured_step_with_the_host_branch_keeps_the_layer_output(ft):
    """The split with a real external share ([Review] §2.5, the exact merge; §2.6, the CPU
    branch in the captured step): 30% of each wave's misses are evaluated by the host
    expert executor from the pinned pool, as a host node of the graph, and their partial
    output is added by the combine.  Every layer's output must equal the oracle's full
    layer, whatever the split, and the cache must follow the simulator."""
    cfg = synth.MoEConfig("hostbranch", 256, 32, 4, 128, 2, synth.W_BF16, "bf16", seed=17, zipf_s=1.1)
    L, E, k, T = cfg.n_layers, cfg.n_experts, cfg.top_k, 8
    pool = ft.ExpertPool(cfg, L)
    pool.fill(DEV)
    S = pool.S
    cache = ft.Cache(L, E, L, 20, 20, S, pool.ptr, torch.empty(20 * S, dtype=torch.uint8, device=DEV))
    sim = LRUSim(20, E)
    lay = ft.MoELayer(cfg, T)
    cpu = ft.CpuExperts(threads=4)
    hb = ft.HostBranch(cfg, T, pool, cpu, DEV)
    routers = [synth.router_weights(cfg, l, DEV) for l in range(L)]
    src = [moe.ExpertSource(lambda e, l=l: synth.expert_weights(cfg, l, e, DEV), cfg.wtype) for l in range(L)]
    x_buf = torch.empty(T, cfg.hidden, dtype=torch.bfloat16, device=DEV)
    outs = torch.empty(L, T, cfg.hidden, dtype=torch.float32, device=DEV)
    counts = torch.zeros(L, 4, 4, dtype=torch.int32, device=DEV)
    fs = torch.cuda.Stream(device=DEV)
    trace = synth.AR1Trace(cfg, T, DEV, tag=6)
    ratio = 0.7

    def decode_step():
        for l in range(L):
            lay.route(x_buf, *routers[l])
            nw = cache.n_waves()
            for w in range(nw):
                after = (lambda l=l: hb.launch(lay, x_buf, l)) if w == nw - 1 else None
                lay.cached_wave(x_buf, l, cache, S, ratio, w, counts[l, w], fill_stream=fs, after_control=after)
            hb.join()
            ft.ft_combine(lay.y[: T * k], lay.inv, lay.idx[:T], lay.w[:T], lay.ext, hb.P[:T], E, outs[l])

    externals = 0

    def check():
        nonlocal externals
        x64 = formats.to_f64(x_buf)
        got = outs.cpu().numpy()
        for l in range(L):
            wr, b = routers[l]
            idx, w = moe.route(moe.router_logits(x64, formats.to_f64(wr), formats.to_f64(b)), k)
            events, _ = sim.step(l, idx.reshape(-1), ratio)
            externals += sum(e[0] == "ext" for e in events)
            ref = moe.moe_layer(x64, idx, w, src[l], act_round=formats.round_to_bf16)   # every expert
            assert_close_layer(got[l], ref, fro=1e-2)
        key, stamp, clock = cache.export()
        sk, ss = sim.state()
        assert key.tolist() == sk.tolist() and stamp.tolist() == ss.tolist()

    x_buf.copy_(trace.next())
    decode_step()                         # eager
    torch.cuda.synchronize()
    assert cpu.status() == 0
    check()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        decode_step()
    for _ in range(5):
        x_buf.copy_(trace.next())
        g.replay()
        torch.cuda.synchronize()
        assert cpu.status() == 0
        check()
    assert externals > 0
    del g
    assert ft.ft_get_device_error() == 0
    cache.destroy()
    cpu.destroy()
    pool.free()
