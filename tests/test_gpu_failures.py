"""Failure paths, driven from the host: refused pins and allocations, and a
stream handle whose creation fails half way.

Nothing here faults or hangs the GPU.  ft_debug_inject_failure makes one
chosen runtime call fail on the host (the call is never issued), and the tests
check the promised error status, that no handle is returned, that the
library holds no more device allocations, streams or events than before, and
that the cache's tables are exactly what they were (compared with the LRU
simulator), so that the next steps still match it.
"""
import numpy as np
import pytest
import torch

import synth
from oracle.lru import LRUSim

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def ft(ftlib):
    assert torch.cuda.is_available()
    yield ftlib
    for site in (1, 2, 3):
        ftlib.ft_debug_inject_failure(site, -1)


def test_impossible_pin_is_refused_without_fallback(ft):
    before = ft.ft_debug_live_resources()
    with pytest.raises(ft.FTError) as ei:
        ft.PinnedBuffer(1 << 60)
    assert ei.value.status == ft.FT_ENOMEM
    assert ft.ft_debug_live_resources() == before
    torch.cuda.synchronize()
    assert ft.ft_get_device_error() == 0


def test_injected_pin_failures(ft):
    ft.ft_debug_inject_failure(ft.FT_INJECT_HOST_PIN, 0)
    with pytest.raises(ft.FTError) as ei:
        ft.PinnedBuffer(1 << 20)
    assert ei.value.status == ft.FT_ENOMEM
    b = ft.PinnedBuffer(1 << 20)           # the site disarmed itself
    b.free()
    r = ft.RegisteredBuffer(1 << 20)
    ft.ft_debug_inject_failure(ft.FT_INJECT_HOST_PIN, 0)
    with pytest.raises(ft.FTError) as ei:
        r.pin()
    assert ei.value.status == ft.FT_ENOMEM and not r.pinned
    r.pin()
    assert r.pinned
    r.free()


def _cfg():
    return synth.MoEConfig("fail", 256, 16, 2, 128, 2, synth.W_BF16, "bf16", seed=9)


def test_cache_create_allocation_failures_leave_nothing(ft):
    cfg = _cfg()
    pool = ft.ExpertPool(cfg, 2)
    sp = torch.empty(40 * pool.S, dtype=torch.uint8, device=DEV)
    base = ft.ft_debug_live_resources()
    # every one of the eight table allocations, then each of the two events
    for after in range(8):
        ft.ft_debug_inject_failure(ft.FT_INJECT_DEVICE_ALLOC, after)
        with pytest.raises(ft.FTError) as ei:
            ft.Cache(2, 16, 2, 40, 40, pool.S, pool.ptr, sp)
        assert ei.value.status == ft.FT_ENOMEM
        assert ft.ft_debug_live_resources() == base
    for after in range(2):
        ft.ft_debug_inject_failure(ft.FT_INJECT_STREAM_EVENT, after)
        with pytest.raises(ft.FTError) as ei:
            ft.Cache(2, 16, 2, 40, 40, pool.S, pool.ptr, sp)
        assert ei.value.status == ft.FT_ECUDA
        assert ft.ft_debug_live_resources() == base
    c = ft.Cache(2, 16, 2, 40, 40, pool.S, pool.ptr, sp)
    assert ft.ft_debug_live_resources() == (base[0] + 8, base[1] + 2)
    c.destroy()
    assert ft.ft_debug_live_resources() == base
    pool.free()


def test_stream_create_failure_leaves_the_cache_as_it_was(ft):
    cfg = _cfg()
    E = cfg.n_experts
    pool = ft.ExpertPool(cfg, 2)
    pool.fill(DEV)
    N = 40
    sp = torch.empty(N * pool.S, dtype=torch.uint8, device=DEV)
    cache = ft.Cache(2, E, 2, N, N, pool.S, pool.ptr, sp)
    sim = LRUSim(N, E)
    lay = ft.MoELayer(cfg, 8)
    routers = [synth.router_weights(cfg, l, DEV) for l in range(2)]
    tr = synth.AR1Trace(cfg, 8, DEV, tag=3)

    def step(l, x):
        lay.route(x, *routers[l])
        idx = lay.idx[: x.shape[0]].cpu().numpy().reshape(-1)
        _, sim_slot_of = sim.step(l, idx, 1.0)
        for w in range(cache.n_waves()):
            cache.step(l, lay.counts, 1.0, w, lay.slot_of, lay.ext, lay.step_counts)
            assert lay.slot_of.cpu().numpy().tolist() == list(sim_slot_of[w])

    for s in range(6):
        x = tr.next()
        step(s % 2, x)
    torch.cuda.synchronize()
    key0, stamp0, clock0 = cache.export()
    sk, ss = sim.state()
    assert key0.tolist() == sk.tolist() and stamp0.tolist() == ss.tolist()
    res0 = ft.ft_debug_live_resources()
    # the stream and each of its four events
    for after in range(5):
        ft.ft_debug_inject_failure(ft.FT_INJECT_STREAM_EVENT, after)
        with pytest.raises(ft.FTError) as ei:
            ft.Stream(cache)
        assert ei.value.status == ft.FT_ECUDA
        assert ft.ft_debug_live_resources() == res0
        key, stamp, clock = cache.export()
        assert key.tolist() == key0.tolist() and stamp.tolist() == stamp0.tolist() and clock == clock0
    # the cache is usable and still agrees with the simulator
    for s in range(6):
        step(s % 2, tr.next())
    key, stamp, clock = cache.export()
    sk, ss = sim.state()
    assert key.tolist() == sk.tolist() and stamp.tolist() == ss.tolist() and clock == sim.clock
    # and a stream can still be created, used and destroyed
    st = ft.Stream(cache)
    slot_of = torch.empty(E, dtype=torch.int32, device=DEV)
    st.layer(0, 1, slot_of)
    st.layer_done(0)
    st.layer(1, -1, slot_of)
    st.layer_done(1)
    st.destroy()
    sim.stream_begin()
    sim.stream_end([(0, 0), (1, 1)])
    key, stamp, clock = cache.export()
    sk, ss = sim.state()
    assert key.tolist() == sk.tolist() and stamp.tolist() == ss.tolist()
    assert ft.ft_debug_live_resources() == res0
    cache.destroy()
    pool.free()
    assert ft.ft_get_device_error() == 0


def test_read_then_pin_pool_serves_the_same_layer(ft, tmp_path):
    """A pool saved to a file and loaded both ways holds the same bytes, and a
    cached layer step over the read-then-pinned pool gives the same output as
    over the pool that was pinned first."""
    cfg = _cfg()
    E = cfg.n_experts
    pool = ft.ExpertPool(cfg, 2)
    pool.fill(DEV)
    path = str(tmp_path / "pool.bin")
    pool.save(path)
    a = ft.ExpertPool.load(cfg, 2, path, read_then_pin=True, threads=4)
    b = ft.ExpertPool.load(cfg, 2, path, read_then_pin=False, threads=3)
    assert set(a.setup_s) == {"alloc_pageable", "read", "pin"} and set(b.setup_s) == {"alloc_pinned", "read"}
    assert torch.equal(a.host, pool.host) and torch.equal(b.host, pool.host)
    outs = []
    x = synth.activations(cfg, 8, tag=4, device=DEV)
    wr, bias = synth.router_weights(cfg, 1, DEV)
    for p in (pool, a):
        sp = torch.empty(20 * p.S, dtype=torch.uint8, device=DEV)
        c = ft.Cache(2, E, 2, 20, 20, p.S, p.ptr, sp)
        lay = ft.MoELayer(cfg, 8)
        outs.append(lay.forward_cached(x, wr, bias, 1, c, p.S).clone())
        torch.cuda.synchronize()
        c.destroy()
    assert torch.equal(outs[0], outs[1])
    for p in (pool, a, b):
        p.free()
    assert ft.ft_get_device_error() == 0
