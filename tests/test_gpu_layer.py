"""Layer-level parity: routing, cache decisions, streaming and layer outputs against the oracle and the LRU simulator."""
import numpy as np
import pytest
import torch

import synth
from conftest import assert_close_layer, bf16_act_round
from oracle import formats, moe
from oracle.lru import LRUSim

pytestmark = pytest.mark.gpu
DEV = "cuda"
# bf16 expert weights run on the tensor cores, which round the intermediate
# silu(G)*U to bf16: the oracle applies the same rounding, and the bar is 1e-2
TC_ROUND = formats.round_to_bf16


@pytest.fixture(scope="module")
def ft(ftlib):
    assert torch.cuda.is_available()
    return ftlib


def make_cache(ft, cfg, n_phys, N, max_slots):
    pool = ft.ExpertPool(cfg, n_phys)
    pool.fill(DEV)
    sp = torch.empty(max_slots * pool.S, dtype=torch.uint8, device=DEV)
    cache = ft.Cache(cfg.n_layers, cfg.n_experts, n_phys, N, max_slots, pool.S, pool.ptr, sp)
    return pool, sp, cache


class OracleLayer:
    """fp64 experts of a config, decoded once per (physical layer, expert)."""

    def __init__(self, cfg, n_phys):
        self.cfg, self.n_phys, self.src = cfg, n_phys, {}

    def experts(self, layer):
        p = layer % self.n_phys
        if p not in self.src:
            self.src[p] = moe.ExpertSource(lambda e, p=p: synth.expert_weights(self.cfg, p, e, DEV), self.cfg.wtype)
        return self.src[p]


def run_waves(ft, layer_obj, cache, layer, x, ratio, sim=None, events=None, fill_stream=None):
    """All waves of one cached layer step, checking slot_of against the simulator after each wave.

    With ``fill_stream`` each wave runs in the split form (hits evaluated while
    the fill copies on that stream); the simulator then checks the hit and fill
    slots merged."""
    idx = layer_obj.idx[: x.shape[0]].cpu().numpy()
    if sim is not None:
        ev, sim_slot_of = sim.step(layer, idx.reshape(-1), ratio)
        if events is not None:
            events.extend(ev)
    for w in range(cache.n_waves()):
        if fill_stream is None:
            cache.step(layer, layer_obj.counts, ratio, w, layer_obj.slot_of, layer_obj.ext, layer_obj.step_counts)
            got = layer_obj.slot_of
        else:
            cache.step_split(layer, layer_obj.counts, ratio, w, layer_obj.slot_of, layer_obj.slot_fill,
                             layer_obj.ext, layer_obj.step_counts, fill_stream=fill_stream)
            hit, fil = layer_obj.slot_of, layer_obj.slot_fill
            assert not bool(((hit >= 0) & (fil >= 0)).any()), "an expert is both a hit and a fill"
            got = torch.where(fil >= 0, fil, hit)
        if sim is not None:
            exp = sim_slot_of[w] if w < len(sim_slot_of) else [-1] * cache.E
            assert got.cpu().numpy().tolist() == list(exp), f"layer {layer} wave {w}"
        layer_obj.experts(x, layer_obj.slot_of, cache.slot_pool, layer_obj_S(cache), cache.max_slots)
        if fill_stream is not None:
            cache.fill_join()
            layer_obj.experts(x, layer_obj.slot_fill, cache.slot_pool, layer_obj_S(cache), cache.max_slots)


def layer_obj_S(cache):
    return cache.slot_pool.numel() // cache.max_slots


# ---------------------------------------------------------------- the tiny fp32 layer

def test_tiny_fp32_layer_one_step_and_sequential(ft):
    cfg = synth.TINY_F32
    pool, sp, cache = make_cache(ft, cfg, 1, 6, 6)
    L = ft.MoELayer(cfg, 64)
    wr, b = synth.router_weights(cfg, 0, DEV)
    x = synth.activations(cfg, 64, device=DEV)
    ol = OracleLayer(cfg, 1)
    x64, wr64 = formats.to_f64(x), formats.to_f64(wr)
    sim = LRUSim(6, 16)

    # (i) one step of 64 tokens: about 16 unique experts over 6 slots -> 3 waves
    L.route(x, wr, b)
    z = L.logits[:64].cpu().numpy()
    idx = L.idx[:64].cpu().numpy()
    ri, rw = moe.route(z.astype(np.float64), 2)
    assert np.array_equal(idx, ri)
    assert cache.n_waves() == 3
    run_waves(ft, L, cache, 0, x, 1.0, sim)
    out = L.combine(64, L.ext, None).cpu().numpy()
    z_ref = moe.router_logits(x64, wr64)
    assert np.abs(z - z_ref).max() < 1e-5
    ri2, rw2 = moe.route(z_ref, 2)
    tie = moe.near_ties(z_ref, 2)
    assert not tie.any()
    assert np.array_equal(idx, ri2)
    ref = moe.moe_layer(x64, ri2, rw2, ol.experts(0))
    assert_close_layer(out, ref)

    # (ii) 64 sequential single-token steps over the same cache
    for t in range(64):
        xt = x[t:t + 1]
        L.route(xt, wr, b)
        run_waves(ft, L, cache, 0, xt, 1.0, sim)
        o = L.combine(1, L.ext, None).cpu().numpy()
        assert_close_layer(o, ref[t:t + 1])
    key, stamp, clock = cache.export()
    sk, ss = sim.state()
    assert key.tolist() == sk.tolist() and stamp.tolist() == ss.tolist() and clock == sim.clock
    st = cache.stats()
    assert (st.hits, st.fills, st.externals) == (sim.hits, sim.fills, sim.externals)
    assert ft.ft_get_device_error() == 0


# ---------------------------------------------------------------- a cache trace with resizes and splits

def test_cache_trace_resize_split_matches_simulator(ft):
    cfg = synth.MoEConfig("trace", 256, 64, 4, 256, 4, synth.W_BF16, "bf16", seed=5, zipf_s=1.1)
    pool, sp, cache = make_cache(ft, cfg, 4, 40, 60)
    big_pool_sp = torch.empty(256 * pool.S, dtype=torch.uint8, device=DEV)
    big = ft.Cache(cfg.n_layers, cfg.n_experts, 4, 256, 256, pool.S, pool.ptr, big_pool_sp)
    L = ft.MoELayer(cfg, 16)
    Lb = ft.MoELayer(cfg, 16)
    sim = LRUSim(40, 64)
    ol = OracleLayer(cfg, 4)
    routers = [synth.router_weights(cfg, l, DEV) for l in range(4)]
    traces = {T: synth.AR1Trace(cfg, T, DEV, tag=T) for T in (1, 4, 16)}
    for step in range(45):
        T = (1, 4, 16)[step % 3]
        x = traces[T].next()
        ratio = 1.0 if step < 15 else 0.6
        if step == 25:
            cache.resize(25)
            sim.resize(25)
        if step == 35:
            cache.resize(55)
            sim.resize(55)
        for l in range(4):
            wr, b = routers[l]
            L.route(x, wr, b)
            run_waves(ft, L, cache, l, x, ratio, sim)
            # the external experts' partial output, as the host branch would supply it (fp64 -> fp32)
            idx = L.idx[:T].cpu().numpy()
            z = L.logits[:T].cpu().numpy().astype(np.float64)
            ri, rw = moe.route(z, cfg.top_k)
            assert np.array_equal(idx, ri)
            ext = L.ext.cpu().numpy()
            C = [e for e in range(64) if ext[e]]
            P = None
            if C:
                P = torch.from_numpy(moe.moe_layer(formats.to_f64(x), ri, rw, ol.experts(l), only=C)
                                     .astype(np.float32)).to(DEV)
            out = L.combine(T, L.ext, P).cpu().numpy()
            # the same step with every expert resident: bitwise equal when nothing went external
            Lb.route(x, wr, b)
            for w in range(big.n_waves()):
                big.step(l, Lb.counts, 1.0, w, Lb.slot_of, Lb.ext, Lb.step_counts)
                Lb.experts(x, Lb.slot_of, big.slot_pool, pool.S, 256)
            out_b = Lb.combine(T, Lb.ext, None).cpu().numpy()
            if not C:
                assert np.array_equal(out, out_b), f"step {step} layer {l}: output depends on the cache"
            if step % 5 == 0 or C:
                ref = moe.moe_layer(formats.to_f64(x), ri, rw, ol.experts(l), act_round=bf16_act_round(T, cfg.top_k))
                assert_close_layer(out, ref, fro=1e-2)
    key, stamp, clock = cache.export()
    sk, ss = sim.state()
    assert key.tolist() == sk.tolist() and stamp.tolist() == ss.tolist() and clock == sim.clock
    st = cache.stats()
    assert (st.hits, st.fills, st.externals) == (sim.hits, sim.fills, sim.externals)
    assert st.externals > 0 and st.fills > 0
    # every resident slot holds the bytes of its key's host record
    for s, kk in enumerate(key.tolist()):
        if kk >= 0:
            l, e = divmod(kk, 64)
            host = pool.row(l % 4, e).to(DEV)
            assert torch.equal(sp[s * pool.S:(s + 1) * pool.S], host), f"slot {s}"
    assert ft.ft_get_device_error() == 0


def test_split_fill_step_equals_plain_step(ft):
    """ft_cache_step_split + two expert calls == ft_cache_step + one call, bit for bit.

    Two caches over one host pool follow the same trace (T = 1, 4, 16; two waves
    per step; miss split 0.6 from step 12).  The split side runs eagerly, then
    from step 20 as CUDA graphs captured per layer step (the fill stream forks
    from and joins the capture stream).  Decisions, step counts, outputs,
    counters and the final tables must be identical."""
    cfg = synth.MoEConfig("trace", 256, 64, 4, 256, 4, synth.W_BF16, "bf16", seed=5, zipf_s=1.1)
    pool, sp, cache = make_cache(ft, cfg, 4, 40, 40)
    sp2 = torch.empty(40 * pool.S, dtype=torch.uint8, device=DEV)
    split = ft.Cache(cfg.n_layers, cfg.n_experts, 4, 40, 40, pool.S, pool.ptr, sp2)
    assert cache.n_waves() == 2
    routers = [synth.router_weights(cfg, l, DEV) for l in range(4)]
    L, Ls = ft.MoELayer(cfg, 16), ft.MoELayer(cfg, 16)
    fs = torch.cuda.Stream()
    traces = {T: synth.AR1Trace(cfg, T, DEV, tag=T) for T in (1, 4, 16)}
    xs = torch.empty(16, cfg.hidden, dtype=torch.bfloat16, device=DEV)
    sc_p = torch.zeros(2, 4, dtype=torch.int32, device=DEV)
    sc_s = torch.zeros(2, 4, dtype=torch.int32, device=DEV)
    merged = torch.empty(2, cfg.n_experts, dtype=torch.int32, device=DEV)
    graphs = []

    def split_layer(T, l, ratio):
        x = xs[:T]
        Ls.route(x, *routers[l])
        for w in range(2):
            split.step_split(l, Ls.counts, ratio, w, Ls.slot_of, Ls.slot_fill, Ls.ext, sc_s[w], fill_stream=fs)
            Ls.experts(x, Ls.slot_of, sp2, pool.S, 40)
            split.fill_join()
            merged[w].copy_(torch.where(Ls.slot_fill >= 0, Ls.slot_fill, Ls.slot_of))
            Ls.experts(x, Ls.slot_fill, sp2, pool.S, 40)
        return Ls.combine(T, Ls.ext, None)

    n_fill = 0
    for step in range(30):
        T = (1, 4, 16)[step % 3]
        x = traces[T].next()
        xs[:T].copy_(x)
        ratio = 1.0 if step < 12 else 0.6
        for l in range(4):
            L.route(x, *routers[l])
            exp_slots = []
            for w in range(2):
                cache.step(l, L.counts, ratio, w, L.slot_of, L.ext, sc_p[w])
                exp_slots.append(L.slot_of.clone())
                L.experts(x, L.slot_of, sp, pool.S, 40)
            out = L.combine(T, L.ext, None).clone()
            if step < 20:
                out_s = split_layer(T, l, ratio).clone()
            else:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    out_g = split_layer(T, l, ratio)
                g.replay()
                graphs.append(g)
                out_s = out_g.clone()
            torch.cuda.synchronize()
            for w in range(2):
                assert torch.equal(merged[w], exp_slots[w]), f"step {step} layer {l} wave {w}"
            assert torch.equal(sc_p, sc_s)
            assert torch.equal(L.ext, Ls.ext)
            assert torch.equal(out, out_s), f"step {step} layer {l}"
            n_fill += int(sc_p[:, 2].sum())
    assert n_fill > 0
    a, b = cache.stats(), split.stats()
    assert (a.steps, a.hits, a.fills, a.externals, a.bytes_h2d) == (b.steps, b.hits, b.fills, b.externals, b.bytes_h2d)
    assert a.externals > 0
    ka, sa, ca = cache.export()
    kb, sb, cb = split.export()
    assert ka.tolist() == kb.tolist() and sa.tolist() == sb.tolist() and ca == cb
    for slot, key in enumerate(ka.tolist()):              # resident slots hold the same bytes
        if key >= 0:
            assert torch.equal(sp[slot * pool.S:(slot + 1) * pool.S], sp2[slot * pool.S:(slot + 1) * pool.S])
    del graphs
    assert ft.ft_get_device_error() == 0


def test_split_fill_needs_join(ft):
    """Until ft_cache_fill_join, the handle refuses the next step, a resize and streaming (FT_ESTATE)."""
    cfg = synth.MoEConfig("trace", 256, 64, 4, 256, 4, synth.W_BF16, "bf16", seed=5, zipf_s=1.1)
    pool, sp, cache = make_cache(ft, cfg, 4, 64, 64)
    L = ft.MoELayer(cfg, 4)
    x = synth.activations(cfg, 4, device=DEV)
    L.route(x, *synth.router_weights(cfg, 0, DEV))
    fs = torch.cuda.Stream()
    cache.step_split(0, L.counts, 1.0, 0, L.slot_of, L.slot_fill, L.ext, L.step_counts, fill_stream=fs)
    for call in (lambda: cache.step(1, L.counts, 1.0, 0, L.slot_of, L.ext),
                 lambda: cache.step_split(1, L.counts, 1.0, 0, L.slot_of, L.slot_fill, L.ext, fill_stream=fs),
                 lambda: cache.resize(32),
                 lambda: ft.Stream(cache)):
        with pytest.raises(ft.FTError) as ei:
            call()
        assert ei.value.status == ft.FT_ESTATE
    cache.fill_join()
    cache.fill_join()                                 # a second join is a no-op
    cache.step(1, L.counts, 1.0, 0, L.slot_of, L.ext)
    # fill_stream == stream: both launches on one stream, nothing to join
    cache.step_split(2, L.counts, 1.0, 0, L.slot_of, L.slot_fill, L.ext)
    cache.step(3, L.counts, 1.0, 0, L.slot_of, L.ext)
    torch.cuda.synchronize()
    assert cache.stats().steps == 4
    assert ft.ft_get_device_error() == 0


def test_fill_blocks_setting(ft):
    """The fill's block count changes its speed only: one block still copies every record exactly."""
    cfg = synth.MoEConfig("trace", 256, 64, 4, 256, 4, synth.W_BF16, "bf16", seed=5, zipf_s=1.1)
    pool, sp, cache = make_cache(ft, cfg, 4, 64, 64)
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    for bad in (0, -1, 4 * n_sm + 1):
        with pytest.raises(ft.FTError) as ei:
            cache.set_fill_blocks(bad)
        assert ei.value.status == ft.FT_EINVAL
    cache.set_fill_blocks(4 * n_sm)
    cache.set_fill_blocks(1)
    L = ft.MoELayer(cfg, 16)
    x = synth.activations(cfg, 16, device=DEV)
    L.route(x, *synth.router_weights(cfg, 2, DEV))
    cache.step(2, L.counts, 1.0, 0, L.slot_of, L.ext, L.step_counts)
    torch.cuda.synchronize()
    assert int(L.step_counts[2]) > 1
    key, _, _ = cache.export()
    for slot, kk in enumerate(key.tolist()):
        if kk >= 0:
            l, e = divmod(kk, 64)
            assert torch.equal(sp[slot * pool.S:(slot + 1) * pool.S], pool.row(l % 4, e).to(DEV)), f"slot {slot}"
    assert ft.ft_get_device_error() == 0


# ---------------------------------------------------------------- prefill streaming

def test_stream_double_buffered_and_serialized(ft):
    cfg = synth.MoEConfig("stream", 512, 32, 4, 256, 6, synth.W_BF16, "bf16", seed=6)
    n_phys = 3
    pool, sp, cache = make_cache(ft, cfg, n_phys, 80, 80)
    L = ft.MoELayer(cfg, 300)
    sim = LRUSim(80, 32)
    routers = [synth.router_weights(cfg, l, DEV) for l in range(6)]
    # warm the cache with a few decode steps
    tr = synth.AR1Trace(cfg, 2, DEV)
    for step in range(3):
        x = tr.next()
        for l in range(6):
            L.route(x, *routers[l])
            run_waves(ft, L, cache, l, x, 1.0, sim)
    # reference: every record resident in a fused pool, slot = phys_layer * E + e
    fused = pool.host.to(DEV)
    xp = synth.activations(cfg, 300, tag=9, device=DEV)
    ref_out = []
    for l in range(6):
        so = torch.arange(32, dtype=torch.int32, device=DEV) + (l % n_phys) * 32
        ref_out.append(L.forward_slots(xp, *routers[l], so, fused, pool.S, n_phys * 32).clone())
    slot_of = torch.empty(32, dtype=torch.int32, device=DEV)
    for serialized in (False, True):
        st = ft.Stream(cache, serialized)
        base, _ = sim.stream_begin()
        for l in range(6):
            st.layer(l, l + 1 if l < 5 else -1, slot_of)
            out = L.forward_slots(xp, *routers[l], slot_of, sp, pool.S, 80)
            st.layer_done(l)
            assert torch.equal(out, ref_out[l]), f"layer {l} serialized={serialized}"
        assert st.bytes() == 6 * 32 * pool.S
        st.destroy()
        sim.stream_end([(4, 0), (5, 1)])
        key, stamp, clock = cache.export()
        sk, ss = sim.state()
        assert key.tolist() == sk.tolist() and stamp.tolist() == ss.tolist() and clock == sim.clock
        # decode after prefill: the adopted layers hit
        x = tr.next()
        L.route(x, *routers[5])
        run_waves(ft, L, cache, 5, x, 1.0, sim)
        assert int(L.step_counts[2]) == 0          # no fills: layer 5 is resident
    # one streamed layer against the oracle on sampled tokens
    rows = np.arange(0, 300, 37)
    ol = OracleLayer(cfg, n_phys)
    z = moe.router_logits(formats.to_f64(xp[rows]), formats.to_f64(routers[2][0]), formats.to_f64(routers[2][1]))
    ri, rw = moe.route(z, 4)
    assert not moe.near_ties(z, 4).any()
    ref = moe.moe_layer(formats.to_f64(xp[rows]), ri, rw, ol.experts(2), act_round=TC_ROUND)
    assert_close_layer(ref_out[2].cpu().numpy()[rows], ref, fro=1e-2)
    assert ft.ft_get_device_error() == 0


def test_stream_needs_two_layers_of_slots(ft):
    cfg = synth.MoEConfig("small", 256, 32, 2, 256, 2, synth.W_BF16, "bf16", seed=8)
    pool, sp, cache = make_cache(ft, cfg, 2, 40, 64)
    with pytest.raises(ft.FTError) as ei:
        ft.Stream(cache)
    assert ei.value.status == ft.FT_EUNSUPPORTED
    cache.resize(64)
    st = ft.Stream(cache)
    with pytest.raises(ft.FTError) as ei:
        cache.resize(30)                         # not a safe point: buffers are held
    assert ei.value.status == ft.FT_ESTATE
    st.destroy()


# ---------------------------------------------------------------- full-size decode and prefill shapes

def test_decode_full_size_sampled(ft):
    """H=2048, E=256, k=8, I=512, 40 logical layers over 2 physical layers, 4096 slots, T=64;
    the first step with ft_cache_step, the others with the split form."""
    cfg = synth.DECODE_BF16
    n_phys = 2
    pool, sp, cache = make_cache(ft, cfg, n_phys, 4096, 4096)
    L = ft.MoELayer(cfg, 64)
    sim = LRUSim(4096, 256)
    ol = OracleLayer(cfg, n_phys)
    routers = [synth.router_weights(cfg, l, DEV) for l in range(cfg.n_layers)]
    tr = synth.AR1Trace(cfg, 64, DEV)
    sample = [0, 9, 33, 63]
    fill_stream = torch.cuda.Stream()
    for step in range(3):
        x = tr.next()
        for l in range(cfg.n_layers):
            L.route(x, *routers[l])
            z = L.logits[:64].cpu().numpy().astype(np.float64)
            ri, rw = moe.route(z, 8)
            assert np.array_equal(L.idx[:64].cpu().numpy(), ri)
            # steps 1 and 2 overlap the fill with the hits (split form)
            run_waves(ft, L, cache, l, x, 1.0, sim, fill_stream=fill_stream if step else None)
            out = L.combine(64, L.ext, None)
            if (step, l) in ((0, 0), (0, 21), (2, 39), (2, 7)):
                xs = formats.to_f64(x[sample])
                zr = moe.router_logits(xs, formats.to_f64(routers[l][0]), formats.to_f64(routers[l][1]))
                r2, w2 = moe.route(zr, 8)
                ok = ~moe.near_ties(zr, 8)
                assert np.array_equal(r2[ok], ri[sample][ok])
                ref = moe.moe_layer(xs, ri[sample], rw[sample], ol.experts(l), act_round=TC_ROUND)
                assert_close_layer(out.cpu().numpy()[sample], ref, fro=1e-2)
    st = cache.stats()
    assert (st.hits, st.fills) == (sim.hits, sim.fills)
    assert ft.ft_get_device_error() == 0


def test_prefill_chunk_full_size_sampled(ft):
    """8192 tokens through one H=2048, E=256, k=8, I=512 layer with every expert resident."""
    cfg = synth.PREFILL_BF16
    L_ = ft.ft_expert_layout_get(cfg.wtype, cfg.hidden, cfg.inter)
    S = int(L_.bytes)
    fused = torch.empty(256 * S, dtype=torch.uint8, device=DEV)
    for e in range(256):
        ft.pack_expert(synth.expert_weights(cfg, 0, e, DEV), cfg.wtype, L_, fused[e * S:(e + 1) * S])
    L = ft.MoELayer(cfg, 8192)
    wr, b = synth.router_weights(cfg, 0, DEV)
    x = synth.activations(cfg, 8192, tag=1, device=DEV)
    so = torch.arange(256, dtype=torch.int32, device=DEV)
    out = L.forward_slots(x, wr, b, so, fused, S, 256).cpu().numpy()
    counts = L.counts.cpu().numpy()
    assert counts.sum() == 8192 * 8 and (counts > 0).sum() >= 250    # near-uniform routing touches ~all experts
    z = L.logits.cpu().numpy().astype(np.float64)
    ri, rw = moe.route(z, 8)
    assert np.array_equal(L.idx.cpu().numpy(), ri)
    rows = np.random.default_rng(0).choice(8192, 24, replace=False)
    ol = OracleLayer(cfg, 1)
    ref = moe.moe_layer(formats.to_f64(x[rows]), ri[rows], rw[rows], ol.experts(0), act_round=TC_ROUND)
    assert_close_layer(out[rows], ref, fro=1e-2)
