"""Kernel-level parity of libft against the fp64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import synth
from conftest import CC_MAX_ASSIGNMENTS, assert_close_layer, rel_fro
from oracle import formats, moe

pytestmark = pytest.mark.gpu
DEV = "cuda"
TC_FORMATS = (synth.W_BF16, synth.W_NVFP4, synth.W_MXFP4)  # tensor-core path below 2048 assignments


@pytest.fixture(scope="module")
def ft(ftlib):
    assert torch.cuda.is_available()
    return ftlib


def _i32(shape):
    return torch.empty(shape, dtype=torch.int32, device=DEV)


def _f32(shape):
    return torch.empty(shape, dtype=torch.float32, device=DEV)


# ---------------------------------------------------------------- route

@pytest.mark.parametrize("T,E,k,seed", [(1, 16, 2, 0), (37, 256, 8, 1), (4099, 256, 8, 2), (64, 16, 2, 3),
                                        (5, 1024, 16, 4), (3, 40, 6, 5), (9, 33, 1, 6), (2, 4, 4, 7)])
def test_route_bit_exact_indices(ft, T, E, k, seed):
    g = torch.Generator().manual_seed(seed)
    z = torch.randn(T, E, generator=g)
    z[::3] = torch.round(z[::3] * 2) / 2          # rows with many exact ties
    z[1::7] = 0.25                                # rows of all-equal logits
    zd = z.to(DEV)
    idx, w = _i32((T, k)), _f32((T, k))
    ft.ft_route(zd, k, idx, w)
    torch.cuda.synchronize()
    ri, rw = moe.route(z.double().numpy(), k)
    assert np.array_equal(idx.cpu().numpy(), ri)
    assert np.abs(w.cpu().numpy() - rw).max() <= 2e-6
    assert np.allclose(w.cpu().numpy().sum(1), 1.0, atol=3e-6)


def test_route_empty_batch(ft):
    z = _f32((0, 16))
    ft.ft_route(z, 2, _i32((0, 2)), _f32((0, 2)))
    torch.cuda.synchronize()


# ---------------------------------------------------------------- permute

@pytest.mark.parametrize("T,k,E,seed,distinct", [(1, 1, 16, 0, True), (64, 2, 16, 1, True), (8192, 8, 256, 2, True),
                                                 (33, 8, 256, 3, True), (1000, 6, 512, 4, False),
                                                 (129, 3, 5, 5, False), (0, 8, 256, 6, True)])
def test_permute_bit_exact(ft, T, k, E, seed, distinct):
    rng = np.random.default_rng(seed)
    if distinct:
        idx = np.array([rng.permutation(E)[:k] for _ in range(T)], dtype=np.int32).reshape(T, k)
    else:
        idx = rng.integers(0, E, size=(T, k)).astype(np.int32)
    d = torch.from_numpy(idx).to(DEV)
    counts, offsets, perm, inv = _i32(E), _i32(E + 1), _i32(max(T * k, 1)), _i32(max(T * k, 1))
    ft.ft_permute(d, E, counts, offsets, perm, inv)
    torch.cuda.synchronize()
    rc, ro, rp, ri = moe.permute(idx, E)
    assert np.array_equal(counts.cpu().numpy(), rc)
    assert np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(perm.cpu().numpy()[: T * k], rp)
    assert np.array_equal(inv.cpu().numpy()[: T * k], ri)


# ---------------------------------------------------------------- router logits

@pytest.mark.parametrize("T,H,E,dt", [(1, 2048, 256, "bf16"), (64, 2048, 256, "bf16"), (300, 256, 16, "f32"),
                                      (7, 4096, 256, "bf16"), (8192, 2048, 256, "bf16")])
def test_router_logits(ft, T, H, E, dt):
    x = synth.normal((T, H), 1.0, 11, DEV)
    wr = synth.normal((E, H), 0.02, 12, DEV)
    if dt == "bf16":
        x, wr = x.to(torch.bfloat16), wr.to(torch.bfloat16)
    b = synth.normal((E,), 1.0, 13, DEV)
    z = _f32((T, E))
    ft.ft_router_logits(x, wr, b, z)
    torch.cuda.synchronize()
    rows = np.arange(T) if T <= 512 else np.random.default_rng(0).choice(T, 256, replace=False)
    ref = moe.router_logits(formats.to_f64(x[rows]), formats.to_f64(wr), formats.to_f64(b))
    got = z.cpu().numpy()[rows]
    # fp32 accumulation of H products of magnitude ~0.02
    assert np.abs(got - ref).max() <= 2e-5 * (1 + np.abs(ref).max())


# ---------------------------------------------------------------- combine

@pytest.mark.parametrize("T,k,H,E,ext,partial", [(50, 8, 512, 32, False, False), (50, 8, 512, 32, True, True),
                                                 (1, 2, 256, 16, True, False), (300, 6, 4096, 256, False, True)])
def test_combine(ft, T, k, H, E, ext, partial):
    rng = np.random.default_rng(T + k)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    _, _, _, inv = moe.permute(idx, E)
    w = rng.random((T, k)).astype(np.float32)
    w /= w.sum(1, keepdims=True)
    Y = rng.normal(size=(T * k, H)).astype(np.float32)
    flags = (rng.random(E) < 0.3).astype(np.int32) if ext else None
    P = rng.normal(size=(T, H)).astype(np.float32) if partial else None
    out = _f32((T, H))
    t = lambda a: None if a is None else torch.from_numpy(a).to(DEV)
    ft.ft_combine(t(Y), t(inv), t(idx), t(w), t(flags), t(P), E, out)
    torch.cuda.synchronize()
    skip = None if flags is None else flags[idx].astype(bool)
    ref = moe.combine(Y.astype(np.float64), inv, w.astype(np.float64), k, skip=skip,
                      partial=None if P is None else P.astype(np.float64))
    assert np.abs(out.cpu().numpy() - ref).max() <= 1e-5 * (1 + np.abs(ref).max())


# ---------------------------------------------------------------- grouped experts

def _tiny_cfg(wtype, H, I, E, k, xdt="bf16", seed=7):
    return synth.MoEConfig(f"t{wtype}_{H}_{I}", H, E, k, I, 1, wtype, xdt, seed=seed)


@pytest.mark.parametrize("wtype,H,I,E,k,T,xdt", [
    (0, 256, 256, 8, 2, 37, "f32"),
    (1, 512, 256, 8, 2, 37, "bf16"),
    (1, 2048, 512, 16, 8, 64, "bf16"),
    (1, 2048, 512, 16, 8, 1, "bf16"),       # one decode token of bf16 experts: the CUDA-core path
    (1, 512, 256, 8, 2, 3, "bf16"),         # T*k = 6: the CUDA-core path
    (1, 768, 512, 4, 2, 200, "bf16"),       # ~100 rows per expert: many row chunks; H not a power of two
    (2, 1024, 512, 8, 2, 45, "bf16"),
    (3, 1024, 512, 8, 3, 29, "bf16"),
    (3, 768, 256, 6, 2, 11, "bf16"),        # FP4 with a partial 1024-element chunk
    (4, 2048, 1024, 8, 2, 21, "bf16"),
    (4, 256, 256, 5, 1, 3, "bf16"),
])
def test_expert_grouped_parity(ft, wtype, H, I, E, k, T, xdt):
    cfg = _tiny_cfg(wtype, H, I, E, k, xdt)
    L = ft.ft_expert_layout_get(wtype, H, I)
    S = int(L.bytes)
    n_slots = E + 3
    pool = torch.zeros(n_slots * S, dtype=torch.uint8, device=DEV)
    rng = np.random.default_rng(H + I + wtype)
    slot_perm = rng.permutation(n_slots)[:E]
    comps = {}
    for e in range(E):
        comps[e] = synth.expert_weights(cfg, 0, e, DEV)
        ft.pack_expert(comps[e], wtype, L, pool[slot_perm[e] * S:(slot_perm[e] + 1) * S])
    x = synth.activations(cfg, T, tag=3, device=DEV)
    on_tc = wtype in TC_FORMATS and not (wtype == synth.W_BF16 and T * k <= CC_MAX_ASSIGNMENTS)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    counts, offsets, perm, inv = moe.permute(idx, E)
    slot_of = slot_perm.astype(np.int32).copy()
    skipped = {int(E - 1)}                       # one expert not evaluated (rows untouched)
    slot_of[E - 1] = -1
    if E > 3:
        slot_of[1] = -2                          # one expert evaluated elsewhere
        skipped.add(1)
    y = torch.full((T * k, H), float("nan"), dtype=torch.float32, device=DEV)
    ws = torch.empty(ft.ft_expert_grouped_workspace(T, k, H, I), dtype=torch.uint8, device=DEV)
    ft.ft_expert_grouped(x, k, I, E, wtype, torch.from_numpy(perm).to(DEV), torch.from_numpy(offsets).to(DEV),
                         torch.from_numpy(slot_of).to(DEV), pool, S, n_slots, y, ws)
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
        # bf16 weights on the tensor cores round the intermediate to bf16 (one-token batches of
        # bf16 weights run on the CUDA cores, fp32 throughout); NVFP4 / MXFP4 weights at small
        # batches (H and I multiples of 256) take the block-scaled FP4 MMA, which quantises the
        # token rows and the intermediate to the weights' format
        x_round, act_round = None, (formats.round_to_bf16 if on_tc else None)
        if wtype in (synth.W_NVFP4, synth.W_MXFP4) and H % 256 == 0 and I % 256 == 0:
            act_round = x_round = (formats.quant_act_nvfp4 if wtype == synth.W_NVFP4 else formats.quant_act_mxfp4)
        ref.append(moe.expert_ffn(xs[perm[rows] // k], g, u, d, act_round=act_round, x_round=x_round))
        got.append(Y[rows])
    got, ref = np.concatenate(got), np.concatenate(ref)
    if on_tc:
        assert_close_layer(got, ref, fro=1e-2)
        assert rel_fro(got, ref) < 2e-3
    else:
        assert_close_layer(got, ref)
        # the declared arithmetic is fp32 throughout (fp32 intermediate): far tighter than the bar
        assert rel_fro(got, ref) < 2e-5


def test_expert_grouped_independent_of_slot_and_batch(ft):
    """Same expert, same rows: bitwise equal output whatever the slot or the other experts in the call."""
    cfg = _tiny_cfg(1, 512, 256, 6, 2)
    L = ft.ft_expert_layout_get(1, 512, 256)
    S = int(L.bytes)
    pool = torch.zeros(12 * S, dtype=torch.uint8, device=DEV)
    comps = [synth.expert_weights(cfg, 0, e, DEV) for e in range(6)]
    for e in range(6):
        ft.pack_expert(comps[e], 1, L, pool[e * S:(e + 1) * S])
        ft.pack_expert(comps[e], 1, L, pool[(11 - e) * S:(12 - e) * S])
    T, k = 40, 2
    rng = np.random.default_rng(1)
    idx = np.stack([rng.permutation(6)[:k] for _ in range(T)]).astype(np.int32)
    counts, offsets, perm, inv = moe.permute(idx, 6)
    x = synth.activations(cfg, T, tag=1, device=DEV)
    ws = torch.empty(ft.ft_expert_grouped_workspace(T, k, 512, 256), dtype=torch.uint8, device=DEV)
    args = (torch.from_numpy(perm).to(DEV), torch.from_numpy(offsets).to(DEV))
    y1 = torch.zeros(T * k, 512, device=DEV)
    ft.ft_expert_grouped(x, k, 256, 6, 1, *args, torch.arange(6, dtype=torch.int32, device=DEV), pool, S, 12, y1, ws)
    y2 = torch.zeros(T * k, 512, device=DEV)
    only2 = torch.full((6,), -1, dtype=torch.int32, device=DEV)
    only2[2] = 11 - 2
    ft.ft_expert_grouped(x, k, 256, 6, 1, *args, only2, pool, S, 12, y2, ws)
    torch.cuda.synchronize()
    r = slice(int(offsets[2]), int(offsets[3]))
    assert torch.equal(y1[r], y2[r])


# ---------------------------------------------------------------- device error word

def test_out_of_range_expert_is_recorded_not_faulted(ft):
    T, k, H, E = 4, 2, 256, 8
    idx = torch.tensor([[0, 1], [2, 3], [4, 99], [6, 7]], dtype=torch.int32, device=DEV)  # 99 is out of range
    inv = torch.arange(T * k, dtype=torch.int32, device=DEV)
    w = torch.full((T, k), 0.5, device=DEV)
    y = torch.ones(T * k, H, device=DEV)
    out = _f32((T, H))
    assert ft.ft_get_device_error() == 0
    ft.ft_combine(y, inv, idx, w, None, None, E, out)
    assert ft.ft_get_device_error() == 1      # FT_DERR_EXPERT_INDEX
    assert ft.ft_get_device_error() == 0      # cleared by the read
    o = out.cpu().numpy()
    assert np.allclose(o[[0, 1, 3]], 1.0) and np.allclose(o[2], 0.5)


def test_bounded_wait_gives_up_and_reports(ft):
    """A barrier wait that nothing completes times out, records FT_DERR_TIMEOUT and returns.

    This is the failure path of every on-chip wait in the tensor-core kernels,
    run on purpose with a 20 ms limit; afterwards the context keeps working."""
    assert ft.ft_get_device_error() == 0
    done = torch.full((1,), 7, dtype=torch.int32, device=DEV)
    ft.ft_debug_bounded_wait(20_000_000, done)
    torch.cuda.synchronize()
    assert int(done) == 0                       # the wait did not complete
    assert ft.ft_get_device_error() == 5        # FT_DERR_TIMEOUT, cleared by the read
    assert ft.ft_get_device_error() == 0
    # the context is still usable: a routing call gives the oracle's answer
    z = torch.tensor([[0.5, 2.0, -1.0, 2.0]], device=DEV)
    idx, w = _i32((1, 2)), _f32((1, 2))
    ft.ft_route(z, 2, idx, w)
    assert idx.cpu().tolist() == [[1, 3]]


# ---------------------------------------------------------------- fused routing (one grid launch)

@pytest.mark.parametrize("T,H,E,k,dt,zipf", [(1, 2048, 256, 8, "bf16", True), (4, 2048, 256, 8, "bf16", True),
                                             (16, 2048, 256, 8, "bf16", False), (3, 4096, 256, 6, "bf16", True),
                                             (9, 6144, 256, 8, "bf16", False), (5, 256, 16, 2, "f32", False),
                                             (16, 512, 512, 16, "bf16", False), (7, 256, 40, 3, "f32", True),
                                             (17, 2048, 256, 8, "bf16", True), (64, 2048, 256, 8, "bf16", True),
                                             (8, 2048, 256, 8, "bf16", True), (6, 512, 512, 16, "bf16", False),
                                             (2, 6144, 128, 8, "bf16", True), (8, 6144, 256, 8, "bf16", False),
                                             (3, 512, 512, 16, "f32", False), (61, 6144, 128, 8, "bf16", True)])
def test_route_fused_equals_the_three_kernels_and_the_oracle(ft, T, H, E, k, dt, zipf):
    """ft_route_fused gives bit for bit the logits, routing and permutation of
    ft_router_logits + ft_route + ft_permute (one grid launch up to 8 tokens,
    the grouping by one warp up to 32 assignments, else by the CTA; the three
    kernels above), and the oracle's routing and grouping of those logits; its
    arrival counters are zero again after every call."""
    x = synth.normal((T, H), 1.0, 21 + T, DEV)
    wr = synth.normal((E, H), 0.02, 22 + E, DEV)
    if dt == "bf16":
        x, wr = x.to(torch.bfloat16), wr.to(torch.bfloat16)
    cfg = synth.MoEConfig("rf", H, E, k, 128, 1, synth.W_BF16, dt, seed=3, zipf_s=1.1 if zipf else 0.0)
    b = synth.zipf_bias(cfg, 0).to(DEV)
    arrivals = torch.zeros(ft.FT_ROUTE_ARRIVAL_WORDS, dtype=torch.int32, device=DEV)
    outs = []
    for fused in (True, True, False):          # the fused call twice: the counters are reused
        z, idx, w = _f32((T, E)), _i32((T, k)), _f32((T, k))
        counts, offsets, perm, inv = _i32(E), _i32(E + 1), _i32(max(T * k, 1)), _i32(max(T * k, 1))
        if fused:
            ft.ft_route_fused(x, wr, b, k, z, idx, w, counts, offsets, perm, inv, arrivals)
        else:
            ft.ft_router_logits(x, wr, b, z)
            ft.ft_route(z, k, idx, w)
            ft.ft_permute(idx, E, counts, offsets, perm, inv)
        torch.cuda.synchronize()
        outs.append([t.cpu().numpy() for t in (z, idx, w, counts, offsets, perm[: T * k], inv[: T * k])])
        assert not arrivals.any()
    for run in outs[1:]:
        for a, c in zip(outs[0], run):
            assert np.array_equal(a, c)
    z, idx, w, counts, offsets, perm, inv = outs[0]
    ref = moe.router_logits(formats.to_f64(x), formats.to_f64(wr), formats.to_f64(b))
    assert np.abs(z - ref).max() <= 2e-5 * (1 + np.abs(ref).max())
    ri, rw = moe.route(z.astype(np.float64), k)
    assert np.array_equal(idx, ri)
    assert np.abs(w - rw).max() <= 1e-6
    rc, ro, rp, rinv = moe.permute(idx, E)
    for got, want in ((counts, rc), (offsets, ro), (perm, rp), (inv, rinv)):
        assert np.array_equal(got, want)
    assert ft.ft_get_device_error() == 0


def test_route_fused_in_a_graph_and_on_two_streams(ft):
    """Replays of one captured call, and two calls in flight on two streams with
    one counter array each, give the eager results; the counters end at zero."""
    T, H, E, k = 8, 2048, 256, 8
    xs = [synth.normal((T, H), 1.0, 40 + i, DEV).to(torch.bfloat16) for i in range(2)]
    wr = synth.normal((E, H), 0.02, 42, DEV).to(torch.bfloat16)

    def bufs():
        return [_f32((T, E)), _i32((T, k)), _f32((T, k)), _i32(E), _i32(E + 1), _i32(T * k), _i32(T * k),
                torch.zeros(ft.FT_ROUTE_ARRIVAL_WORDS, dtype=torch.int32, device=DEV)]

    want = []
    for x in xs:
        o = bufs()
        ft.ft_route_fused(x, wr, None, k, *o)
        torch.cuda.synchronize()
        want.append([t.cpu() for t in o[:7]])
    # graph replay
    o = bufs()
    xg = xs[0].clone()
    g = torch.cuda.CUDAGraph()
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        with torch.cuda.graph(g, stream=st):
            ft.ft_route_fused(xg, wr, None, k, *o, stream=st)
    for i in (1, 0, 1):
        xg.copy_(xs[i])
        g.replay()
        torch.cuda.synchronize()
        assert all(torch.equal(a.cpu(), b) for a, b in zip(o[:7], want[i]))
        assert not o[7].any()
    # two streams at once
    outs = [bufs(), bufs()]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for rep in range(20):
        for i in range(2):
            ft.ft_route_fused(xs[i], wr, None, k, *outs[i], stream=streams[i])
    torch.cuda.synchronize()
    for i in range(2):
        assert all(torch.equal(a.cpu(), b) for a, b in zip(outs[i][:7], want[i]))
        assert not outs[i][7].any()
    assert ft.ft_get_device_error() == 0


def test_route_fused_reports_counters_that_were_not_zero(ft):
    """A nonzero arrival counter at launch is recorded as FT_DERR_TABLE (no wait, no fault)."""
    T, H, E, k = 8, 512, 64, 4
    x = synth.normal((T, H), 1.0, 50, DEV)
    wr = synth.normal((E, H), 0.02, 51, DEV)
    arrivals = torch.zeros(ft.FT_ROUTE_ARRIVAL_WORDS, dtype=torch.int32, device=DEV)
    arrivals[0] = 1 << 20
    assert ft.ft_get_device_error() == 0
    o = [_f32((T, E)), _i32((T, k)), _f32((T, k)), _i32(E), _i32(E + 1), _i32(T * k), _i32(T * k)]
    ft.ft_route_fused(x, wr, None, k, *o, arrivals)
    torch.cuda.synchronize()
    assert ft.ft_get_device_error() == 4        # FT_DERR_TABLE, cleared by the read
    arrivals.zero_()
    ft.ft_route_fused(x, wr, None, k, *o, arrivals)
    torch.cuda.synchronize()
    assert ft.ft_get_device_error() == 0 and not arrivals.any()
    ri, _ = moe.route(o[0].cpu().numpy().astype(np.float64), k)
    assert np.array_equal(o[1].cpu().numpy(), ri)


def test_route_fused_empty_batch(ft):
    E, k = 256, 8
    counts, offsets = _i32(E), _i32(E + 1)
    x = torch.zeros(0, 2048, dtype=torch.bfloat16, device=DEV)
    wr = torch.zeros(E, 2048, dtype=torch.bfloat16, device=DEV)
    one = _i32(1)
    ft.ft_route_fused(x, wr, None, k, _f32((1, E)), _i32((1, k)), _f32((1, k)), counts, offsets, one, one, None)
    torch.cuda.synchronize()
    assert (counts.cpu().numpy() == 0).all() and (offsets.cpu().numpy() == 0).all()
