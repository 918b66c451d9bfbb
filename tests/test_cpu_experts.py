"""The host-side expert executor against the fp64 oracle, on the CPU ([Review] §2.5).

ft_cpu_experts evaluates the experts marked external from the host pool's
records with a pool of CPU threads and writes the gate-weighted partial output
per token.  The records here live in ordinary host memory (the executor reads
any host memory), so these tests need no GPU.  Every weight format is checked
on a second physical layer of the pool, with duplicate and absent experts.
"""
import numpy as np
import pytest
import torch

import synth
from conftest import assert_close_layer, rel_fro
from oracle import formats, moe


def available_forms(ft):
    """The row forms this CPU runs (0 portable, 1 AVX2, 2 AVX-512)."""
    prev = ft.ft_debug_host_simd(-1)
    forms = []
    for f in (0, 1, 2):
        ft.ft_debug_host_simd(f)
        if ft.ft_debug_host_simd(-1) == f:
            forms.append(f)
    ft.ft_debug_host_simd(prev)
    return forms


@pytest.fixture(params=[2, 1, 0], ids=["avx512", "avx2", "portable"])
def host_form(request, ftlib):
    """One row form of the host executor; skipped where this CPU does not run it."""
    if request.param not in available_forms(ftlib):
        pytest.skip(f"this CPU does not run the {ftlib.HOST_FORMS[request.param]} form")
    prev = ftlib.ft_debug_host_simd(-1)
    ftlib.ft_debug_host_simd(request.param)
    yield request.param
    ftlib.ft_debug_host_simd(prev)


@pytest.mark.parametrize("wtype,x_dtype", [(synth.W_F32, "f32"), (synth.W_BF16, "bf16"), (synth.W_FP8, "bf16"),
                                           (synth.W_NVFP4, "bf16"), (synth.W_MXFP4, "f32")])
def test_cpu_executor_matches_oracle(ftlib, host_form, wtype, x_dtype):
    ft = ftlib
    H, I, E, k, T = 256, 128, 8, 3, 6
    cfg = synth.MoEConfig(f"cpu{wtype}", H, E, k, I, 2, wtype, x_dtype, seed=60 + wtype)
    L = ft.ft_expert_layout_get(wtype, H, I)
    S = int(L.bytes)
    pool = torch.zeros(2 * E * S, dtype=torch.uint8)
    for l in range(2):
        for e in range(E):
            ft.pack_expert(synth.expert_weights(cfg, l, e, "cpu"), wtype, L, pool[(l * E + e) * S:(l * E + e + 1) * S])
    rng = np.random.default_rng(wtype)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    ext = np.zeros(E, dtype=np.int32)
    ext[[1, 4, 6]] = 1
    idx[0] = [1, 4, 6]                        # a token with all its experts external
    idx[1] = [0, 2, 3]                        # and one with none
    x = synth.activations(cfg, T, tag=2)
    part = torch.full((T, H), float("nan"))
    cpu = ft.CpuExperts(threads=3)
    tid, tw, te = torch.from_numpy(idx), torch.from_numpy(w), torch.from_numpy(ext)
    job = cpu.job(pool.data_ptr(), S, wtype, H, I, E, 1, x, T, k, tid, tw, te, part)
    cpu.run(job)
    got = part.numpy()
    src = moe.ExpertSource(lambda e: synth.expert_weights(cfg, 1, e, "cpu"), wtype)
    ref = moe.moe_layer(formats.to_f64(x), idx, w.astype(np.float64), src, only=[1, 4, 6])
    assert np.all(got[1] == 0.0)
    assert_close_layer(got, ref)
    assert rel_fro(got, ref) < 2e-5
    # a second run on the same handle (scratch reused) gives the same bytes
    part2 = torch.full((T, H), float("nan"))
    cpu.run(cpu.job(pool.data_ptr(), S, wtype, H, I, E, 1, x, T, k, tid, tw, te, part2))
    assert torch.equal(part, part2)
    cpu.destroy()


def test_cpu_executor_rejects_bad_jobs(ftlib):
    ft = ftlib
    cpu = ft.CpuExperts(threads=1)
    x = torch.zeros(2, 256, dtype=torch.bfloat16)
    i32 = torch.zeros(2, 2, dtype=torch.int32)
    job = cpu.job(0, 1 << 20, ft.FT_W_BF16, 256, 128, 4, 0, x, 2, 2, i32, torch.zeros(2, 2),
                  torch.zeros(4, dtype=torch.int32), torch.zeros(2, 256))
    with pytest.raises(ft.FTError):           # no host pool
        cpu.run(job)
    job.host_pool = x.data_ptr()
    job.inter = 100                           # not a multiple of 128
    with pytest.raises(ft.FTError):
        cpu.run(job)
    cpu.destroy()


@pytest.mark.parametrize("wtype", [synth.W_F32, synth.W_BF16, synth.W_FP8, synth.W_NVFP4, synth.W_MXFP4])
def test_cpu_executor_forms_agree(ftlib, wtype):
    """Every vector form this CPU runs against the portable row decode, on many
    tokens per expert (more than one pass of tokens) and several 32-element
    groups per row: the same values up to fp32 summation order."""
    ft = ftlib
    forms = available_forms(ft)
    if len(forms) < 2:
        pytest.skip("no vector form on this CPU")
    H, I, E, k, T = 384, 256, 4, 2, 11
    cfg = synth.MoEConfig(f"forms{wtype}", H, E, k, I, 1, wtype, "bf16", seed=80 + wtype)
    L = ft.ft_expert_layout_get(wtype, H, I)
    S = int(L.bytes)
    pool = torch.zeros(E * S, dtype=torch.uint8)
    for e in range(E):
        ft.pack_expert(synth.expert_weights(cfg, 0, e, "cpu"), wtype, L, pool[e * S:(e + 1) * S])
    idx = torch.tensor([[0, 1]] * 9 + [[2, 0], [3, 2]], dtype=torch.int32)   # expert 0: 10 tokens
    w = torch.rand(T, k, generator=torch.Generator().manual_seed(5))
    ext = torch.tensor([1, 1, 1, 0], dtype=torch.int32)
    x = synth.activations(cfg, T, tag=4)
    outs = {}
    prev = ft.ft_debug_host_simd(-1)
    cpu = ft.CpuExperts(threads=2)
    try:
        for f in forms:
            ft.ft_debug_host_simd(f)
            part = torch.full((T, H), float("nan"))
            cpu.run(cpu.job(pool.data_ptr(), S, wtype, H, I, E, 0, x, T, k, idx, w, ext, part))
            outs[f] = part.numpy().astype(np.float64)
    finally:
        ft.ft_debug_host_simd(prev)
        cpu.destroy()
    src = moe.ExpertSource(lambda e: synth.expert_weights(cfg, 0, e, "cpu"), wtype)
    ref = moe.moe_layer(formats.to_f64(x), idx.numpy(), w.numpy().astype(np.float64), src, only=[0, 1, 2])
    for f in forms[1:]:
        assert np.all(np.isfinite(outs[f]))
        assert rel_fro(outs[f], outs[0]) < 1e-6, ft.HOST_FORMS[f]
        assert rel_fro(outs[f], ref) < 2e-5, ft.HOST_FORMS[f]


_FULL_WEIGHTS = {}


def _full_weights(cfg, e):
    if e not in _FULL_WEIGHTS:
        _FULL_WEIGHTS[e] = synth.expert_weights(cfg, 0, e, "cpu")
    return _FULL_WEIGHTS[e]


def test_cpu_executor_mxfp4_full_shape(ftlib, host_form):
    """The MXFP4 mixed-trace expert shape (H=6144, I=2048) on the host executor, both
    forms, two external experts of three tokens, against the oracle."""
    ft = ftlib
    cfg = synth.MXFP4_MIXED
    H, I, E, k, T = cfg.hidden, cfg.inter, 4, 2, 3
    L = ft.ft_expert_layout_get(cfg.wtype, H, I)
    S = int(L.bytes)
    pool = torch.zeros(E * S, dtype=torch.uint8)
    for e in (1, 2):
        ft.pack_expert(_full_weights(cfg, e), cfg.wtype, L, pool[e * S:(e + 1) * S])
    idx = torch.tensor([[1, 2], [2, 0], [1, 3]], dtype=torch.int32)
    w = torch.tensor([[0.6, 0.4], [0.7, 0.3], [0.5, 0.5]])
    ext = torch.tensor([0, 1, 1, 0], dtype=torch.int32)
    x = synth.activations(cfg, T, tag=7)
    part = torch.full((T, H), float("nan"))
    cpu = ft.CpuExperts(threads=3)
    cpu.run(cpu.job(pool.data_ptr(), S, cfg.wtype, H, I, E, 0, x, T, k, idx, w, ext, part))
    cpu.destroy()
    src = moe.ExpertSource(lambda e: _full_weights(cfg, e), cfg.wtype)
    ref = moe.moe_layer(formats.to_f64(x), idx.numpy(), w.numpy().astype(np.float64), src, only=[1, 2])
    got = part.numpy()
    assert_close_layer(got, ref)
    assert rel_fro(got, ref) < 2e-5


def test_cpu_executor_fp8_every_code(ftlib):
    """Every finite e4m3 byte through every form: gate row i holds byte i in
    column p (zeros elsewhere), the up rows hold 1.0 there, the down matrix is
    the identity and x is one-hot at p, so partial[h] = silu(e4m3(h)) with a
    single product in every sum.  Every form must give the same bits, and the
    oracle's e4m3 table the same values."""
    ft = ftlib
    H = I = 256
    p = 37
    wtype = synth.W_FP8
    L = ft.ft_expert_layout_get(wtype, H, I)
    S = int(L.bytes)
    rec = np.zeros(S, dtype=np.uint8)
    codes = np.arange(256, dtype=np.uint8)
    codes[[0x7F, 0xFF]] = 0                                   # the two NaN bytes
    gate = np.zeros((I, H), dtype=np.uint8)
    gate[:, p] = codes
    up = np.zeros((I, H), dtype=np.uint8)
    up[:, p] = 0x38                                           # e4m3 1.0
    down = np.zeros((H, I), dtype=np.uint8)
    down[np.arange(H), np.arange(I)] = 0x38
    for m, mat in enumerate((gate, up, down)):
        o = int(L.off_val[m])
        rec[o:o + mat.size] = mat.reshape(-1)
        ns = mat.shape[0] * (mat.shape[1] // 128)
        so = int(L.off_scale[m])
        rec[so:so + 4 * ns] = np.ones(ns, dtype=np.float32).view(np.uint8)
    pool = torch.from_numpy(rec.copy())
    x = torch.zeros(1, H, dtype=torch.bfloat16)
    x[0, p] = 1.0
    idx = torch.zeros(1, 1, dtype=torch.int32)
    w = torch.ones(1, 1)
    ext = torch.ones(1, dtype=torch.int32)
    outs = {}
    forms = available_forms(ft)
    prev = ft.ft_debug_host_simd(-1)
    cpu = ft.CpuExperts(threads=2)
    try:
        for f in forms:
            ft.ft_debug_host_simd(f)
            part = torch.full((1, H), float("nan"))
            cpu.run(cpu.job(pool.data_ptr(), S, wtype, H, I, 1, 0, x, 1, 1, idx, w, ext, part))
            outs[f] = part.numpy().copy()
    finally:
        ft.ft_debug_host_simd(prev)
        cpu.destroy()
    for f in forms[1:]:
        assert np.array_equal(outs[f].view(np.uint32), outs[0].view(np.uint32)), ft.HOST_FORMS[f]
    g = formats.E4M3_TABLE[codes]
    ref = g / (1.0 + np.exp(-g))
    np.testing.assert_allclose(outs[0][0], ref, rtol=1e-6, atol=1e-30)


@pytest.mark.parametrize("threads", [1, 5, 12])
def test_cpu_executor_pool_repeats_bitwise(ftlib, threads):
    """The thread pool under many back-to-back and spaced jobs of different sizes
    (loops of one task run inline, larger ones on every worker), with more
    workers than this machine may have cores: every repeat of a job gives the
    same bytes, and handles are created and destroyed while idle workers spin."""
    import time
    ft = ftlib
    H, I, E, k = 256, 128, 6, 2
    wtype = synth.W_BF16
    cfg = synth.MoEConfig("pool", H, E, k, I, 1, wtype, "bf16", seed=90)
    L = ft.ft_expert_layout_get(wtype, H, I)
    S = int(L.bytes)
    pool = torch.zeros(E * S, dtype=torch.uint8)
    for e in range(E):
        ft.pack_expert(synth.expert_weights(cfg, 0, e, "cpu"), wtype, L, pool[e * S:(e + 1) * S])
    jobs = []
    for T in (1, 3, 8):
        idx = torch.tensor([[(t + j) % E for j in range(k)] for t in range(T)], dtype=torch.int32)
        w = torch.full((T, k), 0.5)
        ext = torch.ones(E, dtype=torch.int32)
        jobs.append((T, idx, w, ext, synth.activations(cfg, T, tag=T)))
    for rnd in range(3):
        cpu = ft.CpuExperts(threads=threads)
        first = {}
        for it in range(40):
            T, idx, w, ext, x = jobs[it % 3]
            part = torch.empty(T, H)
            cpu.run(cpu.job(pool.data_ptr(), S, wtype, H, I, E, 0, x, T, k, idx, w, ext, part))
            if T not in first:
                first[T] = part.clone()
            else:
                assert torch.equal(part, first[T])
            if it % 10 == 9:
                time.sleep(0.002)                 # let the workers fall asleep
        cpu.destroy()


def test_cpu_executor_empty_jobs(ftlib, host_form):
    """No tokens, and tokens with no external expert: nothing to evaluate, the
    partial is all zeros (and nothing is written for T = 0)."""
    ft = ftlib
    H, I, E, k = 256, 128, 4, 2
    wtype = synth.W_MXFP4
    L = ft.ft_expert_layout_get(wtype, H, I)
    S = int(L.bytes)
    pool = torch.zeros(E * S, dtype=torch.uint8)
    cpu = ft.CpuExperts(threads=3)
    x0 = torch.zeros(0, H, dtype=torch.bfloat16)
    i0 = torch.zeros(0, k, dtype=torch.int32)
    p0 = torch.zeros(0, H)
    cpu.run(cpu.job(pool.data_ptr(), S, wtype, H, I, E, 0, x0, 0, k, i0, torch.zeros(0, k),
                    torch.ones(E, dtype=torch.int32), p0))
    T = 5
    x = torch.ones(T, H, dtype=torch.bfloat16)
    idx = torch.tensor([[0, 1]] * T, dtype=torch.int32)
    part = torch.full((T, H), float("nan"))
    cpu.run(cpu.job(pool.data_ptr(), S, wtype, H, I, E, 0, x, T, k, idx, torch.ones(T, k),
                    torch.tensor([0, 0, 1, 1], dtype=torch.int32), part))
    assert torch.equal(part, torch.zeros(T, H))
    cpu.destroy()


def test_host_records_decode_to_finite_weights(ftlib):
    """The host executor case's stand-in records hold in-range values and scales: the
    executor's output over them is finite for every format."""
    import bench
    ft = ftlib
    H, I, n, k = 256, 128, 4, 2
    cpu = ft.CpuExperts(threads=2)
    try:
        for wt in (synth.W_BF16, synth.W_FP8, synth.W_NVFP4, synth.W_MXFP4):
            pool, S, payload = bench.host_records(ft, wt, H, I, n)
            assert pool.numel() == n * S and payload <= S
            idx = torch.arange(n, dtype=torch.int32).reshape(n // k, k)
            part = torch.full((n // k, H), float("nan"))
            x = torch.randn(n // k, H).to(torch.bfloat16)
            cpu.run(cpu.job(pool.data_ptr(), S, wt, H, I, n, 0, x, n // k, k, idx, torch.full((n // k, k), 0.5),
                            torch.ones(n, dtype=torch.int32), part))
            assert torch.isfinite(part).all() and part.abs().max() > 0
    finally:
        cpu.destroy()
