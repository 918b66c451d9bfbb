"""Expert pool setup and the per-layer call sequence over libft.

``ExpertPool`` owns the pinned host pool (all experts of ``n_phys_layers``
layers as records, row l*E + e) and writes synthetic weights into it.
``MoELayer`` owns the per-step device buffers and issues the libft calls of
one MoE layer step in order:

    ft_router_logits -> ft_route -> ft_permute -> [ft_cache_step per wave ->
    ft_expert_grouped] -> ft_combine

or, with a fill stream, per wave: ft_cache_step_split -> ft_expert_grouped
(hits, while the fill copies) -> ft_cache_fill_join -> ft_expert_grouped
(the filled experts).

Nothing here computes: it allocates buffers and sequences the C calls.
"""
from __future__ import annotations

import time
from typing import Optional

import torch

from . import (FT_ROUTE_ARRIVAL_WORDS, FT_TC_WIDE_ASSIGNMENTS, FT_W_BF16, FT_W_F32, FT_W_FP8E4M3, FT_W_MXFP4, FT_W_NVFP4, Cache,
               CpuExperts, PinnedBuffer, RegisteredBuffer, ft_combine, ft_pool_read,
               ft_expert_grouped, ft_expert_grouped_workspace, ft_expert_layout_get, ft_permute, ft_route,
               ft_route_fused, ft_router_logits)


# Decode batches of at least this many assignments (T*k) evaluate their hits
# while the miss fill copies (ft_cache_step_split); smaller batches take
# ft_cache_step.  The split form adds a second expert call after the fill, and
# only layer steps with a fill gain from it.  Measured on B300 per batch size
# (tokens/s, plain -> split):
#   BF16, 40 layers, H=2048, I=512, k=8: T=1 186 -> 174, T=4 504 -> 498,
#     T=16 1364 -> 1435, T=64 4270 -> 4655;
#   NVFP4, 43 layers, H=4096, I=2048, k=6: T=1 61.5 -> 64.3, T=4 139 -> 160;
#   MXFP4, 4 layers, H=6144, I=2048, k=8, T=1: 2-6% more with the split form.
# (The FP4 figures were taken with the exact bf16 expansion of the weights.)  An
# FP4 record is 2.25x to 3.2x the bytes of a bf16 one of the same hidden size, so
# its hits cover the extra call already at T=1.
SPLIT_MIN_ASSIGNMENTS = {FT_W_F32: 64, FT_W_BF16: 64, FT_W_FP8E4M3: 64, FT_W_NVFP4: 1, FT_W_MXFP4: 1}
# Batches on the large-batch tensor-core tiling (prefill waves) take
# ft_cache_step too: beside those kernels, which fill every SM, the fill's
# reads wait behind theirs and the copy slowed to a third of the link.
SPLIT_MAX_ASSIGNMENTS = FT_TC_WIDE_ASSIGNMENTS


def split_pays(T: int, k: int, wtype: int, min_assignments: int = 0) -> bool:
    """Whether a cached layer step of T tokens should use the split form."""
    lo = min_assignments or SPLIT_MIN_ASSIGNMENTS[wtype]
    return lo <= T * k < SPLIT_MAX_ASSIGNMENTS


def pack_expert(comps: dict, wtype: int, layout, out: torch.Tensor) -> None:
    """Writes one expert's stored components into a record (uint8 tensor of S bytes)."""
    out.zero_()
    for m, name in enumerate(("gate", "up", "down")):
        c = comps[name]
        vals = c["w"] if wtype in (FT_W_F32, FT_W_BF16) else c["codes"]
        vb = vals.contiguous().view(torch.uint8).reshape(-1)
        o = layout.off_val[m]
        out[o:o + vb.numel()].copy_(vb)
        if wtype in (FT_W_FP8E4M3, FT_W_NVFP4, FT_W_MXFP4):
            sb = c["scales"].contiguous().view(torch.uint8).reshape(-1)
            o = layout.off_scale[m]
            out[o:o + sb.numel()].copy_(sb)
    if wtype == FT_W_NVFP4:
        g = torch.tensor([comps[n]["gscale"] for n in ("gate", "up", "down")], dtype=torch.float32)
        o = layout.off_gscale
        out[o:o + 12].copy_(g.view(torch.uint8).to(out.device))


class ExpertPool:
    """Pinned host pool of expert records for ``n_phys_layers`` layers of a config.

    Built empty and pinned (``ExpertPool(cfg, n)``, then ``fill``), or from a
    pool file with ``ExpertPool.load`` (read first, pinned afterwards by
    default).  ``setup_s`` records the setup phases in seconds."""

    def __init__(self, cfg, n_phys_layers: int, _buf=None):
        self.cfg = cfg
        self.n_phys = n_phys_layers
        self.layout = ft_expert_layout_get(cfg.wtype, cfg.hidden, cfg.inter)
        self.S = int(self.layout.bytes)
        self.E = cfg.n_experts
        self.setup_s = {}
        if _buf is None:
            t0 = time.perf_counter()
            _buf = PinnedBuffer(self.n_phys * self.E * self.S)
            self.setup_s["alloc_pinned"] = time.perf_counter() - t0
        self.buf = _buf
        self.host = self.buf.tensor

    @property
    def nbytes(self) -> int:
        return self.n_phys * self.E * self.S

    @classmethod
    def load(cls, cfg, n_phys_layers: int, path: str, read_then_pin: bool = True, threads: int = 0):
        """A pool read from a pool file (records in row order l*E + e, as ``save`` writes them).

        read_then_pin: the records are read into fresh pageable memory, which the
        read itself faults in, and the filled buffer is pinned afterwards
        (ft_pool_read, then ft_host_register).  Otherwise the pool is pinned
        first (ft_host_alloc) and the file read into the pinned pages."""
        layout = ft_expert_layout_get(cfg.wtype, cfg.hidden, cfg.inter)
        n = n_phys_layers * cfg.n_experts * int(layout.bytes)
        times = {}
        t0 = time.perf_counter()
        if read_then_pin:
            buf = RegisteredBuffer(n)
            t1 = time.perf_counter()
            buf.read(path, 0, threads)
            t2 = time.perf_counter()
            buf.pin()
            t3 = time.perf_counter()
            times = {"alloc_pageable": t1 - t0, "read": t2 - t1, "pin": t3 - t2}
        else:
            buf = PinnedBuffer(n)
            t1 = time.perf_counter()
            ft_pool_read(path, 0, buf.ptr, n, threads)
            t2 = time.perf_counter()
            times = {"alloc_pinned": t1 - t0, "read": t2 - t1}
        pool = cls(cfg, n_phys_layers, _buf=buf)
        pool.setup_s = times
        return pool

    def save(self, path: str) -> None:
        """Writes the pool's records, in row order, to a pool file."""
        with open(path, "wb") as f:
            f.write(memoryview(self.host.numpy()))

    @property
    def ptr(self) -> int:
        return self.buf.ptr

    def row(self, phys_layer: int, expert: int) -> torch.Tensor:
        o = (phys_layer * self.E + expert) * self.S
        return self.host[o:o + self.S]

    def fill(self, device="cuda", layers=None) -> None:
        """Generates every expert with ``synth`` on ``device`` and copies each layer into the pool."""
        import synth
        staging = torch.empty(self.E * self.S, dtype=torch.uint8, device=device)
        for l in (range(self.n_phys) if layers is None else layers):
            for e in range(self.E):
                rec = staging[e * self.S:(e + 1) * self.S]
                pack_expert(synth.expert_weights(self.cfg, l, e, device), self.cfg.wtype, self.layout, rec)
            o = l * self.E * self.S
            self.host[o:o + self.E * self.S].copy_(staging, non_blocking=False)
        del staging

    def free(self):
        self.buf.free()


class MoELayer:
    """Per-step device buffers for batches of up to ``T_max`` tokens, and the call sequence."""

    def __init__(self, cfg, T_max: int, device="cuda"):
        self.cfg = cfg
        E, k, H, I = cfg.n_experts, cfg.top_k, cfg.hidden, cfg.inter
        self.T_max = T_max
        i32 = dict(dtype=torch.int32, device=device)
        f32 = dict(dtype=torch.float32, device=device)
        self.logits = torch.empty(T_max, E, **f32)
        self.idx = torch.empty(T_max, k, **i32)
        self.w = torch.empty(T_max, k, **f32)
        self.counts = torch.empty(E, **i32)
        self.offsets = torch.empty(E + 1, **i32)
        self.perm = torch.empty(T_max * k, **i32)
        self.inv = torch.empty(T_max * k, **i32)
        self.arrivals = torch.zeros(FT_ROUTE_ARRIVAL_WORDS, **i32)   # ft_route_fused's counters, kept zero
        self.slot_of = torch.empty(E, **i32)
        self.slot_fill = torch.empty(E, **i32)
        self.ext = torch.zeros(E, **i32)
        self.step_counts = torch.zeros(4, **i32)
        self.y = torch.empty(T_max * k, H, **f32)
        self.out = torch.empty(T_max, H, **f32)
        ws = ft_expert_grouped_workspace(T_max, k, H, I)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=device)

    def route(self, x, w_router, bias, stream=None):
        """Router logits, top-k and permutation (one launch for decode batches: ft_route_fused)."""
        T = x.shape[0]
        ft_route_fused(x, w_router, bias, self.cfg.top_k, self.logits[:T], self.idx[:T], self.w[:T], self.counts,
                       self.offsets, self.perm, self.inv, self.arrivals, stream)

    def route_unfused(self, x, w_router, bias, stream=None):
        """The same as ``route`` with the three separate kernels."""
        T = x.shape[0]
        ft_router_logits(x, w_router, bias, self.logits[:T], stream)
        ft_route(self.logits[:T], self.cfg.top_k, self.idx[:T], self.w[:T], stream)
        ft_permute(self.idx[:T], self.cfg.n_experts, self.counts, self.offsets, self.perm, self.inv, stream)

    def experts(self, x, slot_of, slot_pool, slot_bytes, pool_slots, stream=None):
        ft_expert_grouped(x, self.cfg.top_k, self.cfg.inter, self.cfg.n_experts, self.cfg.wtype, self.perm,
                          self.offsets, slot_of, slot_pool, slot_bytes, pool_slots,
                          self.y[: x.shape[0] * self.cfg.top_k], self.workspace, stream)

    def combine(self, T, ext_flags=None, ext_partial=None, stream=None):
        ft_combine(self.y[: T * self.cfg.top_k], self.inv, self.idx[:T], self.w[:T], ext_flags, ext_partial,
                   self.cfg.n_experts, self.out[:T], stream)
        return self.out[:T]

    def cached_wave(self, x, layer: int, cache: Cache, slot_bytes: int, fill_ratio: float, wave: int,
                    step_counts=None, stream=None, fill_stream=None, after_control=None):
        """Cache control, miss fill and expert evaluation of one wave.

        With ``fill_stream`` the fill runs there while the hits are evaluated on
        ``stream``; the filled experts follow after the join.  ``after_control``
        (split form only) is called right after the control launch, before the
        hits' evaluation: the point from which the wave's external set is known."""
        sc = self.step_counts if step_counts is None else step_counts
        if fill_stream is None:
            assert after_control is None, "the host branch needs the split form"
            cache.step(layer, self.counts, fill_ratio, wave, self.slot_of, self.ext, sc, stream)
            self.experts(x, self.slot_of, cache.slot_pool, slot_bytes, cache.max_slots, stream)
            return
        cache.step_split(layer, self.counts, fill_ratio, wave, self.slot_of, self.slot_fill, self.ext, sc, stream,
                         fill_stream)
        if after_control is not None:
            after_control()
        self.experts(x, self.slot_of, cache.slot_pool, slot_bytes, cache.max_slots, stream)
        cache.fill_join(stream)
        self.experts(x, self.slot_fill, cache.slot_pool, slot_bytes, cache.max_slots, stream)

    def forward_cached(self, x, w_router, bias, layer: int, cache: Cache, slot_bytes: int,
                       fill_ratio: float = 1.0, ext_partial: Optional[torch.Tensor] = None, stream=None,
                       fill_stream=None):
        """One layer step over the LRU cache (all waves), returning out [T, H] fp32."""
        T = x.shape[0]
        self.route(x, w_router, bias, stream)
        for wv in range(cache.n_waves()):
            self.cached_wave(x, layer, cache, slot_bytes, fill_ratio, wv, None, stream, fill_stream)
        return self.combine(T, self.ext, ext_partial, stream)

    def forward_slots(self, x, w_router, bias, slot_of, slot_pool, slot_bytes, pool_slots, stream=None):
        """One layer step with every expert already resident at slot_of[e] (streaming, fused mode)."""
        T = x.shape[0]
        self.route(x, w_router, bias, stream)
        self.experts(x, slot_of, slot_pool, slot_bytes, pool_slots, stream)
        return self.combine(T, None, None, stream)


class HostBranch:
    """The external experts of a layer step evaluated on the host (the CPU branch).

    After the last wave's control launch, a side stream copies the step's
    external marks, routing and tokens to pinned host buffers, runs the host
    expert executor on them as a host function (a host node when captured),
    and copies the partial output back to the device; ``P`` is then the
    ``ext_partial`` of the combine, which waits for ``done``.  The fill and the
    GPU experts run meanwhile.  Each layer's job is kept by the executor, so a
    captured step enqueues it once and every replay runs it again."""

    def __init__(self, cfg, T_max: int, pool: "ExpertPool", cpu: CpuExperts, device="cuda"):
        self.cfg, self.pool, self.cpu, self.T_max = cfg, pool, cpu, T_max
        H, k, E = cfg.hidden, cfg.top_k, cfg.n_experts
        xdt = torch.bfloat16 if cfg.x_dtype == "bf16" else torch.float32
        self.x_h = torch.empty(T_max, H, dtype=xdt).pin_memory()
        self.idx_h = torch.empty(T_max, k, dtype=torch.int32).pin_memory()
        self.w_h = torch.empty(T_max, k, dtype=torch.float32).pin_memory()
        self.ext_h = torch.empty(E, dtype=torch.int32).pin_memory()
        self.part_h = torch.empty(T_max, H, dtype=torch.float32).pin_memory()
        self.P = torch.zeros(T_max, H, dtype=torch.float32, device=device)
        self.stream = torch.cuda.Stream(device=device)
        self.done = torch.cuda.Event()

    def launch(self, lay: MoELayer, x, layer: int):
        """Issues the branch for layer ``layer`` of the current step (tokens x on the device)."""
        T = x.shape[0]
        cur = torch.cuda.current_stream()
        self.stream.wait_stream(cur)
        with torch.cuda.stream(self.stream):
            self.x_h[:T].copy_(x, non_blocking=True)
            self.idx_h[:T].copy_(lay.idx[:T], non_blocking=True)
            self.w_h[:T].copy_(lay.w[:T], non_blocking=True)
            self.ext_h.copy_(lay.ext, non_blocking=True)
            job = self.cpu.job(self.pool.ptr, self.pool.S, self.cfg.wtype, self.cfg.hidden, self.cfg.inter,
                               self.cfg.n_experts, layer % self.pool.n_phys, self.x_h[:T], T, self.cfg.top_k,
                               self.idx_h[:T], self.w_h[:T], self.ext_h, self.part_h[:T])
            self.cpu.enqueue(job, self.stream)
            self.P[:T].copy_(self.part_h[:T], non_blocking=True)
            self.done.record(self.stream)

    def join(self):
        torch.cuda.current_stream().wait_event(self.done)
