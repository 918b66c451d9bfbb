#!/usr/bin/env python
"""MoE-layer tokens/s over the slot-pool expert cache, and % of the layer roofline.

Workload (one GPU): the 40-layer BF16 MoE stack (hidden 2048, 256 experts,
top-8, SwiGLU intermediate 512, weights N(0, 0.02)), whose 10,240 experts
(64.4 GB) sit in pinned host memory.  One step is one pass of the decode
trace: at each batch size T = 1, 4, 16, 64, 256 decode steps of every layer
(T independent AR(1) chains h_t = 0.9 h_{t-1} + 0.436 N(0,1), Zipf(1.1) router
prior) over an LRU expert cache holding 40% of the (layer, expert) slots
(4096 slots), starting from an empty cache, so the cold start is counted.
Further legs: prefill chunks streamed through two whole-layer buffers
(double-buffered and serialized), pool setup pin-first vs read-then-pin, the
NVFP4 stack and the MXFP4 mixed trace.

Output: one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

BATCHES = (1, 4, 16, 64)

# DRAM traffic per algorithmic byte, from one ncu capture of each kernel
# (dram__bytes_read.sum + dram__bytes_write.sum over the algorithmic bytes of the
# same launch: the 32-expert fill case, and the 64-token bf16 expert call).  The
# bench scales these to its own launches and labels the result as scaled.  The
# fill's reads come over the host link, so its DRAM traffic is the writes of the
# filled experts that reached DRAM before the launch ended.
TRAFFIC_PER_BYTE = {"fill": (0.073e6 + 140.229e6) / 201.327e6,
                    "experts": (207.776e6 + 3.545e6 + 103.355e6 + 2.734e6) / (205.5e6 + 0.5e6 + 102.8e6)}
CACHE_FRAC = 0.40
ROUTE_FUSED_MAX_T = 8             # batches routed by one ft_route_fused launch
CC_MAX_ASSIGNMENTS = 8            # FT_CC_MAX_ASSIGNMENTS: bf16 experts of one token run on the CUDA cores
FP4_OVER_BF16 = 13.5 / 2.25       # nominal dense FP4 / bf16 tensor rates of the B300
METRIC = "MoE-layer tokens/s (decode T=1..64, prefill 8192) and % of layer roofline"
WORKLOAD = ("decode_bf16_40L: H=2048 E=256 top-8 I=512, bf16 weights, 40 layers, 64.4 GB pinned host pool, "
            "LRU cache of 40% (4096 slots), 256-step AR(1)+Zipf(1.1) decode trace at T=1,4,16,64, each from a "
            "cold cache")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2, help="timed passes of the whole decode trace")
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--phys-layers", type=int, default=0, help="host pool layers (0: all 40 when RAM allows)")
    p.add_argument("--batches", default=",".join(map(str, BATCHES)))
    p.add_argument("--prompts", default="4096,8192,16384", help="prefill prompt lengths (chunks of <= 8192)")
    p.add_argument("--no-prefill", action="store_true")
    p.add_argument("--no-fp4", action="store_true", help="skip the NVFP4 stack and the MXFP4 mixed-trace legs")
    p.add_argument("--fp4-steps", type=int, default=24, help="decode steps per batch size from a cold cache, NVFP4 stack")
    p.add_argument("--trace-steps", type=int, default=256, help="decode steps of the trace per batch size")
    p.add_argument("--steady-from", type=int, default=32, help="first step of the steady-state figures")
    p.add_argument("--cpu-tokens", type=int, default=2, help="T=1 tokens per round of the CPU oracle baseline")
    p.add_argument("--cpu-budget-s", type=float, default=12.0, help="wall seconds of timed CPU baseline rounds")
    p.add_argument("--no-pool-setup", action="store_true", help="skip the pin-first vs read-then-pin setup leg")
    p.add_argument("--no-placement", action="store_true", help="skip the placement-policy replay")
    p.add_argument("--profile-eager-steps", type=int, default=0,
                   help="after the timed region: per batch size, the trace's last N steps again, eagerly (no graphs), "
                        "inside the NVTX range profile_steps (for an ncu launch list; 0: none)")
    p.add_argument("--timed-spans", action="store_true",
                   help="record the per-kernel timing events inside the timed passes (instead of one extra pass)")
    p.add_argument("--setup-layers", type=int, default=2, help="layers of the pool file in the setup leg")
    p.add_argument("--mixed-decode-steps", type=int, default=512)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--split-min-assignments", type=int, default=0,
                   help="smallest decode batch T*k for the split form, every format (0: the policy per format)")
    p.add_argument("--fill-blocks", type=int, default=0,
                   help="blocks of the decode stack's fill launch (0: the library's default)")
    p.add_argument("--no-split-fill", action="store_true",
                   help="decode with ft_cache_step (fill, then all experts) instead of the split form "
                        "(hits evaluated while the fill copies)")
    p.add_argument("--kernel-case", default="", choices=["", "experts_decode", "experts_prefill", "fill",
                                                         "fill_overlap", "route", "host_experts"],
                   help="time one expert-kernel case on a small resident pool (profiling aid; prints its own line)")
    p.add_argument("--reps", type=int, default=5)
    p.add_argument("--fp4-path", default="block_scaled", choices=["block_scaled", "expand"],
                   help="small-batch NVFP4/MXFP4 experts: block-scaled FP4 MMA, or exact expansion to bf16")
    p.add_argument("--case-config", default="", help="workload of --kernel-case (a synth config name)")
    p.add_argument("--case-experts", type=int, default=0,
                   help="experts per layer of --kernel-case (0: the config's; fewer keep a profiled pool small)")
    return p.parse_args()


def log(msg: str) -> None:
    """Phase marker on stderr (the JSON line goes to stdout)."""
    sys.stderr.write(f"[bench {time.strftime('%H:%M:%S')}] {msg}\n")
    sys.stderr.flush()


# ---------------------------------------------------------------- distributed plumbing

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        if torch.cuda.is_available():
            torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _reduce(world, v: float, op_name: str) -> float:
    """All-reduce of one float over the ranks (device tensor for NCCL, host tensor for gloo)."""
    if world == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=getattr(dist.ReduceOp, op_name))
    return float(t.item())


def max_over_ranks(world, v: float) -> float:
    """The slowest rank's time: the job takes as long as its slowest replica."""
    return _reduce(world, v, "MAX")


def sum_over_ranks(world, v: float) -> float:
    """Work summed over the replicas (each rank runs its own traces)."""
    return _reduce(world, v, "SUM")


# ---------------------------------------------------------------- measurement helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                       "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        self.f.seek(0)
        sm, smax, reasons, n = [], None, set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f.read().strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            n += 1
            for nm, v in zip(names, parts[5:9]):
                if v.lower() in ("active", "1"):
                    reasons.add(nm)
        self.f.close()
        os.unlink(self.f.name)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": n}


def link_peak_gbs(pool_host: torch.Tensor, nbytes: int, dev) -> float:
    """Best of three pinned host -> device cudaMemcpyAsync of one whole layer."""
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    best = 0.0
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        d.copy_(pool_host[:nbytes], non_blocking=True)
        e1.record()
        e1.synchronize()
        best = max(best, nbytes / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    del d
    return best


def host_ram_bytes() -> int:
    with open("/proc/meminfo") as f:
        for line in f:
            if line.startswith("MemAvailable"):
                return int(line.split()[1]) * 1024
    return 0


# ---------------------------------------------------------------- the decode workload

class DecodeRun:
    """The decode trace of one stacked workload, every batch size from a cold cache.

    For each batch size T: ``n_steps`` decode steps of all layers (T independent
    AR(1) chains, inputs resident on the device), starting from an empty cache
    ([Review] §2.7: no warm-up, the first request meets a cold cache).  One slot
    pool and one cache handle serve the batch sizes in turn: ``ft_cache_reset``
    empties the cache before each.  Every (T, step) is one CUDA graph, captured
    once and replayed in every pass; its layer outputs go to a per-T device
    buffer, and its per-wave cache counters to a per-step record."""

    def __init__(self, ft, cfg, pool, routers, batches, n_steps, dev, n_slots, split_min=0, e2e=False,
                 fill_blocks=0):
        self.ft, self.cfg, self.pool, self.routers = ft, cfg, pool, routers
        self.batches, self.n_steps, self.dev = list(batches), n_steps, dev
        L, E, H = cfg.n_layers, cfg.n_experts, cfg.hidden
        self.S, self.n_slots = pool.S, n_slots
        self.sp = torch.empty(n_slots * pool.S, dtype=torch.uint8, device=dev)
        self.cache = ft.Cache(L, E, pool.n_phys, n_slots, n_slots, pool.S, pool.ptr, self.sp)
        if fill_blocks > 0:
            self.cache.set_fill_blocks(fill_blocks)
        self.n_waves = self.cache.n_waves()
        self.fs = torch.cuda.Stream(device=dev)
        self.b = {}
        for T in self.batches:
            tr = synth.AR1Trace(cfg, T, dev, tag=T)
            d = {"layer": ft.MoELayer(cfg, T, dev),
                 "split": split_min >= 0 and ft.split_pays(T, cfg.top_k, cfg.wtype, split_min),
                 "xs": torch.stack([tr.next() for _ in range(n_steps)]),                 # [steps, T, H] resident
                 "hist": torch.zeros(n_steps, L, self.n_waves, 4, dtype=torch.int32, device=dev),
                 "outs": torch.empty(L, T, H, dtype=torch.float32, device=dev)}
            if e2e:
                d["x_host"] = torch.empty(n_steps, T, H, dtype=d["xs"].dtype).pin_memory()
                d["x_host"].copy_(d["xs"].cpu())
                d["out_host"] = torch.empty(L, T, H, dtype=torch.float32).pin_memory()
            self.b[T] = d
        self.graphs, self.igraphs = {}, {}

    def launches_per_step(self, T) -> int:
        # routing (one fused launch, or router_logits + route + permute), (control, fill, expert
        # kernels) per wave, combine;
        # bf16 experts run gather + gate/up + down on the tensor cores (gate/up + down on the CUDA
        # cores for one token), other formats gate/up + down
        # (the split form evaluates hits and filled experts in two expert calls)
        if self.cfg.wtype == synth.W_BF16:
            n_exp = 2 if T * self.cfg.top_k <= CC_MAX_ASSIGNMENTS else 3
        else:
            n_exp = 2
        if self.b[T]["split"]:
            n_exp *= 2
        n_route = 1 if T <= ROUTE_FUSED_MAX_T else 3       # ft_route_fused: one grid launch up to 8 tokens
        return self.cfg.n_layers * (n_route + (2 + n_exp) * self.n_waves + 1)

    def launches_per_pass(self) -> int:
        return sum(self.n_steps * self.launches_per_step(T) for T in self.batches)

    def step(self, T, t, ev=None):
        """Decode step t of batch size T through every layer (eager, or recorded under capture)."""
        ft, cfg, d = self.ft, self.cfg, self.b[T]
        lay, cache, x = d["layer"], self.cache, d["xs"][t]
        fs = self.fs if d["split"] else None
        k, S, N = cfg.top_k, self.S, self.n_slots
        for l in range(cfg.n_layers):
            lay.route(x, *self.routers[l])
            for w in range(self.n_waves):
                sc = d["hist"][t, l, w]
                if ev is not None:
                    ev.rec("cache")
                if fs is None:
                    cache.step(l, lay.counts, 1.0, w, lay.slot_of, lay.ext, sc)
                    if ev is not None:
                        ev.rec("fill_end")
                    lay.experts(x, lay.slot_of, self.sp, S, N)
                    if ev is not None:
                        ev.rec("expert_end")
                    continue
                cache.step_split(l, lay.counts, 1.0, w, lay.slot_of, lay.slot_fill, lay.ext, sc, fill_stream=fs)
                if ev is not None:
                    ev.rec("ctrl_end")
                    ev.rec("fill_end", fs)
                lay.experts(x, lay.slot_of, self.sp, S, N)          # hits, during the fill
                if ev is not None:
                    ev.rec("hit_end")
                cache.fill_join()
                if ev is not None:
                    torch.cuda.current_stream().wait_stream(fs)     # joins the timing event too
                    ev.rec("join")
                lay.experts(x, lay.slot_fill, self.sp, S, N)        # the filled experts
                if ev is not None:
                    ev.rec("expert_end")
            ft.ft_combine(lay.y[: T * k], lay.inv, lay.idx[:T], lay.w[:T], lay.ext, None, cfg.n_experts,
                          d["outs"][l])

    def capture(self, instrumented=False):
        """One eager step per batch size (kernel attributes and modules set up outside capture),
        a cold reset, then one graph per (T, step).  ``instrumented`` graphs also record timing
        events around the cache step and the expert calls (event-record nodes, kept in the
        graph's EventLog); they go to a second set, since an event node between two launches
        stops the second from launching early, which the plain graphs keep."""
        for T in self.batches:
            self.step(T, 0)
        torch.cuda.synchronize()
        self.cache.reset()
        dst = self.igraphs if instrumented else self.graphs
        for T in self.batches:
            for t in range(self.n_steps):
                g = torch.cuda.CUDAGraph()
                ev = EventLog(external=True) if instrumented else None
                with torch.cuda.graph(g):
                    self.step(T, t, ev)
                dst[(T, t)] = (g, ev)
        torch.cuda.synchronize()

    def run_pass(self, marks=None, e2e=False, instrumented=False):
        """The whole trace once: per batch size, a cold reset and every step's graph.

        ``marks`` (a list) receives (T, t, event) before each step and (T, -1,
        event) after each batch size's last step.  With ``e2e`` each step's input is first copied from
        pinned host memory and every layer's output copied back to it."""
        graphs = self.igraphs if instrumented else self.graphs
        for T in self.batches:
            d = self.b[T]
            self.cache.reset()                      # cold start (synchronises)
            for t in range(self.n_steps):
                if e2e:
                    d["xs"][t].copy_(d["x_host"][t], non_blocking=True)
                if marks is not None:
                    e = torch.cuda.Event(enable_timing=True)
                    e.record()
                    marks.append((T, t, e))
                graphs[(T, t)][0].replay()
                if e2e:
                    d["out_host"].copy_(d["outs"], non_blocking=True)
            if marks is not None:
                e = torch.cuda.Event(enable_timing=True)
                e.record()
                marks.append((T, -1, e))

    def hist(self, T) -> np.ndarray:
        """Per (step, layer, wave) {experts, hits, fills, externals} of the last pass."""
        return self.b[T]["hist"].cpu().numpy()

    def logs(self, T, t0=0):
        """EventLogs of the instrumented graphs (their last replay)."""
        return [self.igraphs[(T, t)][1] for t in range(t0, self.n_steps)]

    def release(self):
        self.graphs.clear()
        self.igraphs.clear()
        torch.cuda.synchronize()
        self.cache.destroy()


def profile_eager(run, n):
    """Per batch size: the trace from a cold cache through its graphs up to its last n steps,
    then those n steps eagerly inside the NVTX range "profile_steps" (a warm cache, launches
    that a profiler can list one by one)."""
    for T in run.batches:
        run.cache.reset()
        for t in range(run.n_steps - n):
            run.graphs[(T, t)][0].replay()
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("profile_steps")
        for t in range(run.n_steps - n, run.n_steps):
            run.step(T, t)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()


def step_times_ms(marks):
    """{T: [ms of each step]} from the events recorded before each step and after each T's last."""
    out = {}
    for i in range(len(marks) - 1):
        T, t, e = marks[i]
        if t >= 0:
            out.setdefault(T, []).append(e.elapsed_time(marks[i + 1][2]))
    return out


class EventLog:
    """CUDA events recorded on the launching (current) stream, in order.

    With ``external`` the events become event-record nodes when recorded under
    graph capture, so each replay of the graph records them again."""

    def __init__(self, external=False):
        self.ev = []
        self.external = external

    def rec(self, tag, stream=None):
        e = torch.cuda.Event(enable_timing=True, external=self.external)
        e.record(stream)
        self.ev.append((tag, e))

    def spans(self, start_tag, end_tag):
        """Each start_tag event to the next end_tag event after it."""
        out = []
        for i, (tag, e) in enumerate(self.ev):
            if tag == start_tag:
                j = next(j for j in range(i + 1, len(self.ev)) if self.ev[j][0] == end_tag)
                out.append(e.elapsed_time(self.ev[j][1]))
        return out

    def cache_expert_spans(self):
        """Per wave: (control + fill span, expert span).  In the split form the
        expert span is the hits' call plus the filled experts' call after the join."""
        cache = self.spans("cache", "fill_end")
        if any(tag == "hit_end" for tag, _ in self.ev):
            hit, miss = self.spans("ctrl_end", "hit_end"), self.spans("join", "expert_end")
            return cache, [a + b for a, b in zip(hit, miss)]
        return cache, self.spans("fill_end", "expert_end")


def spans_us(logs):
    """Mean CUDA-event spans per wave (us): control + fill, and the expert calls
    (in the split form: the hits' call, which runs beside the fill, and the
    filled experts' call after the join)."""
    def mean(v):
        return 1e3 * sum(v) / max(len(v), 1)
    out = {"control_fill": mean([v for ev in logs for v in ev.spans("cache", "fill_end")])}
    if any(tag == "hit_end" for tag, _ in logs[0].ev):
        out["hits"] = mean([v for ev in logs for v in ev.spans("ctrl_end", "hit_end")])
        out["wait_for_fill"] = mean([v for ev in logs for v in ev.spans("hit_end", "join")])
        out["filled"] = mean([v for ev in logs for v in ev.spans("join", "expert_end")])
    else:
        out["experts"] = mean([v for ev in logs for v in ev.spans("fill_end", "expert_end")])
    return out


def layer_roofline_seconds(hist: np.ndarray, T: int, cfg, S_payload: int, peaks, link_gbs: float):
    """Per layer step: max(FLOPs / tensor peak, HBM bytes / HBM peak, link bytes / link peak), summed."""
    H, E, k, I = cfg.hidden, cfg.n_experts, cfg.top_k, cfg.inter
    hits, fills = hist[..., 1].astype(np.float64), hist[..., 2].astype(np.float64)
    weights = (hits + fills) * S_payload                 # expert weights read once from HBM
    fill_writes = fills * S_payload
    router = E * H * 2
    act = T * H * 2 * 3 + T * k * H * 4 * 2 + T * H * 4 + T * k * I * 4 * 2
    hbm = weights + fill_writes + router + act
    link = fills * S_payload
    flops = 2.0 * T * k * 3 * H * I + 2.0 * T * H * E
    t_hbm = hbm / (peaks["hbm_gbs"] * 1e9)
    t_link = link / (link_gbs * 1e9)
    t_flop = flops / (peaks["bf16_tflops_sustained"] * 1e12)
    t = np.maximum(np.maximum(t_hbm, t_link), t_flop)
    return float(t.sum()), {"hbm_bytes": float(hbm.sum()), "link_bytes": float(link.sum()), "flops": float(flops * hits.size),
                            "bound_layer_steps": {"hbm": int((t == t_hbm).sum()), "link": int((t == t_link).sum()),
                                                  "tensor": int((t == t_flop).sum())}}


# ---------------------------------------------------------------- prefill streaming leg

def prefill_leg(ft, cfg, pool, routers0, dev, prompts, link_gbs, peaks, chunk=8192):
    """Prompts of the given lengths streamed through ft_stream in chunks of at most ``chunk`` tokens.

    For each prompt length: double-buffered and serialized runs; each chunk
    streams every layer once (zero router bias: near-uniform routing)."""
    L, E = cfg.n_layers, cfg.n_experts
    n_slots = 2 * E + 16                      # the two whole-layer buffers (+ a few LRU slots)
    sp = torch.empty(n_slots * pool.S, dtype=torch.uint8, device=dev)
    cache = ft.Cache(L, E, pool.n_phys, n_slots, n_slots, pool.S, pool.ptr, sp)
    lay = ft.MoELayer(cfg, chunk, dev)
    max_chunks = max((p + chunk - 1) // chunk for p in prompts)
    xs = [synth.activations(cfg, chunk, tag=c, device=dev) for c in range(max_chunks)]
    zero = torch.zeros(E, dtype=torch.float32, device=dev)
    slot_of = torch.empty(E, dtype=torch.int32, device=dev)
    res = {"prompts": {}}
    for P in prompts:
        sizes = [min(chunk, P - c0) for c0 in range(0, P, chunk)]
        r = {}
        for mode in ("overlapped", "serialized"):
            st = ft.Stream(cache, serialized=(mode == "serialized"))
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for c, n in enumerate(sizes):
                for l in range(L):
                    nxt = l + 1 if l + 1 < L else (0 if c + 1 < len(sizes) else -1)
                    st.layer(l, nxt, slot_of)
                    lay.forward_slots(xs[c][:n], routers0[l][0], zero, slot_of, sp, pool.S, n_slots)
                    st.layer_done(l)
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            nbytes = st.bytes()
            st.destroy()
            r[mode] = {"tokens_per_s": P / (ms * 1e-3), "ms": ms, "h2d_gbs": nbytes / (ms * 1e-3) / 1e9,
                       "link_frac": nbytes / (ms * 1e-3) / 1e9 / link_gbs}
        r["loss_without_overlap"] = 1.0 - r["serialized"]["tokens_per_s"] / r["overlapped"]["tokens_per_s"]
        res["prompts"][str(P)] = r
    res["overlapped"] = res["prompts"][str(prompts[-1] if chunk not in prompts else chunk)]["overlapped"]
    res["serialized"] = res["prompts"][str(prompts[-1] if chunk not in prompts else chunk)]["serialized"]
    # compute alone (weights resident in a buffer): one 8192-token layer through the grouped experts
    st = ft.Stream(cache)
    st.layer(0, -1, slot_of)
    torch.cuda.synchronize()
    lay.forward_slots(xs[0], routers0[0][0], zero, slot_of, sp, pool.S, n_slots)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 5
    e0.record()
    for _ in range(reps):
        lay.forward_slots(xs[0], routers0[0][0], zero, slot_of, sp, pool.S, n_slots)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    # the expert call alone (ft_expert_grouped on the resident layer), timed the same way
    xq = xs[0]
    e0.record()
    for _ in range(reps):
        lay.experts(xq, slot_of, sp, pool.S, n_slots)
    e1.record()
    torch.cuda.synchronize()
    ms_exp = e0.elapsed_time(e1) / reps
    st.layer_done(0)
    st.destroy()
    Tk, H, I, E_ = chunk * cfg.top_k, cfg.hidden, cfg.inter, cfg.n_experts
    U = int((lay.counts > 0).sum())
    wb = int(ft.ft_expert_layout_get(cfg.wtype, H, I).payload_bytes) / 3.0   # bytes of one weight matrix
    flops_gu, flops_dn = 2.0 * Tk * 2 * H * I, 2.0 * Tk * H * I
    bytes_gu = U * 2 * wb + chunk * H * 2 + Tk * I * 2                         # weights, rows of x, intermediate
    bytes_dn = U * wb + Tk * I * 2 + Tk * H * 4                                # weights, intermediate, fp32 output
    roof_s = (max(flops_gu / (peaks["bf16_tflops"] * 1e12), bytes_gu / (peaks["hbm_gbs"] * 1e9)) +
              max(flops_dn / (peaks["bf16_tflops"] * 1e12), bytes_dn / (peaks["hbm_gbs"] * 1e9)))
    flops = flops_gu + flops_dn
    res["compute_only_ms_per_layer"] = ms
    res["expert_call_ms"] = ms_exp
    res["expert_tflops"] = flops / (ms_exp * 1e-3) / 1e12
    res["expert_tensor_frac_of_bf16"] = res["expert_tflops"] / peaks["bf16_tflops"]
    if cfg.wtype in (synth.W_NVFP4, synth.W_MXFP4):
        # the peak of the weights' own dtype: FP4 dense = bf16 measured x the nominal ratio 13.5 / 2.25
        fp4 = peaks["bf16_tflops"] * FP4_OVER_BF16
        res["expert_tensor_frac_of_fp4"] = res["expert_tflops"] / fp4
        res["fp4_peak_tflops"] = fp4
        res["fp4_peak_source"] = (f"bf16 measured burst x {FP4_OVER_BF16:g} (nominal dense FP4 / bf16); the "
                                  "products run as kind::f16 MMAs on weights expanded exactly to bf16")
    res["expert_roofline_frac"] = roof_s / (ms_exp * 1e-3)
    res["expert_roofline_note"] = ("per product max(FLOPs / bf16 peak, bytes / HBM peak): gate/up and down are "
                                   "both near the ridge (about 256 rows per expert); down writes fp32 output")
    res["loss_without_overlap"] = 1.0 - res["serialized"]["tokens_per_s"] / res["overlapped"]["tokens_per_s"]
    cache.destroy()
    del sp, lay
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------- secondary workloads

def decode_report(run, marks, cfg, peaks, link, payload, steady_from):
    """Per batch size and overall: tokens/s over the whole trace (cold start included) and
    from step ``steady_from`` on, the layer-roofline fractions, hit rates, and the fill and
    expert spans of the captured steps (CUDA events on the launching streams, last pass)."""
    st = step_times_ms(marks)
    per = {}
    acc = {"ms": 0.0, "tok": 0, "roof": 0.0, "ms_s": 0.0, "tok_s": 0, "roof_s": 0.0}
    cache_ms, expert_ms, fills, unique = [], [], 0, 0
    for T in run.batches:
        h = run.hist(T).sum(axis=2)                     # [steps, L, 4], summed over waves
        ms = np.asarray(st[T], dtype=np.float64)
        n = len(ms)
        sf = min(steady_from, n - 1)
        r_all, _ = layer_roofline_seconds(h, T, cfg, payload, peaks, link)
        r_st, _ = layer_roofline_seconds(h[sf:], T, cfg, payload, peaks, link)
        logs = run.logs(T)
        for ev in logs:
            c, e = ev.cache_expert_spans()
            cache_ms += c
            expert_ms += e
        fills += int(h[..., 2].sum())
        unique += int(h[..., 0].sum())
        per[str(T)] = {
            "tokens_per_s": T * n / (ms.sum() * 1e-3), "ms_per_step": float(ms.mean()),
            "first_step_ms": float(ms[0]), "layer_roofline_frac": r_all / (ms.sum() * 1e-3),
            "hit_rate": float(h[..., 1].sum() / max(h[..., 0].sum(), 1)),
            "steady_tokens_per_s": T * (n - sf) / (ms[sf:].sum() * 1e-3),
            "steady_layer_roofline_frac": r_st / (ms[sf:].sum() * 1e-3),
            "steady_hit_rate": float(h[sf:, :, 1].sum() / max(h[sf:, :, 0].sum(), 1)),
            "us_per_wave": spans_us(logs)}
        acc["ms"] += ms.sum()
        acc["tok"] += T * n
        acc["roof"] += r_all
        acc["ms_s"] += ms[sf:].sum()
        acc["tok_s"] += T * (n - sf)
        acc["roof_s"] += r_st
    n_ls = len(cache_ms)
    fill_bytes = fills * payload
    cache_s, expert_s = sum(cache_ms) * 1e-3, sum(expert_ms) * 1e-3
    expert_hbm = unique * payload
    scaled = ("scaled, not measured in this run: DRAM bytes per algorithmic byte from one ncu capture of the "
              "same kernel (profiles/)")
    roof_fill = {"kernel": "ft_cache_step (control + fill launches)", "bound": "link",
                 "achieved": fill_bytes / cache_s / 1e9, "peak": link, "unit": "GB/s",
                 "frac": fill_bytes / cache_s / 1e9 / link,
                 "traffic": TRAFFIC_PER_BYTE["fill"] * fill_bytes / max(n_ls, 1), "traffic_source": scaled,
                 "algorithmic_bytes_per_launch": fill_bytes / max(n_ls, 1),
                 "avg_launch_ms": sum(cache_ms) / max(n_ls, 1),
                 "peak_source": "cudaMemcpyAsync pinned->device, measured in this run"}
    roof_exp = {"kernel": "ft_expert_grouped (tcgen05 expert launches)", "bound": "hbm",
                "achieved": expert_hbm / expert_s / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": expert_hbm / expert_s / 1e9 / peaks["hbm_gbs"],
                "traffic": TRAFFIC_PER_BYTE["experts"] * expert_hbm / max(n_ls, 1), "traffic_source": scaled,
                "algorithmic_bytes_per_launch": expert_hbm / max(n_ls, 1),
                "avg_launch_ms": sum(expert_ms) / max(n_ls, 1),
                "peak_source": f"MEASURED_PEAKS hbm_gbs ({peaks['source']}, of measured)"}
    return {"per_batch": per,
            "layer_roofline_frac": acc["roof"] / (acc["ms"] * 1e-3),
            "steady_state": {"from_step": steady_from, "tokens_per_s": acc["tok_s"] / (acc["ms_s"] * 1e-3),
                             "layer_roofline_frac": acc["roof_s"] / (acc["ms_s"] * 1e-3)},
            "trace_tokens_per_s": acc["tok"] / (acc["ms"] * 1e-3),
            "roofline": roof_fill if cache_s >= expert_s else roof_exp,
            "roofline_fill": roof_fill, "roofline_experts": roof_exp}


def nvfp4_leg(ft, dev, peaks, link, batches, steps, split_min=0):
    """The 43-layer NVFP4 stack: ``steps`` decode steps per batch size from a cold 40% cache,
    and 8192-token streamed prefill.

    The host pool stores a cyclic window of 4 physical layers (logical layer l
    reads physical l mod 4); cache keys and bytes moved stay logical."""
    cfg = synth.NVFP4_43L
    pool = ft.ExpertPool(cfg, 4)
    pool.fill(dev)
    payload = int(ft.ft_expert_layout_get(cfg.wtype, cfg.hidden, cfg.inter).payload_bytes)
    routers = [synth.router_weights(cfg, l, dev) for l in range(cfg.n_layers)]
    n_slots = int(round(CACHE_FRAC * cfg.n_layers * cfg.n_experts))
    run = DecodeRun(ft, cfg, pool, routers, batches, steps, dev, n_slots, split_min)
    run.capture()
    marks = []
    run.run_pass(marks)
    torch.cuda.synchronize()
    run.capture(instrumented=True)
    run.run_pass(instrumented=True)
    torch.cuda.synchronize()
    rep = decode_report(run, marks, cfg, peaks, link, payload, steady_from=min(8, steps - 1))
    run.release()
    del run
    torch.cuda.empty_cache()
    res = {"workload": "nvfp4_43L: H=4096 E=256 top-6 I=2048, NVFP4 weights, 43 layers over a 4-layer host window",
           "cache_slots": n_slots, "decode_steps": steps,
           "decode": {"from_cold": rep["per_batch"], "layer_roofline_frac": rep["layer_roofline_frac"],
                      "steady_state": rep["steady_state"], "roofline_experts": rep["roofline_experts"],
                      "roofline_fill": rep["roofline_fill"]}}
    log("nvfp4 prefill")
    res["prefill_8192"] = prefill_leg(ft, cfg, pool, routers, dev, [8192], link, peaks)
    pool.free()
    return res


def host_bandwidth(ft, cfg, pool, cpu, payload, tokens=8, reps=3):
    """B_H ([Review] §2.5, Table 1): expert bytes per second of the host executor, one
    token per expert, measured on ``tokens`` x top-k distinct experts of physical layer
    0; with B_P (the pinned-copy rate of the same records) the ratio that sets q*."""
    k, E = cfg.top_k, cfg.n_experts
    n = min(tokens * k, E)
    T = n // k
    idx = torch.arange(T * k, dtype=torch.int32).reshape(T, k)
    w = torch.full((T, k), 1.0 / k)
    ext = torch.ones(E, dtype=torch.int32)
    x = synth.activations(cfg, T, tag=9).to(torch.bfloat16 if cfg.x_dtype == "bf16" else torch.float32)
    part = torch.empty(T, cfg.hidden)
    job = cpu.job(pool.ptr, pool.S, cfg.wtype, cfg.hidden, cfg.inter, E, 0, x, T, k, idx, w, ext, part)
    cpu.run(job)
    best = float("inf")
    for _ in range(reps):
        t0 = time.perf_counter()
        cpu.run(job)
        best = min(best, time.perf_counter() - t0)
    d = torch.empty(n * pool.S, dtype=torch.uint8, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    bp = 0.0
    for _ in range(reps):
        e0.record()
        d.copy_(pool.host[: n * pool.S], non_blocking=True)
        e1.record()
        e1.synchronize()
        bp = max(bp, n * payload / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    del d
    bh = n * payload / best / 1e9
    return {"experts": n, "bw_host_gbs": bh, "bw_fill_gbs": bp, "ratio_fill_over_host": bp / bh,
            "q_for_m": {m: ft.ft_qsplit(m, bp, bh) for m in (1, 2, 3, 4, 6, 8, 16)},
            "threads": cpu_threads(), "host_cpu": host_cpu_model(), "host_rows_form": ft.HOST_FORMS[ft.ft_debug_host_simd(-1)]}


def host_cpu_model() -> str:
    """The host CPU's model name (/proc/cpuinfo), or "" where it cannot be read."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return ""


def cpu_threads() -> int:
    """Threads of an executor created with threads=0: the hardware threads, at most 256."""
    return min(256, os.cpu_count() or 1)


def mxfp4_mixed_leg(ft, dev, peaks, link, decode_steps=512, cycles=4, split_min=0):
    """The MXFP4 agent-like trace on 4 layers: cycles of (8192-token prefill, T=1 decode run).

    The cache is resized at the safe point before each cycle (57.8% -> 40% ->
    20% -> 57.8% of the 1024 (layer, expert) slots); misses are split with
    ratio 0.7, so 30% of them go to the external path.  In decode the host
    expert executor evaluates them from the pinned pool, as a host node of the
    captured step, and the combine adds its partial output; in the 8192-token
    on-demand prefill waves their partial is a zero placeholder (thousands of
    token-expert products per wave, beyond a bounded bench run on host cores).
    With fewer slots than two whole layers the prefill runs on demand through
    the cache in waves; otherwise it streams.  Every resize re-captures the
    decode graph, since the wave count can change.  Before the trace, the host
    executor's expert bandwidth B_H is measured against the pinned-copy B_P."""
    cfg = synth.MXFP4_MIXED
    L, E, H = cfg.n_layers, cfg.n_experts, cfg.hidden
    budgets = [592, 410, 205, 592][:cycles]
    pool = ft.ExpertPool(cfg, L)
    pool.fill(dev)
    payload = int(ft.ft_expert_layout_get(cfg.wtype, cfg.hidden, cfg.inter).payload_bytes)
    routers = [synth.router_weights(cfg, l, dev) for l in range(L)]
    zero_b = torch.zeros(E, dtype=torch.float32, device=dev)
    max_slots = max(budgets)
    sp = torch.empty(max_slots * pool.S, dtype=torch.uint8, device=dev)
    cache = ft.Cache(L, E, L, budgets[0], max_slots, pool.S, pool.ptr, sp)
    lay_p = ft.MoELayer(cfg, 8192, dev)
    lay_d = ft.MoELayer(cfg, 1, dev)
    P_p = torch.zeros(8192, H, dtype=torch.float32, device=dev)
    P_d = torch.zeros(1, H, dtype=torch.float32, device=dev)
    x_d = torch.empty(1, H, dtype=torch.bfloat16, device=dev)
    counts_d = torch.zeros(L, 8, 4, dtype=torch.int32, device=dev)   # per layer, per wave (<= 8 waves)
    trace = synth.AR1Trace(cfg, 1, dev, tag=5)
    slot_of = torch.empty(E, dtype=torch.int32, device=dev)
    ratio = 0.7
    fs = torch.cuda.Stream(device=dev)                        # the fill stream of the split form
    fs_d = fs if split_min >= 0 and ft.split_pays(1, cfg.top_k, cfg.wtype, split_min) else None
    fs_p = fs if split_min >= 0 and ft.split_pays(8192, cfg.top_k, cfg.wtype, split_min) else None
    cpu = ft.CpuExperts(threads=0)
    hb = ft.HostBranch(cfg, 1, pool, cpu, dev) if fs_d is not None else None
    bh = host_bandwidth(ft, cfg, pool, cpu, payload)

    def decode_layers():
        for l in range(L):
            lay_d.route(x_d, *routers[l])
            nw = cache.n_waves()
            for w in range(nw):
                after = (lambda l=l: hb.launch(lay_d, x_d, l)) if hb is not None and w == nw - 1 else None
                lay_d.cached_wave(x_d, l, cache, pool.S, ratio, w, counts_d[l, w], fill_stream=fs_d,
                                  after_control=after)
            if hb is not None:
                hb.join()
                lay_d.combine(1, lay_d.ext, hb.P[:1])
            else:
                lay_d.combine(1, lay_d.ext, P_d)

    cyc = []
    total_ms, total_tokens, roof_s = 0.0, 0, 0.0
    for c, N in enumerate(budgets):
        if c > 0:
            cache.resize(N)                     # safe point: nothing in flight
        xp = synth.activations(cfg, 8192, tag=100 + c, device=dev)
        streamed = N >= 2 * E
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        if streamed:
            st = ft.Stream(cache)
            for l in range(L):
                st.layer(l, l + 1 if l + 1 < L else -1, slot_of)
                lay_p.forward_slots(xp, routers[l][0], zero_b, slot_of, sp, pool.S, max_slots)
                st.layer_done(l)
        else:
            for l in range(L):
                lay_p.forward_cached(xp, routers[l][0], zero_b, l, cache, pool.S, fill_ratio=ratio, ext_partial=P_p,
                                     fill_stream=fs_p)
        e1.record()
        torch.cuda.synchronize()
        p_ms = e0.elapsed_time(e1)
        p_bytes = 0
        if streamed:
            p_bytes = st.bytes()
            st.destroy()
        stats0 = cache.stats()
        # decode run: one graph of the 4 layers, re-captured for this cache size, replayed per step
        for _ in range(3):
            x_d.copy_(trace.next())
            decode_layers()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            decode_layers()
        hist = torch.zeros(decode_steps, L, 4, dtype=torch.int32, device=dev)
        xs = torch.stack([trace.next() for _ in range(decode_steps)])
        torch.cuda.synchronize()
        e0.record()
        counts_d.zero_()
        for t in range(decode_steps):
            x_d.copy_(xs[t])
            g.replay()
            torch.sum(counts_d, dim=1, out=hist[t])   # a step's counts: the sum over its waves
        e1.record()
        torch.cuda.synchronize()
        d_ms = e0.elapsed_time(e1)
        h = hist.cpu().numpy()
        d_roof, _ = layer_roofline_seconds(h, 1, cfg, payload, peaks, link)
        stats1 = cache.stats()
        p_link = p_bytes if streamed else (stats0.bytes_h2d - (cyc[-1]["_bytes_after"] if cyc else 0))
        p_flops = 2.0 * 8192 * cfg.top_k * 3 * cfg.hidden * cfg.inter * L
        p_roof = max(p_link / (link * 1e9), p_flops / (peaks["bf16_tflops_sustained"] * 1e12))
        cyc.append({"slots": N, "prefill_mode": "streamed" if streamed else "on-demand (waves, 30% external)",
                    "prefill_ms": p_ms, "prefill_tokens_per_s": 8192 / (p_ms * 1e-3),
                    "prefill_h2d_gbs": p_link / (p_ms * 1e-3) / 1e9, "prefill_roofline_frac": p_roof / (p_ms * 1e-3),
                    "decode_tokens_per_s": decode_steps / (d_ms * 1e-3), "decode_ms_per_step": d_ms / decode_steps,
                    "decode_layer_roofline_frac": d_roof / (d_ms * 1e-3),
                    "decode_hits": int(h[..., 1].sum()), "decode_fills": int(h[..., 2].sum()),
                    "decode_externals": int(h[..., 3].sum()), "_bytes_after": stats1.bytes_h2d})
        total_ms += p_ms + d_ms
        total_tokens += 8192 + decode_steps
        roof_s += p_roof + d_roof
        del g
    for c in cyc:
        c.pop("_bytes_after")
    torch.cuda.synchronize()
    cpu_status = cpu.status()
    cache.destroy()
    cpu.destroy()
    pool.free()
    del sp
    torch.cuda.empty_cache()
    return {"workload": "mxfp4_mixed_4L: H=6144 E=256 top-8 I=2048, MXFP4 weights, 4 layers; "
                        "4 x (8192-token prefill, 512 T=1 decode steps); cache 592/410/205/592 slots; 30% external",
            "tokens_per_s": total_tokens / (total_ms * 1e-3), "layer_roofline_frac": roof_s / (total_ms * 1e-3),
            "external_path": ("decode: host expert executor (graph host node); prefill waves: zero placeholder"
                              if hb is not None else "zero placeholder"),
            "host_executor_status": cpu_status, "host_bandwidth": bh, "cycles": cyc}


# ---------------------------------------------------------------- CPU oracle baseline

def _oracle_items(cfg, items):
    """Untimed preparation of (token, layer) samples: the token's hidden state, the
    layer's router, and the stored components of the experts it routes to."""
    from oracle import formats, moe
    trace = synth.AR1Trace(cfg, 1, "cpu", tag=1)
    n_tok = 1 + max(t for t, _ in items)
    xs = [trace.next().clone() for _ in range(n_tok)]
    routers, out = {}, []
    for t, l in items:
        if l not in routers:
            routers[l] = synth.router_weights(cfg, l, "cpu")
        wr, b = routers[l]
        z = moe.router_logits(formats.to_f64(xs[t]), formats.to_f64(wr), formats.to_f64(b))
        idx, _ = moe.route(z, cfg.top_k)
        comps = {int(e): synth.expert_weights(cfg, l, int(e), "cpu") for e in sorted(set(idx.reshape(-1).tolist()))}
        out.append((xs[t], wr, b, comps))
    return out


def _oracle_eval(cfg, prepared):
    """The oracle on prepared samples: routing, decoding the stored weights, the expert FFNs and the sum."""
    from oracle import formats, moe
    for x, wr, b, comps in prepared:
        x64 = formats.to_f64(x)
        z = moe.router_logits(x64, formats.to_f64(wr), formats.to_f64(b))
        idx, w = moe.route(z, cfg.top_k)
        moe.moe_layer(x64, idx, w, moe.ExpertSource(lambda e: comps[e], cfg.wtype))


def _oracle_worker(rank, n_workers, cfg_name, items, barrier, more, ready):
    """One process of the CPU baseline: one BLAS thread (set in the environment before
    numpy loaded), its share of the samples, prepared before it reports ready, then
    evaluated once per round."""
    try:
        torch.set_num_threads(1)
        cfg = synth.CONFIGS[cfg_name]
        mine = items[rank::n_workers]
        prepared = _oracle_items(cfg, mine) if mine else []
    except BaseException as e:          # report, so that the parent stops waiting
        ready.put(("error", rank, repr(e)))
        raise
    ready.put(("ready", rank, ""))
    while True:
        barrier.wait()                  # go
        if not more.value:
            return
        _oracle_eval(cfg, prepared)
        barrier.wait()                  # done


class OraclePool:
    """The fp64 oracle on the host cores: one spawned process per core (at most
    ``max_workers``), each with one BLAS thread, evaluating its share of
    (token, layer) samples once per round.  Rounds are timed on the wall clock."""

    THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")

    def __init__(self, cfg, n_tokens, max_workers=32, prepare_timeout_s=600.0):
        import multiprocessing as mp
        import queue
        self.cfg = cfg
        self.cores = max(1, min(len(os.sched_getaffinity(0)), max_workers))
        self.items = [(t, l) for t in range(n_tokens) for l in range(cfg.n_layers)]
        self.n_tokens = n_tokens
        ctx = mp.get_context("spawn")
        n = min(self.cores, len(self.items))
        self.n = n
        self.barrier = ctx.Barrier(n + 1)
        self.more = ctx.Value("i", 1)
        ready = ctx.Queue()
        self.procs = [ctx.Process(target=_oracle_worker, args=(r, n, cfg.name, self.items, self.barrier, self.more,
                                                               ready), daemon=True) for r in range(n)]
        saved = {v: os.environ.get(v) for v in self.THREAD_VARS}
        try:
            for v in self.THREAD_VARS:          # the children load numpy with one BLAS thread each
                os.environ[v] = "1"
            for p in self.procs:
                p.start()
        finally:
            for v, old in saved.items():
                if old is None:
                    os.environ.pop(v, None)
                else:
                    os.environ[v] = old
        got, t0 = 0, time.perf_counter()
        while got < n:
            try:
                kind, rank, msg = ready.get(timeout=2.0)
            except queue.Empty:
                dead = [p.exitcode for p in self.procs if p.exitcode is not None]
                if dead or time.perf_counter() - t0 > prepare_timeout_s:
                    self._kill()
                    raise RuntimeError(f"oracle workers failed to start (exit codes {dead})")
                continue
            if kind == "error":
                self._kill()
                raise RuntimeError(f"oracle worker {rank} failed: {msg}")
            got += 1

    def _kill(self):
        for p in self.procs:
            if p.is_alive():
                p.kill()
            p.join(timeout=10)

    def round(self) -> float:
        """Evaluates every sample once; wall seconds."""
        t0 = time.perf_counter()
        self.barrier.wait(timeout=600)
        self.barrier.wait(timeout=600)
        return time.perf_counter() - t0

    def close(self):
        self.more.value = 0
        try:
            self.barrier.wait(timeout=60)
        except Exception:
            pass
        for p in self.procs:
            p.join(timeout=30)
        self._kill()

    def sample(self) -> str:
        return (f"{self.n_tokens} T=1 decode token(s) of the AR(1) trace through all {self.cfg.n_layers} layers "
                f"({len(self.items)} (token, layer) samples, weights drawn on the CPU with the same generator and "
                f"decoded from the stored format inside the timed region), over {self.n} processes")


def oracle_baseline(cfg, n_tokens=2, reps=None, budget_s=12.0):
    """cpu_baseline: rounds of the oracle pool until about ``budget_s`` seconds of wall time
    (None, with the reason logged, if the pool cannot run)."""
    try:
        op = OraclePool(cfg, n_tokens)
    except RuntimeError as e:
        log(f"cpu baseline skipped: {e}")
        return None
    try:
        t = [op.round()]
        n = reps or max(1, int(budget_s / max(t[0], 1e-3)))
        t = [op.round() for _ in range(n)]
    finally:
        op.close()
    v = n_tokens * len(t) / sum(t)
    return {"value": v, "unit": "tokens/s", "cores": op.n, "kind": "oracle", "sample": op.sample() +
            f", {len(t)} timed rounds"}


def reference_main(args, world, rank):
    """--impl reference: the fp64 oracle, as it stands, on the host cores."""
    if rank != 0:
        return
    cfg = synth.DECODE_BF16
    op = OraclePool(cfg, args.cpu_tokens)
    try:
        for _ in range(args.warmup):
            op.round()
        t = [op.round() for _ in range(args.steps)]
    finally:
        op.close()
    dt = sum(t)
    v = args.cpu_tokens * args.steps / dt
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "batches": [1], "parallelism": "replicas1",
                   "step": f"{args.cpu_tokens} T=1 decode token(s) through all {cfg.n_layers} layers"},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": op.n, "kind": "oracle", "sample": op.sample()},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def placement_leg(ft, cfg, routers, dev, steps=1024, prompt=2048, fracs=(0.37, 0.11)):
    """Placement-policy replay ([Review] §2.4): the routing of a T=1 decode trace and
    of a prompt, both computed by the library's routing kernels, replayed on the host
    (ft_placement_replay) under the shared LRU, a hot set fixed at prefill time and a
    static split by layer, at 37% and 11% of the (layer, expert) pool."""
    L, E, k = cfg.n_layers, cfg.n_experts, cfg.top_k
    lay = ft.MoELayer(cfg, max(prompt, steps), dev)
    x = synth.activations(cfg, prompt, tag=77, device=dev)
    pc = torch.zeros(L, E, dtype=torch.int32, device=dev)
    for l in range(L):
        lay.route(x, *routers[l])
        pc[l].copy_(lay.counts)
    tr = synth.AR1Trace(cfg, 1, dev, tag=1)
    xs = torch.cat([tr.next() for _ in range(steps)])               # [steps, H]: one token per step
    ids = torch.empty(steps, L, k, dtype=torch.int32, device=dev)
    for l in range(L):
        lay.route(xs, *routers[l])
        ids[:, l].copy_(lay.idx[:steps])
    ids_h, pc_h = ids.cpu().numpy(), pc.cpu().numpy().reshape(-1)
    out = {"decode_steps": steps, "batch": 1, "prompt_tokens": prompt,
           "note": "synthetic AR(1)+Zipf(1.1) routing; the pages' 16%/39% (LRU), 41%/59% (prefill-time) and "
                   "62%/89% (static) come from real routing traces that are not available here"}
    names = {ft.FT_PLACE_GLOBAL_LRU: "global_lru", ft.FT_PLACE_PREFILL_HOT: "prefill_hot_set",
             ft.FT_PLACE_STATIC_SPLIT: "static_split"}
    for f in fracs:
        cap = int(round(f * L * E))
        row = {"capacity": cap}
        for pol, name in names.items():
            acc, miss = ft.ft_placement_replay(pol, L, E, cap, ids_h, pc_h if pol == ft.FT_PLACE_PREFILL_HOT else None)
            row[name] = miss / max(acc, 1)
        out[f"{round(f * 100)}%"] = row
    del lay
    torch.cuda.empty_cache()
    return out


def pool_setup_leg(ft, cfg, pool, n_layers):
    """Pool setup from a pool file, pin first (ft_host_alloc, then the read) against read
    then pin (the read into fresh pageable memory, then ft_host_register), for the first
    ``n_layers`` layers of the pool ([Review] §2.7, fast engine start).  The file is
    written once beforehand and read back through the page cache."""
    import shutil
    E, S = cfg.n_experts, pool.S
    n = n_layers * E * S
    d = tempfile.gettempdir()
    if shutil.disk_usage(d).free < 1.5 * n:
        return {"skipped": f"not enough free space in {d} for a {n / 1e9:.1f} GB pool file"}
    path = os.path.join(d, f"ft_pool_{os.getpid()}.bin")
    try:
        with open(path, "wb") as f:
            f.write(memoryview(pool.host[:n].numpy()))
        runs = {"pin_first": [], "read_then_pin": []}
        for _ in range(2):
            for mode in ("pin_first", "read_then_pin"):
                t0 = time.perf_counter()
                p = ft.ExpertPool.load(cfg, n_layers, path, read_then_pin=(mode == "read_then_pin"))
                total = time.perf_counter() - t0
                ok = bool(torch.equal(p.host[: 1 << 20], pool.host[: 1 << 20]))
                runs[mode].append(dict(p.setup_s, total=total, same_bytes=ok))
                p.free()
        best = {m: min(r, key=lambda x: x["total"]) for m, r in runs.items()}
        return {"layers": n_layers, "bytes": n, "runs": runs,
                "gbs": {m: n / b["total"] / 1e9 for m, b in best.items()},
                "speedup_read_then_pin": best["pin_first"]["total"] / best["read_then_pin"]["total"],
                "source": "pool file in the page cache (no disk reads); threads: hardware count, at most 64"}
    finally:
        if os.path.exists(path):
            os.unlink(path)


# ---------------------------------------------------------------- single expert-kernel cases (profiling)

def fill_case(args):
    """Miss fill alone: a 1-layer BF16 pool (1.6 GB pinned), a fresh 64-slot cache, 32 routed experts.

    Each repetition starts from an empty cache, so its one fill launch copies
    all 32 experts (201 MB) over the host link."""
    import expert_cache_streaming_fp32_b300 as ft
    dev = "cuda:0"
    torch.cuda.set_device(0)
    cfg = synth.DECODE_BF16
    E = cfg.n_experts
    pool = ft.ExpertPool(cfg, 1)
    pool.fill(dev)
    payload = int(ft.ft_expert_layout_get(cfg.wtype, cfg.hidden, cfg.inter).payload_bytes)
    counts = torch.zeros(E, dtype=torch.int32, device=dev)
    counts[torch.arange(0, E, E // 32)] = 1
    slot_of = torch.empty(E, dtype=torch.int32, device=dev)
    sc = torch.zeros(4, dtype=torch.int32, device=dev)
    sp = torch.empty(64 * pool.S, dtype=torch.uint8, device=dev)
    ms = []
    for r in range(3 + args.reps):
        cache = ft.Cache(1, E, 1, 64, 64, pool.S, pool.ptr, sp)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        cache.step(0, counts, 1.0, 0, slot_of, None, sc)
        e1.record()
        torch.cuda.synchronize()
        if r >= 3:
            ms.append(e0.elapsed_time(e1))
        cache.destroy()
    link = link_peak_gbs(pool.host, E * pool.S, dev)
    t = float(np.median(ms))
    print(json.dumps({"kernel_case": "fill", "experts": int(sc[2]), "ms": t,
                      "link_gbs": int(sc[2]) * payload / (t * 1e-3) / 1e9, "link_peak_gbs": link,
                      "device_error": ft.ft_get_device_error()}))


def fill_overlap_case(args):
    """Fill blocks vs the fill's rate alone and beside an expert call.

    The 32-expert fill of ``fill`` on a second stream, with 20 back-to-back
    64-token expert calls over a resident layer on the first (the overlap of
    a split cache step), for several fill block counts."""
    import expert_cache_streaming_fp32_b300 as ft
    dev = "cuda:0"
    torch.cuda.set_device(0)
    cfg = synth.DECODE_BF16
    E = cfg.n_experts
    pool = ft.ExpertPool(cfg, 1)
    pool.fill(dev)
    S = pool.S
    payload = int(ft.ft_expert_layout_get(cfg.wtype, cfg.hidden, cfg.inter).payload_bytes)
    resident = pool.host[: E * S].to(dev)
    so = torch.arange(E, dtype=torch.int32, device=dev)
    counts = torch.zeros(E, dtype=torch.int32, device=dev)
    counts[torch.arange(0, E, E // 32)] = 1
    slot_of = torch.empty(E, dtype=torch.int32, device=dev)
    sc = torch.zeros(4, dtype=torch.int32, device=dev)
    sp = torch.empty(64 * S, dtype=torch.uint8, device=dev)
    fs = torch.cuda.Stream()
    T, n_calls = 64, 20
    lay = ft.MoELayer(cfg, T, dev)
    x = synth.activations(cfg, T, tag=1, device=dev)
    lay.route(x, *synth.router_weights(cfg, 0, dev))

    def ev():
        return torch.cuda.Event(enable_timing=True)

    def experts():
        for _ in range(n_calls):
            lay.experts(x, so, resident, S, E)

    def once(blocks, beside):
        cache = ft.Cache(1, E, 1, 64, 64, S, pool.ptr, sp)
        cache.set_fill_blocks(blocks)
        torch.cuda.synchronize()
        f0, f1, m0, m1 = ev(), ev(), ev(), ev()
        f0.record(fs)
        cache.step(0, counts, 1.0, 0, slot_of, None, sc, stream=fs)
        f1.record(fs)
        if beside:
            m0.record()
            experts()
            m1.record()
        torch.cuda.synchronize()
        cache.destroy()
        return f0.elapsed_time(f1), (m0.elapsed_time(m1) if beside else None)

    m0, m1 = ev(), ev()
    alone = []
    for _ in range(3):
        m0.record()
        experts()
        m1.record()
        torch.cuda.synchronize()
        alone.append(m0.elapsed_time(m1))
    # the same bytes by the copy engine (one cudaMemcpyAsync of 32 contiguous records) beside the same calls
    dst = torch.empty(32 * S, dtype=torch.uint8, device=dev)
    ce = []
    for _ in range(3):
        torch.cuda.synchronize()
        f0, f1, c0, c1 = ev(), ev(), ev(), ev()
        f0.record(fs)
        with torch.cuda.stream(fs):
            dst.copy_(pool.host[: 32 * S], non_blocking=True)
        f1.record(fs)
        c0.record()
        experts()
        c1.record()
        torch.cuda.synchronize()
        ce.append((f0.elapsed_time(f1), c0.elapsed_time(c1)))
    ce = ce[1:]
    rows = []
    for blocks in (4, 8, 16, 32, 64, 148, 296):
        a = [once(blocks, False)[0] for _ in range(3)][1:]
        b = [once(blocks, True) for _ in range(3)][1:]
        rows.append({"fill_blocks": blocks,
                     "fill_alone_gbs": 32 * payload / (np.mean(a) * 1e-3) / 1e9,
                     "fill_beside_gbs": 32 * payload / (np.mean([f for f, _ in b]) * 1e-3) / 1e9,
                     "experts_beside_ms": float(np.mean([m for _, m in b]))})
    print(json.dumps({"kernel_case": "fill_overlap", "fill_experts": 32, "expert_calls": n_calls, "T": T,
                      "experts_alone_ms": float(np.median(alone)), "rows": rows,
                      "copy_engine": {"copy_gbs": 32 * S / (np.mean([f for f, _ in ce]) * 1e-3) / 1e9,
                                      "experts_beside_ms": float(np.mean([m for _, m in ce]))},
                      "device_error": ft.ft_get_device_error()}))


def host_records(ft, wtype, H, I, n, seed=1):
    """n expert records of one format in ordinary host memory: seeded random bytes with
    values and scales in range (bf16 values N(0, 0.02), e4m3 bytes below the NaN code,
    e4m3 / E8M0 block scales near 1, NVFP4 tensor scales 0.01)."""
    L = ft.ft_expert_layout_get(wtype, H, I)
    S = int(L.bytes)
    g = torch.Generator().manual_seed(seed)
    pool = torch.randint(0, 256, (n * S,), dtype=torch.uint8, generator=g)
    for e in range(n):
        base = e * S
        for m in range(3):
            K, rows = (H, I) if m < 2 else (I, H)
            v0, s0 = base + int(L.off_val[m]), base + int(L.off_scale[m])
            if wtype == synth.W_BF16:
                vals = (torch.randn(rows * K, generator=g) * 0.02).to(torch.bfloat16)
                pool[v0:v0 + 2 * rows * K] = vals.view(torch.uint8)
            elif wtype == synth.W_FP8:
                pool[v0:v0 + rows * K] = torch.randint(0, 0x78, (rows * K,), dtype=torch.uint8, generator=g)
                pool[s0:s0 + 4 * rows * (K // 128)] = torch.full((rows * (K // 128),), 0.01).view(torch.uint8)
            elif wtype == synth.W_NVFP4:
                ns = rows * (K // 16)
                pool[s0:s0 + ns] = torch.randint(0x30, 0x40, (ns,), dtype=torch.uint8, generator=g)
            elif wtype == synth.W_MXFP4:
                ns = rows * (K // 32)
                pool[s0:s0 + ns] = torch.randint(118, 128, (ns,), dtype=torch.uint8, generator=g)
        if wtype == synth.W_NVFP4:
            o = base + int(L.off_gscale)
            pool[o:o + 12] = torch.full((3,), 0.01).view(torch.uint8)
    return pool, S, int(L.payload_bytes)


def host_experts_case(args):
    """The host expert executor alone (no GPU): one token on each of 16 experts, per weight
    format at its workload's expert shape, in every row form the CPU runs (AVX-512, AVX2,
    portable), in expert bytes per second (B_H, [Review] §2.5).

    The records are seeded random bytes with in-range values and scales (host_records),
    not the weight generator's draws, whose FP4 quantisation of 16 large experts takes
    minutes; the executor does the same work for any in-range values."""
    import expert_cache_streaming_fp32_b300 as ft
    shapes = [("decode_bf16_40L", synth.W_BF16, 2048, 512), ("fp8, decode_bf16_40L shape", synth.W_FP8, 2048, 512),
              ("nvfp4_43L", synth.W_NVFP4, 4096, 2048), ("mxfp4_mixed_4L", synth.W_MXFP4, 6144, 2048)]
    n, k = 16, 8
    T = n // k
    best_form = ft.ft_debug_host_simd(-1)
    forms = []
    for f in (2, 1, 0):
        ft.ft_debug_host_simd(f)
        if ft.ft_debug_host_simd(-1) == f:
            forms.append(f)
    cpu = ft.CpuExperts(threads=0)
    rows = []
    try:
        for name, wt, H, I in shapes:
            pool, S, payload = host_records(ft, wt, H, I, n)
            idx = torch.arange(n, dtype=torch.int32).reshape(T, k)
            w = torch.full((T, k), 1.0 / k)
            ext = torch.ones(n, dtype=torch.int32)
            x = (torch.randn(T, H, generator=torch.Generator().manual_seed(2)) * 0.5).to(torch.bfloat16)
            part = torch.empty(T, H)
            job = cpu.job(pool.data_ptr(), S, wt, H, I, n, 0, x, T, k, idx, w, ext, part)
            row = {"workload": name, "format": synth.WTYPE_NAMES[wt], "experts": n, "expert_bytes": payload}
            for f in forms:
                ft.ft_debug_host_simd(f)
                cpu.run(job)
                best = float("inf")
                for _ in range(max(10, args.reps)):
                    t0 = time.perf_counter()
                    cpu.run(job)
                    best = min(best, time.perf_counter() - t0)
                row[f"{ft.HOST_FORMS[f]}_gbs"] = n * payload / best / 1e9
                row[f"{ft.HOST_FORMS[f]}_ms"] = best * 1e3
            rows.append(row)
    finally:
        ft.ft_debug_host_simd(best_form)
        cpu.destroy()
    print(json.dumps({"kernel_case": "host_experts", "threads": cpu_threads(), "host_cpu": host_cpu_model(),
                      "forms": [ft.HOST_FORMS[f] for f in forms], "rows": rows}))


def route_case(args):
    """Routing of one decode batch (T = --batches[0]) of the 40-layer BF16 stack: the 40 layers'
    ft_route_fused calls (one launch up to 8 tokens), and the three routing kernels, each as one
    CUDA graph over the 40 routers, with a 256 MB write between layers (so that the router rows
    come from HBM, as in a decode step).  Prints ms per layer for both forms and for the writes
    alone.  Holds under 1 GB on the device."""
    import expert_cache_streaming_fp32_b300 as ft
    dev = "cuda:0"
    torch.cuda.set_device(0)
    cfg = synth.DECODE_BF16
    T, H, E, k, L = int(args.batches.split(",")[0]), cfg.hidden, cfg.n_experts, cfg.top_k, cfg.n_layers
    routers = [synth.router_weights(cfg, l, dev) for l in range(L)]
    x = synth.AR1Trace(cfg, T, dev, tag=7).next()
    lay = ft.MoELayer(cfg, T, dev)
    junk = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = {}
    for form in ("fused", "three", "writes"):
        st = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(st):
            lay.route(x, *routers[0], stream=st)
            lay.route_unfused(x, *routers[0], stream=st)
            st.synchronize()
            with torch.cuda.graph(g, stream=st):
                for l in range(L):
                    junk.fill_(l)
                    if form == "fused":
                        lay.route(x, *routers[l], stream=st)
                    elif form == "three":
                        lay.route_unfused(x, *routers[l], stream=st)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        out[form] = e0.elapsed_time(e1) / args.reps / L
    print(json.dumps({"kernel_case": "route", "config": cfg.name, "T": T, "layers": L,
                      "ms_per_layer": {"one_launch": out["fused"] - out["writes"],
                                       "three_kernels": out["three"] - out["writes"]},
                      "write_ms_per_layer": out["writes"], "arrivals_zero": not bool(lay.arrivals.any()),
                      "device_error": ft.ft_get_device_error()}))


def kernel_case(args):
    """One layer's experts resident in a 256-record slot pool (1.6 GB); ft_expert_grouped timed alone.

    experts_decode: T = --batches[0] tokens routed with the Zipf prior of the decode trace.
    experts_prefill: T = 8192 tokens, near-uniform routing (tensor-core path).
    Small enough on the device (< 3 GB) for a multi-pass ncu capture of one launch.
    """
    import expert_cache_streaming_fp32_b300 as ft
    dev = "cuda:0"
    torch.cuda.set_device(0)
    ft.ft_expert_set_fp4_path(ft.FT_FP4_BLOCK_SCALED if args.fp4_path == "block_scaled" else ft.FT_FP4_EXPAND_BF16)
    cfg = synth.DECODE_BF16 if args.kernel_case == "experts_decode" else synth.PREFILL_BF16
    if args.case_config:
        cfg = synth.CONFIGS[args.case_config]
    if args.case_experts:
        import dataclasses
        cfg = dataclasses.replace(cfg, name=f"{cfg.name}_e{args.case_experts}", n_experts=args.case_experts)
    T = int(args.batches.split(",")[0]) if args.kernel_case == "experts_decode" else 8192
    E, k, H, I = cfg.n_experts, cfg.top_k, cfg.hidden, cfg.inter
    lay = ft.ft_expert_layout_get(cfg.wtype, H, I)
    S = int(lay.bytes)
    pool = torch.empty(E * S, dtype=torch.uint8, device=dev)
    for e in range(E):
        ft.pack_expert(synth.expert_weights(cfg, 0, e, dev), cfg.wtype, lay, pool[e * S:(e + 1) * S])
    L = ft.MoELayer(cfg, T, dev)
    wr, b = synth.router_weights(cfg, 0, dev)
    x = synth.AR1Trace(cfg, T, dev, tag=7).next() if args.kernel_case == "experts_decode" else \
        synth.activations(cfg, T, tag=1, device=dev)
    L.route(x, wr, b)
    so = torch.arange(E, dtype=torch.int32, device=dev)
    for _ in range(3):
        L.experts(x, so, pool, S, E)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.reps):
        L.experts(x, so, pool, S, E)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.reps
    U = int((L.counts > 0).sum())
    wbytes = U * int(lay.payload_bytes)
    flops = 2.0 * T * k * 3 * H * I
    peaks = load_peaks()
    print(json.dumps({"kernel_case": args.kernel_case, "config": cfg.name, "fp4_path": args.fp4_path, "T": T,
                      "unique_experts": U, "ms": ms,
                      "weight_gbs": wbytes / (ms * 1e-3) / 1e9, "hbm_frac": wbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                      "tflops": flops / (ms * 1e-3) / 1e12, "bf16_frac": flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                      "device_error": ft.ft_get_device_error()}))


# ---------------------------------------------------------------- main

def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        reference_main(args, world, rank)
        return
    if args.kernel_case == "fill":
        fill_case(args)
        return
    if args.kernel_case == "fill_overlap":
        fill_overlap_case(args)
        return
    if args.kernel_case == "route":
        route_case(args)
        return
    if args.kernel_case == "host_experts":
        host_experts_case(args)
        return
    if args.kernel_case:
        kernel_case(args)
        return
    import expert_cache_streaming_fp32_b300 as ft
    dev = f"cuda:{local}"
    cfg = synth.DECODE_BF16
    peaks = load_peaks()
    ft.ft_expert_set_fp4_path(ft.FT_FP4_BLOCK_SCALED if args.fp4_path == "block_scaled" else ft.FT_FP4_EXPAND_BF16)
    # smallest decode batch (T*k) run in the split form: 0 the library's policy, -1 never
    split_min = -1 if args.no_split_fill else args.split_min_assignments
    batches = [int(b) for b in args.batches.split(",")]
    L, E = cfg.n_layers, cfg.n_experts
    lay_bytes = ft.ft_expert_layout_get(cfg.wtype, cfg.hidden, cfg.inter)
    S = int(lay_bytes.bytes)
    n_phys = args.phys_layers
    if n_phys <= 0:
        per_rank_ram = host_ram_bytes() * 0.75 / world
        n_phys = max(1, min(L, int(per_rank_ram // (E * S))))
    pool = ft.ExpertPool(cfg, n_phys)
    t_fill = time.perf_counter()
    pool.fill(dev)
    t_fill = time.perf_counter() - t_fill
    routers = [synth.router_weights(cfg, l, dev) for l in range(L)]
    link = link_peak_gbs(pool.host, E * S, dev)
    n_trace = args.trace_steps
    run = DecodeRun(ft, cfg, pool, routers, batches, n_trace, dev, int(round(CACHE_FRAC * L * E)), split_min,
                    e2e=not args.no_e2e, fill_blocks=args.fill_blocks)
    tokens_per_pass = n_trace * sum(batches)
    log(f"pool of {n_phys} layers filled in {t_fill:.1f} s; link {link:.1f} GB/s")
    t0 = time.perf_counter()
    run.capture(instrumented=args.timed_spans)
    if args.timed_spans:
        run.graphs = run.igraphs
    log(f"{len(run.graphs)} step graphs captured in {time.perf_counter() - t0:.1f} s")

    # warm-up passes (each the whole trace from cold caches); the first two must make
    # the same cache decisions, since every pass replays the same trace from the same state
    first = []
    for w in range(args.warmup):
        run.run_pass()
        if w < 2:
            first.append({T: run.hist(T) for T in batches})
    deterministic = (all(np.array_equal(first[0][T], first[1][T]) for T in batches) if len(first) == 2 else None)
    log(f"warm-up done ({args.warmup} passes; identical decisions: {deterministic})")

    # timed region: K passes of the whole trace
    barrier(world)
    torch.cuda.synchronize()
    clk = Clocks(local)
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    marks = []
    e_start.record()
    for k in range(args.steps):
        marks = []
        run.run_pass(marks)
    e_end.record()
    torch.cuda.synchronize()
    barrier(world)
    clocks = clk.stop()
    ms = e_start.elapsed_time(e_end)
    ms_max = max_over_ranks(world, ms)
    tokens = sum_over_ranks(world, tokens_per_pass * args.steps)
    value = tokens / (ms_max * 1e-3)
    log(f"timed region: {ms:.1f} ms ({args.steps} passes)")
    # per-kernel spans: the same trace once more through graphs that also hold timing events
    spans_pass_ms = None
    if not args.timed_spans:
        run.capture(instrumented=True)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record()
        run.run_pass(instrumented=True)
        s1.record()
        torch.cuda.synchronize()
        spans_pass_ms = s0.elapsed_time(s1)
        log(f"instrumented pass: {spans_pass_ms:.1f} ms")
    if args.profile_eager_steps > 0:
        profile_eager(run, args.profile_eager_steps)
    payload = int(lay_bytes.payload_bytes)
    rep = decode_report(run, marks, cfg, peaks, link, payload, args.steady_from)

    # end to end through the public API with host buffers: every step copies its input
    # from pinned host memory and every layer's output back to pinned host memory
    e2e = None
    if not args.no_e2e:
        n_e2e = max(1, min(args.steps, 2))
        barrier(world)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n_e2e):
            run.run_pass(e2e=True)
        e1.record()
        torch.cuda.synchronize()
        barrier(world)
        ms_e = max_over_ranks(world, e0.elapsed_time(e1))
        h2d = n_trace * sum(T * cfg.hidden * 2 for T in batches)
        d2h = n_trace * sum(L * T * cfg.hidden * 4 for T in batches)
        e2e = {"value": sum_over_ranks(world, tokens_per_pass * n_e2e) / (ms_e * 1e-3), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "note": "same graphs; each decode step's input copied from pinned host memory first and "
                       "every layer's output copied back after it"}
        log(f"end-to-end: {e2e['value']:.1f} tokens/s over {n_e2e} passes")

    launches = run.launches_per_pass() * args.steps
    run.release()
    del run
    torch.cuda.empty_cache()
    log("decode legs done")
    derr = ft.ft_get_device_error()

    placement = None
    if rank == 0 and not args.no_placement:
        log("placement replay")
        placement = placement_leg(ft, cfg, routers, dev)

    prefill = None
    if not args.no_prefill:
        log("prefill leg")
        prefill = prefill_leg(ft, cfg, pool, routers, dev, [int(p) for p in args.prompts.split(",")], link, peaks)

    setup = None
    if not args.no_pool_setup and rank == 0:
        log("pool setup: pin first vs read then pin")
        setup = pool_setup_leg(ft, cfg, pool, args.setup_layers)

    nvfp4 = mixed = None
    if not args.no_fp4 and world == 1:
        pool.free()
        torch.cuda.empty_cache()
        log("nvfp4 stack")
        nvfp4 = nvfp4_leg(ft, dev, peaks, link, batches, args.fp4_steps, split_min)
        log("mxfp4 mixed trace")
        mixed = mxfp4_mixed_leg(ft, dev, peaks, link, decode_steps=args.mixed_decode_steps,
                                split_min=split_min)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        log("cpu baseline")
        cpu = oracle_baseline(cfg, n_tokens=args.cpu_tokens, reps=None, budget_s=args.cpu_budget_s)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD,
                       "step": (f"one pass of the decode trace: {n_trace} decode steps of all {L} layers at each "
                                f"T in {tuple(batches)}, each T from a cold (empty) cache"),
                       "batches": batches, "trace_steps": n_trace, "tokens_per_step": tokens_per_pass,
                       "steady_from_step": args.steady_from,
                       "host_pool_layers": n_phys, "host_pool_gb": n_phys * E * S / 1e9, "weights": "bf16",
                       "accumulate": "f32",
                       "l2": "inputs larger than L2 (each decode step reads >= 50 MB of expert weights, "
                             "each pass >= 2 GB per T)",
                       "fill": ("ft_cache_step (fill, then all experts)" if args.no_split_fill else
                                f"{split_min or ft.SPLIT_MIN_ASSIGNMENTS[cfg.wtype]} <= T*k < "
                                f"{ft.FT_TC_WIDE_ASSIGNMENTS}: ft_cache_step_split (hits evaluated while the fill "
                                "copies on a second stream); other batches: ft_cache_step"),
                       "parallelism": f"replicas{world}"},
            "layer_roofline_frac": rep["layer_roofline_frac"],
            "steady_state": rep["steady_state"],
            "per_batch": rep["per_batch"],
            "deterministic_passes": deterministic,
            "kernel_spans": ("CUDA events recorded inside the timed passes' graphs" if args.timed_spans else
                             "CUDA events of one more pass of the same trace, from a cold cache, through graphs "
                             "that also hold event-record nodes (which keep the next launch from starting early, "
                             f"so the timed graphs carry none); that pass took {spans_pass_ms:.1f} ms against "
                             f"{ms_max / args.steps:.1f} ms per timed pass"),
            "roofline": rep["roofline"],
            "roofline_experts": rep["roofline_experts"],
            "roofline_fill": rep["roofline_fill"],
            "link_peak_gbs": link,
            "peaks": peaks,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "cuda_graphs": True,
            "clocks": clocks,
            "prefill_bf16": prefill,
            "pool_setup": setup,
            "placement_replay": placement,
            "nvfp4_43L": nvfp4,
            "mxfp4_mixed": mixed,
            "device_error": derr,
            "pool_fill_s": t_fill,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
