"""bench.py's per-kernel span bookkeeping on CPU, with stand-in events (no GPU).

Each wave of a decode step records tagged events; the fill span is "cache" to
"fill_end", and the expert span is "fill_end" to "expert_end" for the plain cache
step, or the hits' call plus the filled experts' call for the split step (whose
"fill_end" is recorded on the fill stream and may come after "hit_end").
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


class FakeEvent:
    def __init__(self, t):
        self.t = t

    def elapsed_time(self, other):
        return other.t - self.t


def log_of(seq):
    ev = bench.EventLog()
    ev.ev = [(tag, FakeEvent(t)) for tag, t in seq]
    return ev


def test_plain_step_spans():
    # two waves: cache 0..10 fill, experts 10..14; cache 20..21, experts 21..30
    ev = log_of([("cache", 0), ("fill_end", 10), ("expert_end", 14),
                 ("cache", 20), ("fill_end", 21), ("expert_end", 30)])
    cache, experts = ev.cache_expert_spans()
    assert cache == [10, 1] and experts == [4, 9]
    s = bench.spans_us([ev])
    assert s == {"control_fill": 5.5e3, "experts": 6.5e3}


def test_split_step_spans():
    # control ends at 2; the fill (other stream) ends at 12; hits run 2..6; join at 12; filled 12..15
    ev = log_of([("cache", 0), ("ctrl_end", 2), ("fill_end", 12), ("hit_end", 6), ("join", 12),
                 ("expert_end", 15),
                 ("cache", 20), ("ctrl_end", 21), ("fill_end", 22), ("hit_end", 25), ("join", 25),
                 ("expert_end", 26)])
    cache, experts = ev.cache_expert_spans()
    assert cache == [12, 2]
    assert experts == [(6 - 2) + (15 - 12), (25 - 21) + (26 - 25)]
    s = bench.spans_us([ev])
    assert s["hits"] == 1e3 * (4 + 4) / 2 and s["filled"] == 1e3 * (3 + 1) / 2
    assert s["wait_for_fill"] == 1e3 * (6 + 0) / 2


def test_launch_count_per_step():
    class Cfg:
        n_layers, wtype, top_k = 40, bench.synth.W_BF16, 8

    class Run:
        cfg, n_waves, n_steps, batches = Cfg, 1, 256, [1, 8, 64]
        launches_per_step = bench.DecodeRun.launches_per_step
        launches_per_pass = bench.DecodeRun.launches_per_pass

    r = Run()
    r.b = {1: {"split": False}, 8: {"split": False}, 64: {"split": True}}
    assert r.launches_per_step(1) == 40 * 6       # fused route, control, fill, gate/up + down (CUDA cores), combine
    assert r.launches_per_step(8) == 40 * 7       # up to 8 tokens: one routing launch; gather + gate/up + down
    assert r.launches_per_step(64) == 40 * 12     # the three routing kernels, a second expert call (split form)
    assert r.launches_per_pass() == 256 * 40 * (6 + 7 + 12)


def test_step_times_per_batch_exclude_the_reset_between_batches():
    # T=1: steps at 0, 2, 5, end 6; (reset); T=4: steps at 10, 11, end 15
    marks = [(1, 0, FakeEvent(0)), (1, 1, FakeEvent(2)), (1, 2, FakeEvent(5)), (1, -1, FakeEvent(6)),
             (4, 0, FakeEvent(10)), (4, 1, FakeEvent(11)), (4, -1, FakeEvent(15))]
    assert bench.step_times_ms(marks) == {1: [2, 3, 1], 4: [1, 4]}


def test_oracle_pool_times_rounds_on_spawned_processes():
    """The CPU baseline's process pool (spawned workers, one BLAS thread each) on the tiny layer."""
    op = bench.OraclePool(bench.synth.TINY_F32, n_tokens=3, max_workers=2)
    try:
        t = [op.round() for _ in range(2)]
    finally:
        op.close()
    assert op.n == min(2, len(os.sched_getaffinity(0))) and all(x > 0 for x in t)
    assert "3 T=1 decode token(s)" in op.sample()
    assert all(not p.is_alive() for p in op.procs)


def test_oracle_pool_reports_a_failing_worker_quickly():
    import time
    import pytest
    cfg = bench.synth.MoEConfig("not_a_registered_config", 256, 16, 2, 128, 1, bench.synth.W_F32, "f32")
    t0 = time.perf_counter()
    with pytest.raises(RuntimeError):
        bench.OraclePool(cfg, n_tokens=1, max_workers=2)
    assert time.perf_counter() - t0 < 120

