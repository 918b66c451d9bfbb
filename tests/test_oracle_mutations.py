"""Plant plausible mistakes in the oracle (CPU only) and check that a pin catches each one."""
import numpy as np
import pytest

import oracle.formats as formats
import oracle.lru as lru
import oracle.moe as moe
import oracle.qsplit as qsplit
import test_oracle_ffn as t_ffn
import test_oracle_formats_qsplit as t_fmt
import test_oracle_lru as t_lru
import test_oracle_route_permute as t_rp


def _fails(fn, *a):
    with pytest.raises(AssertionError):
        fn(*a)


def test_mutant_tie_break_to_higher_index(monkeypatch):
    def route(z, k):
        z = np.asarray(z, np.float64)
        order = (z.shape[1] - 1 - np.argsort(-z[:, ::-1], axis=1, kind="stable"))[:, :k]
        p = moe.softmax(z)
        sel = np.take_along_axis(p, order, axis=1)
        return order.astype(np.int32), sel / sel.sum(axis=1, keepdims=True)
    monkeypatch.setattr(moe, "route", route)
    _fails(t_rp.test_route_matches_brute_force, 7, 5, 2, 0)


def test_mutant_no_renormalisation(monkeypatch):
    def route(z, k):
        order = np.argsort(-z, axis=1, kind="stable")[:, :k]
        return order.astype(np.int32), np.take_along_axis(moe.softmax(z), order, axis=1)
    monkeypatch.setattr(moe, "route", route)
    _fails(t_rp.test_route_weights_sum_to_one_and_descend)


def test_mutant_bias_dropped(monkeypatch):
    monkeypatch.setattr(moe, "router_logits", lambda x, w, b=None: np.asarray(x) @ np.asarray(w).T)
    _fails(t_rp.test_router_logits_hand_example)


def test_mutant_unstable_permutation(monkeypatch):
    def permute(idx, E):
        c, o, p, i = orig(idx, E)
        for e in range(E):
            p[o[e]:o[e + 1]] = p[o[e]:o[e + 1]][::-1]
        i[p] = np.arange(p.size)
        return c, o, p, i
    orig = moe.permute
    monkeypatch.setattr(moe, "permute", permute)
    _fails(t_rp.test_permute_matches_brute_force, 16, 8, 32, 2)


def test_mutant_gate_up_swapped(monkeypatch):
    orig = moe.expert_ffn
    monkeypatch.setattr(moe, "expert_ffn", lambda X, g, u, d, act_round=None: orig(X, u, g, d, act_round))
    _fails(t_ffn.test_ffn_hand_example)


def test_mutant_silu_dropped(monkeypatch):
    monkeypatch.setattr(moe, "silu", lambda g: g)
    _fails(t_ffn.test_ffn_hand_example)


def test_mutant_sigmoid_instead_of_silu(monkeypatch):
    monkeypatch.setattr(moe, "silu", lambda g: 1.0 / (1.0 + np.exp(-g)))
    _fails(t_ffn.test_ffn_matches_scalar_loops_rectangular)


def test_mutant_combine_ignores_weights(monkeypatch):
    orig = moe.combine
    monkeypatch.setattr(moe, "combine", lambda Y, inv, w, k, skip=None, partial=None:
                        orig(Y, inv, np.ones_like(w), k, skip, partial))
    _fails(t_ffn.test_grouped_evaluation_equals_token_loop)


def test_mutant_round_half_even_in_qsplit(monkeypatch):
    def qr(m, ratio):
        if m <= 0:
            return 0
        if ratio >= 1.0:
            return m
        return min(m, max(1, int(round(m * ratio))))
    monkeypatch.setattr(qsplit, "qsplit_ratio", qr)
    _fails(t_fmt.test_qsplit_limits)


def test_mutant_qsplit_without_floor_of_one(monkeypatch):
    monkeypatch.setattr(qsplit, "qsplit_ratio", lambda m, r: m if r >= 1 else int(np.floor(m * r + 0.5)))
    _fails(t_fmt.test_qsplit_table1_worked_values)


def test_mutant_e4m3_wrong_bias(monkeypatch):
    def v(byte):
        s = -1.0 if (byte >> 7) & 1 else 1.0
        e, m = (byte >> 3) & 15, byte & 7
        if e == 15 and m == 7:
            return float("nan")
        if e == 0:
            return s * (m / 8.0) * 2.0 ** -7
        return s * 2.0 ** (e - 8) * (1.0 + m / 8.0)
    monkeypatch.setattr(formats, "e4m3_value", v)
    _fails(t_fmt.test_e4m3_all_bytes_match_library_conversion)


def test_mutant_nvfp4_block_of_32(monkeypatch):
    def deq(codes, scales, g):
        v = formats.E2M1_TABLE[formats.unpack_nibbles(codes)]
        R, K = v.shape
        s = formats.E4M3_TABLE[np.asarray(scales)][:, : K // 32]
        return (v.reshape(R, K // 32, 32) * s[:, :, None]).reshape(R, K) * g
    monkeypatch.setattr(formats, "dequant_nvfp4", deq)
    _fails(t_fmt.test_nvfp4_roundtrip_of_generator_quantiser)


def test_mutant_lru_evicts_most_recent(monkeypatch):
    def victims(self, q, touched):
        cand = [s for s in range(self.N) if s not in touched]
        cand.sort(key=lambda s: (0 if self.key[s] < 0 else 1, -self.stamp[s], s))
        return cand[:q]
    monkeypatch.setattr(lru.LRUSim, "_victims", victims)
    _fails(t_lru.test_single_access_steps_match_ordered_dict_lru, 3, 8, 2, 1)


def test_mutant_lru_hit_does_not_refresh(monkeypatch):
    orig = lru.LRUSim._wave

    def wave(self, layer, W, ratio):
        saved = list(self.stamp)
        ev, so = orig(self, layer, W, ratio)
        for e in W:
            s = so[e]
            if s >= 0 and any(x[0] == "hit" and x[1] == e for x in ev):
                self.stamp[s] = saved[s]
        return ev, so
    monkeypatch.setattr(lru.LRUSim, "_wave", wave)
    _fails(t_lru.test_single_access_steps_match_ordered_dict_lru, 3, 8, 2, 1)


def test_mutant_dispatch_codes_3_and_4_swapped(monkeypatch):
    orig = formats.dequant

    def dequant(component, wtype):
        return orig(component, {3: 4, 4: 3}.get(wtype, wtype))
    monkeypatch.setattr(formats, "dequant", dequant)
    import test_oracle_dispatch as t_disp
    # read as NVFP4, the MXFP4 row lacks the tensor scale or decodes to other values
    for name in ("mxfp4_two_blocks", "nvfp4_three_blocks"):
        with pytest.raises((AssertionError, ValueError, KeyError)):
            t_disp.test_dequant_dispatch_on_hand_worked_blocks(name)


def test_mutant_bf16_read_as_fp16(monkeypatch):
    import torch
    orig = formats.to_f64

    def to_f64(t):
        if isinstance(t, torch.Tensor) and t.dtype == torch.bfloat16:
            return t.view(torch.float16).numpy().astype(np.float64)
        return orig(t)
    monkeypatch.setattr(formats, "to_f64", to_f64)
    import test_oracle_dispatch as t_disp
    _fails(t_disp.test_to_f64_bf16_bit_patterns)


def test_mutant_expert_source_returns_up_first(monkeypatch):
    def call(self, e):
        c = self.fetch(e)
        return tuple(formats.dequant(c[m], self.wtype) for m in ("up", "gate", "down"))
    monkeypatch.setattr(moe.ExpertSource, "__call__", call)
    import test_oracle_dispatch as t_disp
    _fails(t_disp.test_expert_source_order_values_and_caching)


def test_mutant_prefill_hot_set_ties_to_the_higher_key(monkeypatch):
    import oracle.placement as placement
    import test_oracle_placement as t_pl

    def hot(counts, capacity):
        ranked = sorted((k for k, c in counts.items() if c > 0), key=lambda k: (-counts[k], -k))
        return set(ranked[:capacity])
    monkeypatch.setattr(placement, "prefill_hot_set", hot)
    _fails(t_pl.test_hand_worked_trace)


def test_mutant_static_split_by_expert_instead_of_layer(monkeypatch):
    import oracle.placement as placement
    import test_oracle_placement as t_pl
    monkeypatch.setattr(placement, "static_set", lambda L, E, cap: {(i % L) * E + i // L for i in range(cap)})
    _fails(t_pl.test_hand_worked_trace)
