"""Pins of the format decoders (exhaustive), the bf16 rounding rule, the q* split and the stream time model."""
import math

import numpy as np
import pytest
import torch

from conftest import read_golden
from oracle import formats, qsplit, stream
import synth


def test_e2m1_all_codes_match_ocp_table():
    rows = read_golden("e2m1_ocp_table.txt")
    assert len(rows) == 16
    for code, val in rows:
        v = formats.e2m1_value(int(code))
        assert v == float(val) and math.copysign(1, v) == math.copysign(1, float(val))


def test_e4m3_all_bytes_match_library_conversion():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for b in range(256):
        v = formats.e4m3_value(b)
        if math.isnan(ref[b]):
            assert math.isnan(v)
        else:
            assert v == ref[b], b
    assert formats.e4m3_value(0x7E) == 448.0


def test_e8m0_all_bytes():
    for b in range(255):
        assert formats.e8m0_value(b) == math.ldexp(1.0, b - 127)
    assert math.isnan(formats.e8m0_value(255))


def test_bf16_decode_and_rounding_match_library():
    rng = np.random.default_rng(0)
    x32 = (rng.normal(size=20000) * 10.0 ** rng.integers(-6, 6, size=20000)).astype(np.float32)
    x32[:4] = [1.0, -2.0, 0.0, 3.0e38]
    t = torch.from_numpy(x32).to(torch.bfloat16)
    bits = t.view(torch.int16).numpy().view(np.uint16)
    dec = formats.bf16_bits_to_f64(bits)
    assert np.array_equal(dec, t.to(torch.float64).numpy())
    # fp32-exact inputs: one rounding, so ours must equal the library's fp32 -> bf16 RNE
    finite = np.isfinite(dec)
    ours = formats.round_to_bf16(x32.astype(np.float64))
    assert np.array_equal(ours[finite], dec[finite])


def test_bf16_rounding_ties_to_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties to even (1.0)
    assert formats.round_to_bf16(np.array([1.0 + 2 ** -8]))[0] == 1.0
    # 1 + 3*2^-8 is halfway between 1+2^-7 (odd) and 1+2^-6 (even)
    assert formats.round_to_bf16(np.array([1.0 + 3 * 2 ** -8]))[0] == 1.0 + 2 ** -6
    assert formats.round_to_bf16(np.array([-(1.0 + 2 ** -8 + 2 ** -30)]))[0] == -(1.0 + 2 ** -7)


def test_nibble_order():
    packed = np.array([[0x21, 0xF0]], dtype=np.uint8)
    assert formats.unpack_nibbles(packed).tolist() == [[1, 2, 0, 15]]


def _roundtrip_error_bound(w, deq, block, scale_of_block):
    """|w - deq| per element must be within half an e2m1 step (or the saturation gap) times the block scale."""
    R, K = w.shape
    err = np.abs(w - deq).reshape(R, K // block, block)
    return np.all(err <= 2.0 * scale_of_block[:, :, None] + 1e-12)


def test_mxfp4_roundtrip_of_generator_quantiser():
    w = synth.normal((8, 64), 0.02, 123)
    codes, sc = synth.quant_mxfp4(w)
    deq = formats.dequant_mxfp4(codes.numpy(), sc.numpy())
    w64 = w.double().numpy()
    scale = formats.E8M0_TABLE[sc.numpy()]
    assert _roundtrip_error_bound(w64, deq, 32, scale)
    # relative quality of a 4-bit format on Gaussian data
    assert np.linalg.norm(deq - w64) / np.linalg.norm(w64) < 0.2
    # a misread nibble order or scale index shows up as a far larger error
    bad = formats.E2M1_TABLE[formats.unpack_nibbles(codes.numpy())[:, ::-1]]
    assert np.linalg.norm(bad * np.repeat(scale, 32, axis=1) - w64) > 3 * np.linalg.norm(deq - w64)


def test_nvfp4_roundtrip_of_generator_quantiser():
    w = synth.normal((8, 64), 0.02, 321)
    codes, sc, g = synth.quant_nvfp4(w)
    deq = formats.dequant_nvfp4(codes.numpy(), sc.numpy(), g)
    w64 = w.double().numpy()
    scale = formats.E4M3_TABLE[sc.numpy()] * g
    assert _roundtrip_error_bound(w64, deq, 16, scale / 2.0 + 1e-30)
    assert np.linalg.norm(deq - w64) / np.linalg.norm(w64) < 0.15


def test_fp8_roundtrip_of_generator_quantiser():
    w = synth.normal((4, 256), 0.02, 7)
    codes, sc = synth.quant_fp8_rows128(w)
    deq = formats.dequant_fp8_rows128(codes.numpy(), sc.numpy())
    w64 = w.double().numpy()
    # e4m3 has 3 mantissa bits: relative error <= 2^-4 per element above the subnormal range
    rel = np.abs(deq - w64) / np.maximum(np.abs(w64), 1e-3 * np.abs(w64).max())
    assert rel.max() <= 2 ** -4 + 1e-9


# ------------------------------------------------------------------ q*

def test_qsplit_table1_worked_values():
    ms = [1, 2, 3, 4, 6, 8, 16]
    rows = read_golden("table1_bandwidths.txt")
    assert len(rows) == 6
    for name, bp, bh, *qs in rows:
        for m, q in zip(ms, qs):
            assert qsplit.qsplit(m, float(bp), float(bh)) == int(q), (name, m)


def test_qsplit_balance_equation():
    # at the unrounded q*, the fill branch and the host branch take the same time
    S = 6.29e6
    for bp, bh in [(52.7, 77.3), (11.8, 47.5), (51.5, 178.0)]:
        for m in [1, 5, 17, 256]:
            q = qsplit.q_star_real(m, bp, bh)
            assert qsplit.t_fill(q, S, bp) == pytest.approx(qsplit.t_cpu(m - q, S, bp, bh), rel=1e-12)


def test_qsplit_limits():
    assert qsplit.qsplit(0, 10.0, 50.0) == 0
    for m in [1, 2, 7, 100]:
        assert qsplit.qsplit(m, 50.0, 50.0) == m        # B_H -> B_P: fill every miss
        assert qsplit.qsplit(m, 60.0, 50.0) == m        # B_R = 0
        assert qsplit.qsplit(m, 1e-9, 50.0) == 1        # always fill at least one
        assert qsplit.qsplit(m, 49.999999, 50.0) == m
    assert qsplit.residual_bandwidth(60.0, 50.0) == 0.0
    # half-up rounding: 0.5 * 3 = 1.5 -> 2; 0.5 * 5 = 2.5 -> 3
    assert qsplit.qsplit_ratio(3, 0.5) == 2 and qsplit.qsplit_ratio(5, 0.5) == 3


# ------------------------------------------------------------------ streaming time model

def test_prefill_stream_numbers_from_the_page():
    g = {r[0]: float(r[1]) for r in read_golden("prefill_stream_numbers.txt")}
    t = stream.link_bound_time(g["pool_gb"] * 1e9, g["link_gbs"] * 1e9)
    assert g["chunk_s_low"] <= round(t, 2) <= g["chunk_s_high"]
    tok_s = g["prompt_tokens_16k"] / (2 * t)
    assert abs(tok_s - g["tok_per_s_16k"]) / g["tok_per_s_16k"] < 0.01


def test_stream_overlap_model():
    c = [3.0] * 5
    p = [1.0] * 5
    assert stream.serialized_time(c, p) == 20.0
    assert stream.overlapped_time(c, p) == 16.0          # copy-bound: 5 copies + last compute
    assert stream.overlapped_time([1.0] * 4, [2.0] * 4) == 9.0   # compute-bound: first copy + 4 computes
    # two buffers only: layer 2's copy reuses layer 0's buffer and waits for its compute (t = 6)
    assert stream.overlapped_time([1.0, 1.0, 1.0], [5.0, 0.1, 0.1]) == pytest.approx(7.1)
