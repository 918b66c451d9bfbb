"""Pins of the oracle's format dispatch, its exact tensor conversion and its expert source.

``formats.dequant`` picks a decoder by the stored-format code, ``formats.to_f64``
turns stored bf16 / fp32 tensors into fp64, and ``moe.ExpertSource`` decodes an
expert's (gate, up, down).  Each is checked against values worked out by hand
from the format definitions (tests/golden/format_blocks_handworked.txt, which
cites them) or against bit patterns whose values are fixed by IEEE 754 and the
bf16 definition, so that a swapped dispatch code, a bf16 tensor read as fp16,
or gate and up handed out in the wrong order fails here on the CPU.
"""
import math
import os

import numpy as np
import pytest
import torch

from conftest import GOLDEN
from oracle import formats, moe


def _blocks():
    out, cur = {}, None
    with open(os.path.join(GOLDEN, "format_blocks_handworked.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            w = line.split()
            if w[0] == "begin":
                cur = {"wtype": int(w[2]), "K": int(w[3]), "expect": []}
                out[w[1]] = cur
            elif w[0] == "end":
                cur = None
            elif w[0] == "codes":
                if w[1] == "cycle8":
                    cur["codes"] = [int(b, 16) for b in w[2:]] * (cur["K"] // 8)
                else:
                    cur["codes"] = [int(c) for c in w[1:]]
            elif w[0] == "scales":
                cur["scales"] = w[1:]
            elif w[0] == "gscale":
                cur["gscale"] = float(w[1])
            elif w[0] == "expect":
                if w[1] == "cycle8":
                    cur["expect"] += [float(v) for v in w[3:]] * 16
                else:
                    cur["expect"] += [float(v) for v in w[1:]]
    return out


BLOCKS = _blocks()


def _component(b):
    """The stored component of one row, in the shapes ``synth``'s quantisers produce."""
    wt, K = b["wtype"], b["K"]
    if wt in (3, 4):
        c = np.array(b["codes"], dtype=np.uint8)
        assert c.size == K and c.max() < 16
        packed = (c[0::2] | (c[1::2] << 4)).astype(np.uint8).reshape(1, K // 2)
        sc = np.array([int(s, 16) for s in b["scales"]], dtype=np.uint8).reshape(1, -1)
        comp = {"codes": torch.from_numpy(packed), "scales": torch.from_numpy(sc)}
        if wt == 3:
            comp["gscale"] = b["gscale"]
        return comp
    codes = np.array(b["codes"], dtype=np.uint8).reshape(1, K)
    sc = np.array([float(s) for s in b["scales"]], dtype=np.float32).reshape(1, -1)
    return {"codes": torch.from_numpy(codes), "scales": torch.from_numpy(sc)}


def _same(got, want):
    got, want = np.asarray(got, np.float64).reshape(-1), np.asarray(want, np.float64).reshape(-1)
    assert got.shape == want.shape
    assert np.array_equal(got, want), np.flatnonzero(got != want)[:8]
    # signed zeros are part of the format (code 8 is -0)
    assert np.array_equal(np.signbit(got), np.signbit(want))


@pytest.mark.parametrize("name", sorted(BLOCKS))
def test_dequant_dispatch_on_hand_worked_blocks(name):
    b = BLOCKS[name]
    assert len(b["expect"]) == b["K"]
    _same(formats.dequant(_component(b), b["wtype"]), b["expect"])


def test_dequant_dispatch_rejects_a_format_read_as_another():
    # an MXFP4 row handed to the NVFP4 code (or the reverse) cannot give the hand-worked values
    mx, nv = BLOCKS["mxfp4_two_blocks"], BLOCKS["nvfp4_three_blocks"]
    c = _component(mx)
    c["gscale"] = 1.0
    try:
        got = formats.dequant(c, 3)
        assert got.shape != (1, mx["K"]) or not np.array_equal(got.reshape(-1), np.array(mx["expect"]))
    except (ValueError, IndexError):
        pass
    c = _component(nv)
    try:
        got = formats.dequant(c, 4)
        assert got.shape != (1, nv["K"]) or not np.array_equal(got.reshape(-1), np.array(nv["expect"]))
    except (ValueError, IndexError):
        pass
    with pytest.raises(ValueError):
        formats.dequant(c, 7)


def test_dequant_plain_formats():
    # f32 and bf16 components are the stored values themselves
    w32 = torch.tensor([[1.5, -0.1, 3.0e38, -0.0]], dtype=torch.float32)
    got = formats.dequant({"w": w32}, 0)
    _same(got, [1.5, float(np.float32(-0.1)), float(np.float32(3.0e38)), -0.0])
    bits = torch.tensor([[0x3F80, 0xC040, 0x3F81, 0x3C00]], dtype=torch.int32).to(torch.int16)
    got = formats.dequant({"w": bits.view(torch.bfloat16)}, 1)
    _same(got, [1.0, -3.0, 1.0078125, 0.0078125])


def test_to_f64_bf16_bit_patterns():
    # bf16 = the upper half of an IEEE binary32: sign, 8 exponent bits (bias 127), 7 mantissa bits
    pats = [0x3F80, 0xC040, 0x3F81, 0x3C00, 0x0001, 0x7F7F, 0x8000, 0x4049]
    want = [1.0, -3.0, 1.0 + 2.0 ** -7, 2.0 ** -7, 2.0 ** -133, (2.0 - 2.0 ** -7) * 2.0 ** 127, -0.0,
            2.0 * (1.0 + 73.0 / 128.0)]
    t = torch.tensor(pats, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    got = formats.to_f64(t)
    assert got.dtype == np.float64
    _same(got, want)
    # 0x3C00 read as fp16 would be 1.0: the two 16-bit formats must not be confused
    assert got[3] != 1.0


def test_to_f64_fp32_and_numpy_inputs():
    # fp32 values convert exactly: 0.1f is 13421773 * 2^-27
    t = torch.tensor([0.1, -2.5, 1e-45], dtype=torch.float32)
    got = formats.to_f64(t)
    _same(got, [13421773 * 2.0 ** -27, -2.5, 2.0 ** -149])
    _same(formats.to_f64(np.array([0.1], dtype=np.float32)), [13421773 * 2.0 ** -27])
    _same(formats.to_f64([1, 2]), [1.0, 2.0])
    # a tensor that requires grad or lives in a view is read the same way
    v = torch.arange(8, dtype=torch.float32).reshape(2, 4)[:, 1::2]
    _same(formats.to_f64(v), [1.0, 3.0, 5.0, 7.0])


def test_expert_source_order_values_and_caching():
    calls = []

    def bf16(vals):
        return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)

    def fetch(e):
        calls.append(e)
        return {"gate": {"w": bf16([[1.0 + e, 2.0]])}, "up": {"w": bf16([[-4.0, 0.5 * e]])},
                "down": {"w": bf16([[8.0], [16.0 + e]])}}

    src = moe.ExpertSource(fetch, 1)
    g, u, d = src(3)
    _same(g, [4.0, 2.0])
    _same(u, [-4.0, 1.5])
    _same(d, [8.0, 19.0])
    assert g.shape == (1, 2) and u.shape == (1, 2) and d.shape == (2, 1)
    src(3)
    src(5)
    src(3)
    assert calls == [3, 5]


def test_expert_source_decodes_through_the_dispatch():
    nv = BLOCKS["nvfp4_three_blocks"]
    comp = _component(nv)
    src = moe.ExpertSource(lambda e: {"gate": comp, "up": comp, "down": comp}, 3)
    for m in src(0):
        _same(m, nv["expect"])
    assert math.isclose(float(np.abs(src(0)[0]).max()), 9.0)
