"""Pins of the oracle's activation quantisation for the FP4 tensor-core path.

e2m1 and e4m3 rounding are checked against hand-listed values (every midpoint
of the e2m1 grid, saturation, signs) and against torch's float8_e4m3fn
conversion as a library routine; the NVFP4 and MXFP4 block rules against
blocks worked out by hand from the rule's statement in oracle/formats.py.
"""
import numpy as np
import pytest
import torch

from oracle import formats


# (input, nearest e2m1 value with ties to the even code: codes 0, 2, 4, 6 are even)
E2M1_CASES = [
    (0.0, 0.0), (0.24, 0.0), (0.25, 0.0), (0.26, 0.5), (0.5, 0.5), (0.75, 1.0), (1.0, 1.0), (1.25, 1.0),
    (1.5, 1.5), (1.75, 2.0), (2.0, 2.0), (2.5, 2.0), (2.51, 3.0), (3.0, 3.0), (3.5, 4.0), (4.0, 4.0),
    (5.0, 4.0), (5.01, 6.0), (6.0, 6.0), (7.0, 6.0), (1e9, 6.0), (-0.75, -1.0), (-2.5, -2.0), (-7.0, -6.0),
]


def test_e2m1_round_hand_values():
    x = np.array([c[0] for c in E2M1_CASES])
    want = np.array([c[1] for c in E2M1_CASES])
    assert np.array_equal(formats.e2m1_round(x), want)


def test_e4m3_round_matches_library_conversion():
    rng = np.random.default_rng(0)
    vals = formats.E4M3_TABLE[:127]
    mids = (vals[:-1] + vals[1:]) / 2.0                      # every tie between neighbouring codes
    x = np.concatenate([vals, mids, rng.uniform(0, 448, 20000), 2.0 ** rng.uniform(-12, 8, 20000)])
    x = x.astype(np.float32)
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(formats.e4m3_round(x), lib)
    assert formats.e4m3_round(np.array([500.0, 1e6], dtype=np.float32)).tolist() == [448.0, 448.0]


def test_nvfp4_activation_block_by_hand():
    # amax 6 -> s = e4m3(1.0) = 1: values round on the e2m1 grid
    b = np.array([0.3, -1.7, 6.0, 2.4, 0.0, -0.25, 0.75, 5.0, 3.2, -4.4, 1.2, 0.1, -6.0, 2.6, 1.75, 0.6],
                 dtype=np.float32)
    want = [0.5, -1.5, 6.0, 2.0, 0.0, -0.0, 1.0, 4.0, 3.0, -4.0, 1.0, 0.0, -6.0, 3.0, 2.0, 0.5]
    assert np.array_equal(formats.quant_act_nvfp4(b[None, :])[0], np.array(want))
    # amax 1.3 -> 1.3 / 6 = 0.21667 -> e4m3 0.21875 (2^-3 * 1.75); 1.3 / 0.21875 = 5.94 -> 6 -> 1.3125
    b2 = np.zeros(16, dtype=np.float32)
    b2[0], b2[1] = 1.3, 0.3
    got = formats.quant_act_nvfp4(b2[None, :])[0]
    assert got[0] == 6.0 * 0.21875 and got[1] == 1.5 * 0.21875      # 0.3 / 0.21875 = 1.37 -> 1.5
    # an all-zero block stays zero; a huge block saturates the scale at 448 and the values at 6 * 448
    assert not formats.quant_act_nvfp4(np.zeros((1, 16), np.float32)).any()
    big = np.full((1, 16), 5000.0, dtype=np.float32)
    assert np.all(formats.quant_act_nvfp4(big) == 6.0 * 448.0)


def test_mxfp4_activation_block_by_hand():
    b = np.zeros(32, dtype=np.float32)
    b[:4] = [5.0, -0.3, 2.6, 1.2]           # amax 5: floor(log2 5) - 2 = 0, s = 1
    assert formats.quant_act_mxfp4(b[None, :])[0][:4].tolist() == [4.0, -0.5, 3.0, 1.0]
    b[:4] = [4.0, 1.1, 0.0, -3.0]           # amax exactly 4: log2 = 2, s = 1
    assert formats.quant_act_mxfp4(b[None, :])[0][:4].tolist() == [4.0, 1.0, 0.0, -3.0]
    b[:4] = [0.1, 0.05, -0.02, 0.0]         # amax 0.1: floor(log2 0.1) = -4, s = 2^-6; 6.4 -> 6, 3.2 -> 3, 1.28 -> 1.5
    got = formats.quant_act_mxfp4(b[None, :])[0][:4]
    assert got.tolist() == [6.0 / 64, 3.0 / 64, -1.5 / 64, 0.0]
    assert not formats.quant_act_mxfp4(np.zeros((1, 32), np.float32)).any()


def test_quantised_values_are_representable_and_close():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(64, 256)).astype(np.float32)
    grid = np.concatenate([-formats.E2M1_GRID, formats.E2M1_GRID])
    for fn, blk in ((formats.quant_act_nvfp4, 16), (formats.quant_act_mxfp4, 32)):
        q = fn(x)
        assert q.shape == x.shape
        rel = np.linalg.norm(q - x) / np.linalg.norm(x)
        assert 0.02 < rel < 0.2                      # four bits per element
        xb, qb = x.reshape(-1, blk), q.reshape(-1, blk)
        amax = np.abs(xb).max(axis=1)
        if blk == 16:
            sc = formats.e4m3_round((amax / np.float32(6.0)).astype(np.float32))
        else:
            sc = 2.0 ** (np.floor(np.log2(amax)) - 2)
        # every block is e2m1 values times its one scale
        assert np.all(np.isin(qb / sc[:, None], grid))
