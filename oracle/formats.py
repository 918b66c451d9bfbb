"""Decoders of the stored expert-weight formats, and the bf16 rounding rule.

The pages name the formats the engine consumes (MXFP4, NVFP4, FP8, BF16:
[Overview] feature table "广泛兼容"; [Review] §3 model table: native MXFP4 and
NVFP4 routed experts) but do not define them.  The definitions used:

* e2m1 (OCP MX v1.0, FP4): 1 sign, 2 exponent (bias 1), 1 mantissa bit;
  exponent 0 is subnormal (0 or 0.5); no inf/NaN; max 6.
* e4m3 "fn" (OCP FP8): 1 sign, 4 exponent (bias 7), 3 mantissa bits;
  exponent 0 subnormal; S.1111.111 is NaN; no inf; max 448.
* E8M0 (OCP MX v1.0 scale): 2^(b - 127); b = 255 is NaN.
* bf16: the upper 16 bits of an IEEE binary32.
* NVFP4: e2m1 values, one e4m3 scale per 16 consecutive K elements, one fp32
  scale per tensor: w = e2m1 * e4m3 * s_tensor.
* MXFP4: e2m1 values, one E8M0 scale per 32 consecutive K elements.
* FP8 (this library's choice): e4m3 values, one fp32 scale per 128
  consecutive K elements of a row.

Decoding here is bit arithmetic written from those definitions; it shares
nothing with the CUDA decoders.
"""
import numpy as np


def e2m1_value(code: int) -> float:
    """Value of one 4-bit e2m1 code."""
    s = -1.0 if (code >> 3) & 1 else 1.0
    e = (code >> 1) & 3
    m = code & 1
    if e == 0:
        return s * 0.5 * m
    return s * 2.0 ** (e - 1) * (1.0 + 0.5 * m)


def e4m3_value(byte: int) -> float:
    """Value of one e4m3 (fn) byte."""
    s = -1.0 if (byte >> 7) & 1 else 1.0
    e = (byte >> 3) & 15
    m = byte & 7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * 2.0 ** (e - 7) * (1.0 + m / 8.0)


def e8m0_value(byte: int) -> float:
    """Value of one E8M0 scale byte."""
    if byte == 255:
        return float("nan")
    return 2.0 ** (byte - 127)


E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
E4M3_TABLE = np.array([e4m3_value(b) for b in range(256)], dtype=np.float64)
E8M0_TABLE = np.array([e8m0_value(b) for b in range(256)], dtype=np.float64)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> fp64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value, ties to even (finite, normal range)."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    nz = (x != 0) & np.isfinite(x)
    a = np.abs(x[nz])
    e = np.floor(np.log2(a))
    # log2 may be off by one at exact powers of two in floating point: fix up
    e = np.where(2.0 ** e > a, e - 1, e)
    e = np.where(2.0 ** (e + 1) <= a, e + 1, e)
    e = np.maximum(e, -126.0)            # bf16 subnormal spacing below 2^-126
    ulp = 2.0 ** (e - 7)
    out[nz] = np.sign(x[nz]) * np.rint(a / ulp) * ulp   # np.rint: half to even
    out[~np.isfinite(x)] = x[~np.isfinite(x)]
    return out


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    """[..., K/2] bytes -> [..., K] 4-bit codes; element 2i is the low nibble of byte i."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def dequant_nvfp4(codes: np.ndarray, scales: np.ndarray, gscale: float) -> np.ndarray:
    """[R, K/2] packed e2m1, [R, K/16] e4m3 scales, fp32 tensor scale -> [R, K] fp64."""
    v = E2M1_TABLE[unpack_nibbles(codes)]
    R, K = v.shape
    s = E4M3_TABLE[np.asarray(scales, dtype=np.uint8)]
    return (v.reshape(R, K // 16, 16) * s[:, :, None]).reshape(R, K) * float(np.float32(gscale))


def dequant_mxfp4(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """[R, K/2] packed e2m1, [R, K/32] E8M0 scales -> [R, K] fp64."""
    v = E2M1_TABLE[unpack_nibbles(codes)]
    R, K = v.shape
    s = E8M0_TABLE[np.asarray(scales, dtype=np.uint8)]
    return (v.reshape(R, K // 32, 32) * s[:, :, None]).reshape(R, K)


def dequant_fp8_rows128(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """[R, K] e4m3 bytes, [R, K/128] fp32 scales -> [R, K] fp64."""
    v = E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]
    R, K = v.shape
    s = np.asarray(scales, dtype=np.float32).astype(np.float64)
    return (v.reshape(R, K // 128, 128) * s[:, :, None]).reshape(R, K)


def to_f64(t) -> np.ndarray:
    """A stored f32 / bf16 tensor (torch or numpy) -> fp64 ndarray, exactly."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu()
            if t.dtype == torch.bfloat16:
                return bf16_bits_to_f64(t.view(torch.int16).numpy().view(np.uint16))
            return t.numpy().astype(np.float64)
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t, dtype=np.float64)


def dequant(component: dict, wtype: int) -> np.ndarray:
    """One stored matrix (as produced by ``synth``) -> fp64 values.

    wtype: 0 f32, 1 bf16, 2 fp8 e4m3 (rows of 128), 3 NVFP4, 4 MXFP4.
    """
    def np_(t):
        try:
            return t.detach().cpu().numpy()
        except AttributeError:
            return np.asarray(t)
    if wtype in (0, 1):
        return to_f64(component["w"])
    if wtype == 2:
        return dequant_fp8_rows128(np_(component["codes"]), np_(component["scales"]))
    if wtype == 3:
        return dequant_nvfp4(np_(component["codes"]), np_(component["scales"]), component["gscale"])
    if wtype == 4:
        return dequant_mxfp4(np_(component["codes"]), np_(component["scales"]))
    raise ValueError(wtype)


# ---------------------------------------------------------------- activation quantisation for FP4 tensor cores
# When the expert weights are NVFP4 or MXFP4, the block-scaled FP4 MMA of the
# tensor cores needs the other operand -- the token rows, and the intermediate
# silu(G) * U before the down product -- in the same format.  The rule (a
# reading of this build: the pages name the weight formats, not how activations
# meet them) quantises each block of consecutive K elements on its own, in fp32
# arithmetic, and the oracle evaluates the layer on the quantised values:
#
#   NVFP4 (blocks of 16):  s = e4m3(amax / 6), rounded to nearest even and
#                          saturated at 448 (tensor scale 1);
#                          q = e2m1(v / s), nearest even, saturated at +-6;
#                          an all-zero block (s = 0) stays zero.
#   MXFP4 (blocks of 32):  s = 2^(floor(log2 amax) - 2) as an E8M0 byte
#                          (OCP MX v1.0 §6.3), clamped to 2^-127 .. 2^127;
#                          q = e2m1(v / s), nearest even, saturated at +-6.
# The value used is q * s.

E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1_round(v: np.ndarray) -> np.ndarray:
    """Nearest e2m1 value of each element (ties to the code with an even mantissa bit), saturated at +-6."""
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), 6.0)
    # distances to every grid point; ties go to the even code index (mantissa bit 0)
    d = np.abs(a[..., None] - E2M1_GRID)
    best = d.min(axis=-1, keepdims=True)
    cand = d == best
    even = cand & (np.arange(8) % 2 == 0)
    idx = np.where(even.any(axis=-1), even.argmax(axis=-1), cand.argmax(axis=-1))
    return np.sign(v) * E2M1_GRID[idx]


def e4m3_round(v: np.ndarray) -> np.ndarray:
    """Nearest e4m3 ("fn") value of non-negative fp32 numbers, ties to even, saturated at 448."""
    v = np.asarray(v, dtype=np.float64)
    vals = E4M3_TABLE[:127]                          # the non-negative finite codes 0x00 .. 0x7E, ascending
    a = np.minimum(v, 448.0)
    hi = np.searchsorted(vals, a, side="left")       # first value >= a
    hi = np.minimum(hi, len(vals) - 1)
    lo = np.maximum(hi - 1, 0)
    dlo, dhi = a - vals[lo], vals[hi] - a
    take_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    out = np.where(a == vals[hi], vals[hi], np.where(take_hi, vals[hi], vals[lo]))
    return out


def quant_act_nvfp4(v: np.ndarray) -> np.ndarray:
    """Rows [..., K] (K a multiple of 16) quantised by the NVFP4 activation rule, as fp64 values."""
    v32 = np.asarray(v, dtype=np.float32)
    shp = v32.shape
    b = v32.reshape(-1, 16)
    amax = np.abs(b).max(axis=1)
    s = e4m3_round((amax / np.float32(6.0)).astype(np.float32))
    s32 = s.astype(np.float32)
    safe = np.where(s32 > 0, s32, np.float32(1.0))
    q = e2m1_round((b / safe[:, None]).astype(np.float32))
    q = np.where(s32[:, None] > 0, q, 0.0)
    return (q * s[:, None]).reshape(shp)


def quant_act_mxfp4(v: np.ndarray) -> np.ndarray:
    """Rows [..., K] (K a multiple of 32) quantised by the MXFP4 activation rule, as fp64 values."""
    v32 = np.asarray(v, dtype=np.float32)
    shp = v32.shape
    b = v32.reshape(-1, 32).astype(np.float64)
    amax = np.abs(b).max(axis=1)
    e = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 2.0, -127.0)
    # log2 of an exact power of two is exact; guard the floor against representation error
    e = np.where(2.0 ** (e + 2) > amax, e - 1, e)
    e = np.where(2.0 ** (e + 3) <= amax, e + 1, e)
    e = np.clip(e, -127.0, 127.0)
    s = 2.0 ** e
    q = e2m1_round(b / s[:, None])
    return (q * s[:, None]).reshape(shp)
