// Host expert executor: the AVX-512 form of the FP4 row dot products
// (host_simd.cpp).  Internal to libft; not part of the C ABI.
#pragma once

#include <cstdint>

namespace ft {

// True when the CPU has AVX-512F and the form is not switched off.
bool host_simd_supported();
// mode 0 switches the AVX-512 form off, 1 back on where the CPU has it, any
// other value only asks; returns the previous state (1 on, 0 off).
int host_simd_set(int mode);

// One FP4 weight row: K elements (K a multiple of 32), two e2m1 codes per byte
// (element 2b in the low nibble of byte b), one scale byte per `block`
// elements (32: E8M0, MXFP4; 16: e4m3, NVFP4) decoded through scale_lut[256],
// times gscale (the NVFP4 matrix scale; 1 for MXFP4).
struct Fp4Row {
  const uint8_t* codes;
  const uint8_t* scales;
  const float* scale_lut;
  float gscale;
  int K, block;
};

// x of K elements -> the pair-split order the FP4 dot products read: within
// every 32-element group, the 16 even elements, then the 16 odd ones.
void split_pairs32(const float* x, int K, float* out);

// out[j] = sum_k w[k] * x_j[k] for the row w and n vectors xs[j] in pair-split
// order, each weight decoded as e2m1 * (scale * gscale).  AVX-512 only: call it
// only when host_simd_supported().
void fp4_rows(const Fp4Row& r, const float* const* xs, int n, float* out);

}  // namespace ft
