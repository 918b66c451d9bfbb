// Host expert executor: the AVX-512 form of the weight-row dot products
// (host_simd.cpp).  Internal to libft; not part of the C ABI.
#pragma once

#include <cstdint>

#include "ft.h"

namespace ft {

// True when the CPU has AVX-512F and the form is not switched off.
bool host_simd_supported();
// mode 0 switches the AVX-512 form off, 1 back on where the CPU has it, any
// other value only asks; returns the previous state (1 on, 0 off).
int host_simd_set(int mode);

// One weight row of K elements (K a multiple of 128) in record format wt
// (ft_wtype): fp32 or bf16 values; FP8 e4m3 bytes with one fp32 scale per 128;
// NVFP4 / MXFP4 e2m1 codes, two per byte (element 2b in the low nibble of byte
// b), with one scale byte per 16 (e4m3) / 32 (E8M0) elements, times gscale
// (the NVFP4 matrix scale; 1 otherwise).  e4m3 and E8M0 scale bytes are decoded
// through scale_lut[256].
struct HostRow {
  int wt;
  const uint8_t* vals;
  const uint8_t* scales;
  const float* scale_lut;
  float gscale;
  int K;
};

// True for the formats whose dot products read x in pair-split order.
inline bool host_row_pair_split(int wt) { return wt == FT_W_NVFP4 || wt == FT_W_MXFP4; }

// x of K elements -> pair-split order: within every 32-element group, the 16
// even elements, then the 16 odd ones (the order in which FP4 codes unpack).
void split_pairs32(const float* x, int K, float* out);

// out[j] = sum_k w[k] * x_j[k] for the row w and n vectors xs[j] (pair-split
// order for the FP4 formats, natural order otherwise), each weight decoded as
// in the portable path (value * scale).  AVX-512 only: call it only when
// host_simd_supported().
void host_rows(const HostRow& r, const float* const* xs, int n, float* out);

}  // namespace ft
