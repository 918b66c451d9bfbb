// Host expert executor: the AVX2 and AVX-512 forms of the weight-row dot
// products (host_simd.cpp).  Internal to libft; not part of the C ABI.
#pragma once

#include <cstdint>

#include "ft.h"

namespace ft {

// Forms of the row dot products: the portable decode-then-dot loop (in the
// executor), or host_rows in AVX2+FMA or AVX-512F registers.
enum HostSimd { HOST_PORTABLE = 0, HOST_AVX2 = 1, HOST_AVX512 = 2 };

// The form in use (the best this CPU runs, unless set otherwise).
int host_simd_form();
// True when host_rows is to be used (the form is not the portable one).
bool host_simd_supported();
// mode HOST_PORTABLE / HOST_AVX2 / HOST_AVX512 selects that form where the CPU
// runs it (else the best one below it); any other value only asks.  Returns
// the form in use before the call.
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
// in the portable path (value * scale), in the form host_simd_form() names.
// Call it only when host_simd_supported().
void host_rows(const HostRow& r, const float* const* xs, int n, float* out);

}  // namespace ft
