// Host expert executor: weight rows decoded and dotted with the tokens in
// AVX-512 registers.  Compiled by the host compiler (not nvcc's front end) into
// libft.so; every AVX-512 function carries its own target attribute and runs
// only after host_simd_supported() said yes, so the library still loads and
// runs on x86-64 CPUs without AVX-512 (the executor then keeps its portable
// decode-then-dot loop).
#include "host_simd.h"

#include <immintrin.h>

#include <atomic>
#include <cmath>

namespace ft {

namespace {

// e2m1 code -> value: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0;
// exponent 0 gives 0 or 0.5.
float e2m1_value(int c) {
  const float s = (c & 8) ? -1.0f : 1.0f;
  const int e = (c >> 1) & 3, m = c & 1;
  return e == 0 ? s * 0.5f * m : s * std::ldexp(1.0f + 0.5f * m, e - 1);
}

// 0: not yet asked, 1: AVX-512F present and allowed, 2: absent or switched off
std::atomic<int> g_simd{0};

int detect() {
#if defined(__x86_64__)
  __builtin_cpu_init();
  return __builtin_cpu_supports("avx512f") ? 1 : 2;
#else
  return 2;
#endif
}

}  // namespace

bool host_simd_supported() {
  int s = g_simd.load(std::memory_order_relaxed);
  if (s == 0) {
    s = detect();
    g_simd.store(s, std::memory_order_relaxed);
  }
  return s == 1;
}

int host_simd_set(int mode) {
  const int prev = host_simd_supported() ? 1 : 0;
  if (mode == 0) g_simd.store(2, std::memory_order_relaxed);
  if (mode == 1) g_simd.store(detect(), std::memory_order_relaxed);
  return prev;
}

void split_pairs32(const float* x, int K, float* out) {
  for (int g = 0; g < K; g += 32)
    for (int l = 0; l < 16; ++l) {
      out[g + l] = x[g + 2 * l];
      out[g + 16 + l] = x[g + 2 * l + 1];
    }
}

#if defined(__x86_64__)
namespace {

#define FT_AVX512 __attribute__((target("avx512f")))

// Accumulators per token: independent FMA chains, so that one token's sums
// are not bound by the FMA latency.
constexpr int NACC = 4;

// n <= 4 tokens over the row: w16(k0) gives the 16 decoded weights at k0
// (k0 a multiple of 16), which meet x_j[k0 .. k0+15]; step u of every 64
// elements goes to accumulator u.
template <typename W16>
FT_AVX512 inline void dot_rows(int K, const float* const* xs, int nj, __m512 (*acc)[NACC], const W16& w16) {
  for (int k0 = 0; k0 < K; k0 += 16 * NACC) {
#pragma GCC unroll 4
    for (int u = 0; u < NACC; ++u) {
      const __m512 w = w16(k0 + 16 * u);
      for (int j = 0; j < nj; ++j) acc[j][u] = _mm512_fmadd_ps(w, _mm512_loadu_ps(xs[j] + k0 + 16 * u), acc[j][u]);
    }
  }
}

// e4m3 bytes (widened to 32 bits) -> fp32: sign, exponent (bias 7) and
// mantissa moved into place; exponent 0 is m * 2^-9; S.1111.111 is NaN.
FT_AVX512 inline __m512 e4m3_lanes(__m512i b) {
  const __m512i mag = _mm512_and_si512(b, _mm512_set1_epi32(0x7F));
  const __m512i sign = _mm512_slli_epi32(_mm512_and_si512(b, _mm512_set1_epi32(0x80)), 24);
  const __m512i normal = _mm512_add_epi32(_mm512_slli_epi32(mag, 20), _mm512_set1_epi32(120 << 23));
  const __m512 sub = _mm512_mul_ps(_mm512_cvtepi32_ps(_mm512_and_si512(b, _mm512_set1_epi32(7))),
                                   _mm512_set1_ps(1.0f / 512.0f));
  __m512 v = _mm512_mask_mov_ps(_mm512_castsi512_ps(normal), _mm512_cmplt_epi32_mask(mag, _mm512_set1_epi32(8)), sub);
  v = _mm512_castsi512_ps(_mm512_or_si512(_mm512_castps_si512(v), sign));
  return _mm512_mask_mov_ps(v, _mm512_cmpeq_epi32_mask(mag, _mm512_set1_epi32(0x7F)), _mm512_set1_ps(NAN));
}

struct W16F32 {
  const float* v;
  FT_AVX512 __m512 operator()(int k0) const { return _mm512_loadu_ps(v + k0); }
};

struct W16BF16 {
  const uint16_t* v;
  FT_AVX512 __m512 operator()(int k0) const {
    const __m512i w = _mm512_cvtepu16_epi32(_mm256_loadu_si256(reinterpret_cast<const __m256i*>(v + k0)));
    return _mm512_castsi512_ps(_mm512_slli_epi32(w, 16));
  }
};

struct W16FP8 {
  const uint8_t* v;
  const float* sc;  // one scale per 128 elements
  FT_AVX512 __m512 operator()(int k0) const {
    const __m512i b = _mm512_cvtepu8_epi32(_mm_loadu_si128(reinterpret_cast<const __m128i*>(v + k0)));
    return _mm512_mul_ps(e4m3_lanes(b), _mm512_set1_ps(sc[k0 >> 7]));
  }
};

FT_AVX512 void host_rows_avx512(const HostRow& r, const float* const* xs, int n, float* out) {
  alignas(64) float lut_v[16];
  for (int c = 0; c < 16; ++c) lut_v[c] = e2m1_value(c);
  const __m512 lut = _mm512_load_ps(lut_v);
  const __m512i low4 = _mm512_set1_epi32(15);
  for (int j0 = 0; j0 < n; j0 += 4) {
    const int nj = n - j0 < 4 ? n - j0 : 4;
    const float* const* x = xs + j0;
    __m512 acc[4][NACC];
    for (int j = 0; j < 4; ++j)
      for (int u = 0; u < NACC; ++u) acc[j][u] = _mm512_setzero_ps();
    switch (r.wt) {
      case FT_W_F32:
        dot_rows(r.K, x, nj, acc, W16F32{reinterpret_cast<const float*>(r.vals)});
        break;
      case FT_W_BF16:
        dot_rows(r.K, x, nj, acc, W16BF16{reinterpret_cast<const uint16_t*>(r.vals)});
        break;
      case FT_W_FP8E4M3:
        dot_rows(r.K, x, nj, acc, W16FP8{r.vals, reinterpret_cast<const float*>(r.scales)});
        break;
      default: {  // NVFP4, MXFP4: 32 elements (16 code bytes) per group, x in pair-split order
        const bool mx = r.wt == FT_W_MXFP4;
        for (int g0 = 0; g0 < r.K / 32; g0 += 2) {
#pragma GCC unroll 2
          for (int u = 0; u < 2; ++u) {
            const int g = g0 + u;
            // the block scale goes into the 16-entry table once per group
            __m512 sl;
            if (mx) {
              sl = _mm512_mul_ps(lut, _mm512_set1_ps(r.scale_lut[r.scales[g]] * r.gscale));
            } else {
              sl = lut;
            }
            const __m512i b = _mm512_cvtepu8_epi32(_mm_loadu_si128(reinterpret_cast<const __m128i*>(r.vals + 16 * g)));
            __m512 ve = _mm512_permutexvar_ps(_mm512_and_si512(b, low4), sl);   // elements 2b
            __m512 vo = _mm512_permutexvar_ps(_mm512_srli_epi32(b, 4), sl);     // elements 2b+1
            if (!mx) {
              // two 16-element blocks: lanes 0-7 (bytes 0-7) the first, lanes 8-15 the second
              const __m512 sc = _mm512_mask_mov_ps(_mm512_set1_ps(r.scale_lut[r.scales[2 * g]] * r.gscale),
                                                   (__mmask16)0xFF00,
                                                   _mm512_set1_ps(r.scale_lut[r.scales[2 * g + 1]] * r.gscale));
              ve = _mm512_mul_ps(ve, sc);
              vo = _mm512_mul_ps(vo, sc);
            }
            for (int j = 0; j < nj; ++j) {
              acc[j][2 * u] = _mm512_fmadd_ps(ve, _mm512_loadu_ps(x[j] + 32 * g), acc[j][2 * u]);
              acc[j][2 * u + 1] = _mm512_fmadd_ps(vo, _mm512_loadu_ps(x[j] + 32 * g + 16), acc[j][2 * u + 1]);
            }
          }
        }
        break;
      }
    }
    for (int j = 0; j < nj; ++j)
      out[j0 + j] = _mm512_reduce_add_ps(_mm512_add_ps(_mm512_add_ps(acc[j][0], acc[j][1]),
                                                       _mm512_add_ps(acc[j][2], acc[j][3])));
  }
}

}  // namespace
#endif

void host_rows(const HostRow& r, const float* const* xs, int n, float* out) {
#if defined(__x86_64__)
  host_rows_avx512(r, xs, n, out);
#else
  (void)r; (void)xs; (void)n; (void)out;
#endif
}

}  // namespace ft
