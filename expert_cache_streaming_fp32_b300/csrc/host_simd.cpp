// Host expert executor, FP4 rows: decode and dot product fused in AVX-512
// registers.  Compiled by the host compiler (not nvcc's front end) into
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
__attribute__((target("avx512f")))
static void fp4_rows_avx512(const Fp4Row& r, const float* const* xs, int n, float* out) {
  alignas(64) float lut_v[16];
  for (int c = 0; c < 16; ++c) lut_v[c] = e2m1_value(c);
  const __m512 lut = _mm512_load_ps(lut_v);
  const __m512i low4 = _mm512_set1_epi32(15);
  const int groups = r.K / 32;
  for (int j0 = 0; j0 < n; j0 += 4) {
    const int nj = n - j0 < 4 ? n - j0 : 4;
    __m512 acc[4] = {_mm512_setzero_ps(), _mm512_setzero_ps(), _mm512_setzero_ps(), _mm512_setzero_ps()};
    for (int g = 0; g < groups; ++g) {
      // 16 code bytes: byte b holds elements 2b (low nibble) and 2b+1 (high nibble)
      const __m512i b = _mm512_cvtepu8_epi32(_mm_loadu_si128(reinterpret_cast<const __m128i*>(r.codes + 16 * g)));
      __m512 ve = _mm512_permutexvar_ps(_mm512_and_si512(b, low4), lut);
      __m512 vo = _mm512_permutexvar_ps(_mm512_srli_epi32(b, 4), lut);
      __m512 sc;
      if (r.block == 32) {
        sc = _mm512_set1_ps(r.scale_lut[r.scales[g]] * r.gscale);
      } else {
        // two 16-element blocks: lanes 0-7 (bytes 0-7) the first, lanes 8-15 the second
        sc = _mm512_mask_mov_ps(_mm512_set1_ps(r.scale_lut[r.scales[2 * g]] * r.gscale), (__mmask16)0xFF00,
                                _mm512_set1_ps(r.scale_lut[r.scales[2 * g + 1]] * r.gscale));
      }
      ve = _mm512_mul_ps(ve, sc);
      vo = _mm512_mul_ps(vo, sc);
      for (int j = 0; j < nj; ++j) {
        const float* x = xs[j0 + j] + 32 * g;
        acc[j] = _mm512_fmadd_ps(ve, _mm512_loadu_ps(x), acc[j]);
        acc[j] = _mm512_fmadd_ps(vo, _mm512_loadu_ps(x + 16), acc[j]);
      }
    }
    for (int j = 0; j < nj; ++j) out[j0 + j] = _mm512_reduce_add_ps(acc[j]);
  }
}
#endif

void fp4_rows(const Fp4Row& r, const float* const* xs, int n, float* out) {
#if defined(__x86_64__)
  fp4_rows_avx512(r, xs, n, out);
#else
  (void)r; (void)xs; (void)n; (void)out;
#endif
}

}  // namespace ft
