// Host expert executor: weight rows decoded and dotted with the tokens in
// AVX-512 or AVX2 registers.  Compiled by the host compiler (not nvcc's front
// end) into libft.so; every vector function carries its own target attribute
// and runs only in the form the CPU reported, so the library still loads and
// runs on any x86-64 CPU (without AVX2 the executor keeps its portable
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

// The form in use: -1 not yet chosen, else a HostSimd value.
std::atomic<int> g_form{-1};

// The best form this CPU runs.
int best_form() {
#if defined(__x86_64__)
  __builtin_cpu_init();
  if (__builtin_cpu_supports("avx512f")) return HOST_AVX512;
  if (__builtin_cpu_supports("avx2") && __builtin_cpu_supports("fma")) return HOST_AVX2;
#endif
  return HOST_PORTABLE;
}

}  // namespace

int host_simd_form() {
  int f = g_form.load(std::memory_order_relaxed);
  if (f < 0) {
    f = best_form();
    g_form.store(f, std::memory_order_relaxed);
  }
  return f;
}

bool host_simd_supported() { return host_simd_form() != HOST_PORTABLE; }

int host_simd_set(int mode) {
  const int prev = host_simd_form();
  const int best = best_form();
  if (mode == HOST_PORTABLE) g_form.store(HOST_PORTABLE, std::memory_order_relaxed);
  if (mode == HOST_AVX2) g_form.store(best >= HOST_AVX2 ? HOST_AVX2 : HOST_PORTABLE, std::memory_order_relaxed);
  if (mode == HOST_AVX512) g_form.store(best >= HOST_AVX512 ? HOST_AVX512 : best, std::memory_order_relaxed);
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

// ---- AVX2 + FMA: the same steps in 8 lanes.  e2m1 codes take their magnitude
// from an 8-entry register table and their sign from bit 3; two tokens per
// pass keep the 8 accumulators and the operands within the 16 registers.
#define FT_AVX2 __attribute__((target("avx2,fma")))

template <typename W8>
FT_AVX2 inline void dot_rows8(int K, const float* const* xs, int nj, __m256 (*acc)[NACC], const W8& w8) {
  for (int k0 = 0; k0 < K; k0 += 8 * NACC) {
#pragma GCC unroll 4
    for (int u = 0; u < NACC; ++u) {
      const __m256 w = w8(k0 + 8 * u);
      for (int j = 0; j < nj; ++j) acc[j][u] = _mm256_fmadd_ps(w, _mm256_loadu_ps(xs[j] + k0 + 8 * u), acc[j][u]);
    }
  }
}

FT_AVX2 inline __m256 e4m3_lanes8(__m256i b) {
  const __m256i mag = _mm256_and_si256(b, _mm256_set1_epi32(0x7F));
  const __m256i sign = _mm256_slli_epi32(_mm256_and_si256(b, _mm256_set1_epi32(0x80)), 24);
  const __m256i normal = _mm256_add_epi32(_mm256_slli_epi32(mag, 20), _mm256_set1_epi32(120 << 23));
  const __m256 sub = _mm256_mul_ps(_mm256_cvtepi32_ps(_mm256_and_si256(b, _mm256_set1_epi32(7))),
                                   _mm256_set1_ps(1.0f / 512.0f));
  const __m256 is_sub = _mm256_castsi256_ps(_mm256_cmpgt_epi32(_mm256_set1_epi32(8), mag));
  __m256 v = _mm256_blendv_ps(_mm256_castsi256_ps(normal), sub, is_sub);
  v = _mm256_castsi256_ps(_mm256_or_si256(_mm256_castps_si256(v), sign));
  const __m256 is_nan = _mm256_castsi256_ps(_mm256_cmpeq_epi32(mag, _mm256_set1_epi32(0x7F)));
  return _mm256_blendv_ps(v, _mm256_set1_ps(NAN), is_nan);
}

// e2m1 codes (one per lane, 0..15) -> magnitude[c & 7] with the sign of bit 3
FT_AVX2 inline __m256 e2m1_lanes8(__m256i c, __m256 mag) {
  const __m256 m = _mm256_permutevar8x32_ps(mag, c);   // the index's low 3 bits
  const __m256i sign = _mm256_slli_epi32(_mm256_and_si256(c, _mm256_set1_epi32(8)), 28);
  return _mm256_castsi256_ps(_mm256_xor_si256(_mm256_castps_si256(m), sign));
}

struct W8F32 {
  const float* v;
  FT_AVX2 __m256 operator()(int k0) const { return _mm256_loadu_ps(v + k0); }
};

struct W8BF16 {
  const uint16_t* v;
  FT_AVX2 __m256 operator()(int k0) const {
    const __m256i w = _mm256_cvtepu16_epi32(_mm_loadu_si128(reinterpret_cast<const __m128i*>(v + k0)));
    return _mm256_castsi256_ps(_mm256_slli_epi32(w, 16));
  }
};

struct W8FP8 {
  const uint8_t* v;
  const float* sc;
  FT_AVX2 __m256 operator()(int k0) const {
    const __m256i b = _mm256_cvtepu8_epi32(_mm_loadl_epi64(reinterpret_cast<const __m128i*>(v + k0)));
    return _mm256_mul_ps(e4m3_lanes8(b), _mm256_set1_ps(sc[k0 >> 7]));
  }
};

FT_AVX2 inline float hsum8(__m256 s) {
  __m128 t = _mm_add_ps(_mm256_castps256_ps128(s), _mm256_extractf128_ps(s, 1));
  t = _mm_add_ps(t, _mm_movehl_ps(t, t));
  t = _mm_add_ss(t, _mm_movehdup_ps(t));
  return _mm_cvtss_f32(t);
}

FT_AVX2 void host_rows_avx2(const HostRow& r, const float* const* xs, int n, float* out) {
  alignas(32) float mag_v[8];
  for (int c = 0; c < 8; ++c) mag_v[c] = e2m1_value(c);
  const __m256 mag = _mm256_load_ps(mag_v);
  const __m256i low4 = _mm256_set1_epi32(15);
  for (int j0 = 0; j0 < n; j0 += 2) {
    const int nj = n - j0 < 2 ? n - j0 : 2;
    const float* const* x = xs + j0;
    __m256 acc[2][NACC];
    for (int j = 0; j < 2; ++j)
      for (int u = 0; u < NACC; ++u) acc[j][u] = _mm256_setzero_ps();
    switch (r.wt) {
      case FT_W_F32:
        dot_rows8(r.K, x, nj, acc, W8F32{reinterpret_cast<const float*>(r.vals)});
        break;
      case FT_W_BF16:
        dot_rows8(r.K, x, nj, acc, W8BF16{reinterpret_cast<const uint16_t*>(r.vals)});
        break;
      case FT_W_FP8E4M3:
        dot_rows8(r.K, x, nj, acc, W8FP8{r.vals, reinterpret_cast<const float*>(r.scales)});
        break;
      default: {  // NVFP4, MXFP4: 32 elements (16 code bytes) per group, x in pair-split order
        const bool mx = r.wt == FT_W_MXFP4;
        for (int g = 0; g < r.K / 32; ++g) {
          const __m128i q = _mm_loadu_si128(reinterpret_cast<const __m128i*>(r.vals + 16 * g));
          const __m256i ba = _mm256_cvtepu8_epi32(q);                     // bytes 0-7
          const __m256i bb = _mm256_cvtepu8_epi32(_mm_srli_si128(q, 8));  // bytes 8-15
          const __m256 sl = mx ? _mm256_mul_ps(mag, _mm256_set1_ps(r.scale_lut[r.scales[g]] * r.gscale)) : mag;
          __m256 ea = e2m1_lanes8(_mm256_and_si256(ba, low4), sl);   // elements 0, 2, .., 14
          __m256 eb = e2m1_lanes8(_mm256_and_si256(bb, low4), sl);   // elements 16, .., 30
          __m256 oa = e2m1_lanes8(_mm256_srli_epi32(ba, 4), sl);     // elements 1, 3, .., 15
          __m256 ob = e2m1_lanes8(_mm256_srli_epi32(bb, 4), sl);     // elements 17, .., 31
          if (!mx) {
            // two 16-element blocks: bytes 0-7 the first, bytes 8-15 the second
            const __m256 sa = _mm256_set1_ps(r.scale_lut[r.scales[2 * g]] * r.gscale);
            const __m256 sb = _mm256_set1_ps(r.scale_lut[r.scales[2 * g + 1]] * r.gscale);
            ea = _mm256_mul_ps(ea, sa);
            oa = _mm256_mul_ps(oa, sa);
            eb = _mm256_mul_ps(eb, sb);
            ob = _mm256_mul_ps(ob, sb);
          }
          for (int j = 0; j < nj; ++j) {
            const float* xg = x[j] + 32 * g;
            acc[j][0] = _mm256_fmadd_ps(ea, _mm256_loadu_ps(xg), acc[j][0]);
            acc[j][1] = _mm256_fmadd_ps(eb, _mm256_loadu_ps(xg + 8), acc[j][1]);
            acc[j][2] = _mm256_fmadd_ps(oa, _mm256_loadu_ps(xg + 16), acc[j][2]);
            acc[j][3] = _mm256_fmadd_ps(ob, _mm256_loadu_ps(xg + 24), acc[j][3]);
          }
        }
        break;
      }
    }
    for (int j = 0; j < nj; ++j)
      out[j0 + j] = hsum8(_mm256_add_ps(_mm256_add_ps(acc[j][0], acc[j][1]), _mm256_add_ps(acc[j][2], acc[j][3])));
  }
}

}  // namespace
#endif

void host_rows(const HostRow& r, const float* const* xs, int n, float* out) {
#if defined(__x86_64__)
  if (host_simd_form() == HOST_AVX512)
    host_rows_avx512(r, xs, n, out);
  else
    host_rows_avx2(r, xs, n, out);
#else
  (void)r; (void)xs; (void)n; (void)out;
#endif
}

}  // namespace ft
