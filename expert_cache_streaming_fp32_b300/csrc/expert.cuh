// Grouped SwiGLU expert FFN over cache slots, CUDA-core path.
//
// Two persistent launches per call:
//   gate/up:  A[p][n] = silu(sum_h X[p][h] Wg[n][h]) * (sum_h X[p][h] Wu[n][h])
//   down:     Y[p][h] = sum_n A[p][n] Wd[h][n]
// p runs over the permuted assignment rows of every evaluated expert.  The
// weights are the HBM stream: every 16-byte weight load is used for up to
// MR_MAX token rows held in shared memory, so an expert's weights are read
// once per row chunk of MR_MAX rows (once in total at decode sizes).  Work
// items are (expert, output tile, row chunk); every CTA rebuilds the list of
// evaluated experts from offsets/slot_of and walks items with a grid stride,
// so nothing depends on host knowledge of the routing.  Each output is one
// warp's fixed-order reduction: results do not depend on the other experts in
// the call, on the slot or on the tiling of other rows.
#pragma once
#include "common.cuh"

namespace ft {

constexpr int EX_THREADS = 256;
constexpr int EX_WARPS = EX_THREADS / 32;
constexpr int EX_MR = 8;        // token rows per item
constexpr int GU_RPW = 2;       // gate/up: output rows per warp (x2 matrices)
constexpr int GU_NT = EX_WARPS * GU_RPW;
constexpr int DN_RPW = 4;       // down: output rows per warp
constexpr int DN_NT = EX_WARPS * DN_RPW;
constexpr int EX_UNR = 1;       // k-chunks whose loads are issued together (4 rows x 16 B per lane already in flight)
constexpr int EX_UNR_ONE = 4;   // the same for one token row per expert (T = 1), with registers to spare

// ------------------------------------------------------------------ weight formats
// load(): the 16 bytes (and scale) a lane needs for elements k .. k+EPL-1 of a row.
// dot(): sum over those elements of w * x, scales applied per block; the matrix
// scale of NVFP4 is applied once to the finished sum (gscale()).
struct RawF32 { uint4 v; };
struct RawQ { uint4 v; uint32_t s; };

template <int WT> struct WFmt;

template <> struct WFmt<FT_W_F32> {
  static constexpr int EPL = 4;
  using Raw = RawF32;
  __device__ static Raw load(const uint8_t* v, const uint8_t*, int k) {
    return {__ldg(reinterpret_cast<const uint4*>(v + (size_t)k * 4))};
  }
  __device__ static float dot(const Raw& r, const float* x) {
    return __uint_as_float(r.v.x) * x[0] + __uint_as_float(r.v.y) * x[1] + __uint_as_float(r.v.z) * x[2] +
           __uint_as_float(r.v.w) * x[3];
  }
};

template <> struct WFmt<FT_W_BF16> {
  static constexpr int EPL = 8;
  using Raw = RawF32;
  __device__ static Raw load(const uint8_t* v, const uint8_t*, int k) {
    return {__ldg(reinterpret_cast<const uint4*>(v + (size_t)k * 2))};
  }
  __device__ static float dot(const Raw& r, const float* x) {
    return bf16lo(r.v.x) * x[0] + bf16hi(r.v.x) * x[1] + bf16lo(r.v.y) * x[2] + bf16hi(r.v.y) * x[3] +
           bf16lo(r.v.z) * x[4] + bf16hi(r.v.z) * x[5] + bf16lo(r.v.w) * x[6] + bf16hi(r.v.w) * x[7];
  }
};

__device__ __forceinline__ float dot_e4m3x4(uint32_t w, const float* x) {
  float2 a = e4m3x2_to_float2((uint16_t)(w & 0xffffu));
  float2 b = e4m3x2_to_float2((uint16_t)(w >> 16));
  return a.x * x[0] + a.y * x[1] + b.x * x[2] + b.y * x[3];
}

__device__ __forceinline__ float dot_e2m1x8(uint32_t w, const float* x) {
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = e2m1x2_to_float2((uint8_t)(w >> (8 * i)));
    s += f.x * x[2 * i] + f.y * x[2 * i + 1];
  }
  return s;
}

template <> struct WFmt<FT_W_FP8E4M3> {
  static constexpr int EPL = 16;
  using Raw = RawQ;
  __device__ static Raw load(const uint8_t* v, const uint8_t* s, int k) {
    Raw r;
    r.v = __ldg(reinterpret_cast<const uint4*>(v + k));
    r.s = __float_as_uint(__ldg(reinterpret_cast<const float*>(s) + (k >> 7)));
    return r;
  }
  __device__ static float dot(const Raw& r, const float* x) {
    float d = dot_e4m3x4(r.v.x, x) + dot_e4m3x4(r.v.y, x + 4) + dot_e4m3x4(r.v.z, x + 8) + dot_e4m3x4(r.v.w, x + 12);
    return d * __uint_as_float(r.s);
  }
};

template <> struct WFmt<FT_W_NVFP4> {
  static constexpr int EPL = 32;
  using Raw = RawQ;
  __device__ static Raw load(const uint8_t* v, const uint8_t* s, int k) {
    Raw r;
    r.v = __ldg(reinterpret_cast<const uint4*>(v + (k >> 1)));
    r.s = __ldg(reinterpret_cast<const uint16_t*>(s + (k >> 4)));
    return r;
  }
  __device__ static float dot(const Raw& r, const float* x) {
    float d0 = dot_e2m1x8(r.v.x, x) + dot_e2m1x8(r.v.y, x + 8);
    float d1 = dot_e2m1x8(r.v.z, x + 16) + dot_e2m1x8(r.v.w, x + 24);
    return d0 * e4m3_to_float((uint8_t)(r.s & 0xff)) + d1 * e4m3_to_float((uint8_t)(r.s >> 8));
  }
};

template <> struct WFmt<FT_W_MXFP4> {
  static constexpr int EPL = 32;
  using Raw = RawQ;
  __device__ static Raw load(const uint8_t* v, const uint8_t* s, int k) {
    Raw r;
    r.v = __ldg(reinterpret_cast<const uint4*>(v + (k >> 1)));
    r.s = __ldg(s + (k >> 5));
    return r;
  }
  __device__ static float dot(const Raw& r, const float* x) {
    float d = dot_e2m1x8(r.v.x, x) + dot_e2m1x8(r.v.y, x + 8) + dot_e2m1x8(r.v.z, x + 16) + dot_e2m1x8(r.v.w, x + 24);
    return d * e8m0_to_float((uint8_t)r.s);
  }
};

__host__ __device__ constexpr int fmt_bits(int wt) {
  return wt == FT_W_F32 ? 32 : wt == FT_W_BF16 ? 16 : wt == FT_W_FP8E4M3 ? 8 : 4;
}
// bytes of the scale row of a [rows][K] matrix
__host__ __device__ inline uint64_t fmt_scale_row_bytes(int wt, int K) {
  return wt == FT_W_FP8E4M3 ? (uint64_t)(K / 128) * 4 : wt == FT_W_NVFP4 ? (uint64_t)(K / 16)
                                                      : wt == FT_W_MXFP4 ? (uint64_t)(K / 32) : 0;
}

// ------------------------------------------------------------------ staged rows
// Token rows live in shared memory as fp32 in a lane-swizzled order: for chunk
// c of CH = 32*EPL elements, lane l's EPL elements are stored as EPL/4 float4
// at c*CH + j4*128 + l*4, so a warp's float4 reads are consecutive.
template <int EPL>
__device__ __forceinline__ int swz(int k) {
  constexpr int CH = 32 * EPL;
  const int c = k / CH, q = k - c * CH, l = q / EPL, j = q - l * EPL;
  return c * CH + (j >> 2) * 128 + l * 4 + (j & 3);
}

template <int EPL>
__host__ __device__ inline int staged_stride(int K) {
  return ceil_div(K, 32 * EPL) * 32 * EPL;
}

struct ExpertArgs {
  const void* x;
  int x_type, T, k, H, I, E, pool_slots;
  const int32_t* perm;
  const int32_t* offsets;
  const int32_t* slot_of;
  const uint8_t* pool;
  uint64_t S;
  uint64_t off_val[3], off_scale[3], off_gscale;
  float* A;
  float* y;
};

// ------------------------------------------------------------------ plan
// Every CTA lists the evaluated experts (rows > 0, valid slot) in ascending id
// with the prefix sum of their item counts.
struct Plan {
  int n_act;
  int total;
};

__device__ __forceinline__ int block_excl_scan(int v, int* warp_buf, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(FT_FULL_MASK, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_buf[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < EX_WARPS ? warp_buf[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(FT_FULL_MASK, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < EX_WARPS) warp_buf[lane] = wi - w;
    if (lane == EX_WARPS - 1) warp_buf[EX_WARPS] = wi;
  }
  __syncthreads();
  const int r = warp_buf[warp] + incl - v;
  total = warp_buf[EX_WARPS];
  __syncthreads();
  return r;
}

// act_e[E], act_pref[E+1] in shared memory; tiles_per_expert output tiles.
__device__ Plan build_plan(const ExpertArgs& a, int tiles_per_expert, int* act_e, int* act_pref, int* warp_buf) {
  const int per = ceil_div(a.E, EX_THREADS);
  const int e0 = threadIdx.x * per;
  int my_act = 0, my_items = 0;
  for (int i = 0; i < per; ++i) {
    const int e = e0 + i;
    if (e < a.E) {
      const int cnt = a.offsets[e + 1] - a.offsets[e];
      const int s = a.slot_of[e];
      if (cnt > 0 && s >= 0) {
        if (s >= a.pool_slots) { record_error(FT_DERR_SLOT_INDEX); continue; }
        my_act += 1;
        my_items += tiles_per_expert * ceil_div(cnt, EX_MR);
      }
    }
  }
  Plan p;
  int pos = block_excl_scan(my_act, warp_buf, p.n_act);
  int ipos = block_excl_scan(my_items, warp_buf, p.total);
  for (int i = 0; i < per; ++i) {
    const int e = e0 + i;
    if (e < a.E) {
      const int cnt = a.offsets[e + 1] - a.offsets[e];
      const int s = a.slot_of[e];
      if (cnt > 0 && s >= 0 && s < a.pool_slots) {
        act_e[pos] = e;
        act_pref[pos] = ipos;
        pos += 1;
        ipos += tiles_per_expert * ceil_div(cnt, EX_MR);
      }
    }
  }
  if (threadIdx.x == 0) act_pref[p.n_act] = p.total;
  __syncthreads();
  return p;
}

__device__ __forceinline__ int find_act(const int* pref, int n, int item) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (pref[mid] <= item) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ int pow2_rows(int r) { return r <= 1 ? 1 : r <= 2 ? 2 : r <= 4 ? 4 : 8; }

// ------------------------------------------------------------------ gate/up
template <int WT, int MR, int UNR = EX_UNR>
__device__ __forceinline__ void gateup_rows(const ExpertArgs& a, const float* xs, int xstride,
                                            const uint8_t* rec, int n_base, int p0, int rows) {
  using F = WFmt<WT>;
  constexpr int EPL = F::EPL;
  constexpr int CH = 32 * EPL;
  constexpr int V = GU_RPW * 2 * MR;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int K = a.H;
  const uint64_t vrow_bytes = (uint64_t)K * fmt_bits(WT) / 8;
  const uint64_t srow_bytes = fmt_scale_row_bytes(WT, K);
  const uint8_t* vb[GU_RPW][2];
  const uint8_t* sb[GU_RPW][2];
  bool valid[GU_RPW];
#pragma unroll
  for (int i = 0; i < GU_RPW; ++i) {
    const int n = n_base + warp * GU_RPW + i;
    valid[i] = n < a.I;
    const int nn = valid[i] ? n : 0;
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      vb[i][m] = rec + a.off_val[m] + nn * vrow_bytes;
      sb[i][m] = rec + a.off_scale[m] + nn * srow_bytes;
    }
  }
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.0f;
  const int nch = ceil_div(K, CH);
  for (int c0 = 0; c0 < nch; c0 += UNR) {
    typename F::Raw raw[UNR][GU_RPW][2];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int kk = (c0 + u) * CH + lane * EPL;
      const bool in = (c0 + u) < nch && kk < K;
#pragma unroll
      for (int i = 0; i < GU_RPW; ++i)
#pragma unroll
        for (int m = 0; m < 2; ++m)
          if (in && valid[i]) raw[u][i][m] = F::load(vb[i][m], sb[i][m], kk);
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int kk = (c0 + u) * CH + lane * EPL;
      if ((c0 + u) >= nch || kk >= K) break;
#pragma unroll
      for (int r = 0; r < MR; ++r) {
        float xv[EPL];
        const float* xr = xs + r * xstride + (c0 + u) * CH + lane * 4;
#pragma unroll
        for (int j4 = 0; j4 < EPL / 4; ++j4) {
          float4 t = *reinterpret_cast<const float4*>(xr + j4 * 128);
          xv[4 * j4] = t.x; xv[4 * j4 + 1] = t.y; xv[4 * j4 + 2] = t.z; xv[4 * j4 + 3] = t.w;
        }
#pragma unroll
        for (int i = 0; i < GU_RPW; ++i)
#pragma unroll
          for (int m = 0; m < 2; ++m)
            if (valid[i]) acc[(i * 2 + m) * MR + r] += F::dot(raw[u][i][m], xv);
      }
    }
  }
  warp_reduce_scatter<V>(acc, lane);
  constexpr int G = 32 / V;  // lanes sharing one value
  const float up = __shfl_down_sync(FT_FULL_MASK, acc[0], MR * G);
  const int vi = lane / G;
  const int r = vi % MR, m = (vi / MR) % 2, i = vi / (2 * MR);
  if ((lane % G) == 0 && m == 0 && r < rows && valid[i]) {
    float g = acc[0], u = up;
    if (WT == FT_W_NVFP4) {
      const float* gs = reinterpret_cast<const float*>(rec + a.off_gscale);
      g *= gs[0];
      u *= gs[1];
    }
    const int n = n_base + warp * GU_RPW + i;
    a.A[(size_t)(p0 + r) * a.I + n] = silu(g) * u;
  }
}

// ONE: every expert has one token row (T = 1): no row-count dispatch, and the registers
// the wider row blocks would take go to more loads in flight.
template <int WT, typename XT, bool ONE = false>
__global__ void __launch_bounds__(EX_THREADS, 2)
gateup_kernel(ExpertArgs a) {
  pdl_begin();
  constexpr int EPL = WFmt<WT>::EPL;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ int warp_buf[EX_WARPS + 1];
  int* act_e = reinterpret_cast<int*>(smem_raw);
  int* act_pref = act_e + a.E;
  const int xstride = staged_stride<EPL>(a.H);
  float* xs = reinterpret_cast<float*>(smem_raw + ((size_t)(2 * a.E + 1) * 4 + 15) / 16 * 16);
  const int tiles = ceil_div(a.I, GU_NT);
  const Plan p = build_plan(a, tiles, act_e, act_pref, warp_buf);
  const XT* x = reinterpret_cast<const XT*>(a.x);
  for (int item = blockIdx.x; item < p.total; item += gridDim.x) {
    const int ai = find_act(act_pref, p.n_act, item);
    const int e = act_e[ai];
    const int local = item - act_pref[ai];
    const int off = a.offsets[e];
    const int cnt = a.offsets[e + 1] - off;
    const int nrc = ceil_div(cnt, EX_MR);
    const int tile = local / nrc, rc = local - tile * nrc;
    const int p0 = off + rc * EX_MR;
    const int rows = min(EX_MR, cnt - rc * EX_MR);
    const int MRr = pow2_rows(rows);
    // stage token rows (fp32, swizzled); rows beyond `rows` are zero
    for (int i = threadIdx.x; i < MRr * a.H; i += EX_THREADS) {
      const int r = i / a.H, h = i - r * a.H;
      float v = 0.0f;
      if (r < rows) {
        const int pa = a.perm[p0 + r];
        const int t = pa / a.k;
        if ((unsigned)t < (unsigned)a.T) v = (float)x[(size_t)t * a.H + h];
        else record_error(FT_DERR_ROW_INDEX);
      }
      xs[r * xstride + swz<EPL>(h)] = v;
    }
    __syncthreads();
    const uint8_t* rec = a.pool + (uint64_t)a.slot_of[e] * a.S;
    const int n_base = tile * GU_NT;
    if (ONE) {
      // one row at a time (a routing that repeats an expert for one token gives it more)
      for (int r = 0; r < rows; ++r)
        gateup_rows<WT, 1, EX_UNR_ONE>(a, xs + r * xstride, xstride, rec, n_base, p0 + r, 1);
    } else {
      switch (MRr) {
        case 1: gateup_rows<WT, 1>(a, xs, xstride, rec, n_base, p0, rows); break;
        case 2: gateup_rows<WT, 2>(a, xs, xstride, rec, n_base, p0, rows); break;
        case 4: gateup_rows<WT, 4>(a, xs, xstride, rec, n_base, p0, rows); break;
        default: gateup_rows<WT, 8>(a, xs, xstride, rec, n_base, p0, rows); break;
      }
    }
    __syncthreads();
  }
  pdl_end();
}

// ------------------------------------------------------------------ down
template <int WT, int MR, int UNR = EX_UNR>
__device__ __forceinline__ void down_rows(const ExpertArgs& a, const float* as, int astride,
                                          const uint8_t* rec, int h_base, int p0, int rows) {
  using F = WFmt<WT>;
  constexpr int EPL = F::EPL;
  constexpr int CH = 32 * EPL;
  constexpr int V = DN_RPW * MR;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int K = a.I;
  const uint64_t vrow_bytes = (uint64_t)K * fmt_bits(WT) / 8;
  const uint64_t srow_bytes = fmt_scale_row_bytes(WT, K);
  const uint8_t* vb[DN_RPW];
  const uint8_t* sb[DN_RPW];
  bool valid[DN_RPW];
#pragma unroll
  for (int i = 0; i < DN_RPW; ++i) {
    const int h = h_base + warp * DN_RPW + i;
    valid[i] = h < a.H;
    const int hh = valid[i] ? h : 0;
    vb[i] = rec + a.off_val[2] + hh * vrow_bytes;
    sb[i] = rec + a.off_scale[2] + hh * srow_bytes;
  }
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.0f;
  const int nch = ceil_div(K, CH);
  for (int c0 = 0; c0 < nch; c0 += UNR) {
    typename F::Raw raw[UNR][DN_RPW];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int kk = (c0 + u) * CH + lane * EPL;
      const bool in = (c0 + u) < nch && kk < K;
#pragma unroll
      for (int i = 0; i < DN_RPW; ++i)
        if (in && valid[i]) raw[u][i] = F::load(vb[i], sb[i], kk);
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int kk = (c0 + u) * CH + lane * EPL;
      if ((c0 + u) >= nch || kk >= K) break;
#pragma unroll
      for (int r = 0; r < MR; ++r) {
        float xv[EPL];
        const float* xr = as + r * astride + (c0 + u) * CH + lane * 4;
#pragma unroll
        for (int j4 = 0; j4 < EPL / 4; ++j4) {
          float4 t = *reinterpret_cast<const float4*>(xr + j4 * 128);
          xv[4 * j4] = t.x; xv[4 * j4 + 1] = t.y; xv[4 * j4 + 2] = t.z; xv[4 * j4 + 3] = t.w;
        }
#pragma unroll
        for (int i = 0; i < DN_RPW; ++i)
          if (valid[i]) acc[i * MR + r] += F::dot(raw[u][i], xv);
      }
    }
  }
  warp_reduce_scatter<V>(acc, lane);
  constexpr int G = 32 / V;
  const int vi = lane / G;
  const int r = vi % MR, i = vi / MR;
  if ((lane % G) == 0 && r < rows && valid[i]) {
    float v = acc[0];
    if (WT == FT_W_NVFP4) v *= reinterpret_cast<const float*>(rec + a.off_gscale)[2];
    a.y[(size_t)(p0 + r) * a.H + h_base + warp * DN_RPW + i] = v;
  }
}

template <int WT, bool ONE = false>
__global__ void __launch_bounds__(EX_THREADS, 2)
down_kernel(ExpertArgs a) {
  pdl_begin();
  constexpr int EPL = WFmt<WT>::EPL;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ int warp_buf[EX_WARPS + 1];
  int* act_e = reinterpret_cast<int*>(smem_raw);
  int* act_pref = act_e + a.E;
  const int astride = staged_stride<EPL>(a.I);
  float* as = reinterpret_cast<float*>(smem_raw + ((size_t)(2 * a.E + 1) * 4 + 15) / 16 * 16);
  const int tiles = ceil_div(a.H, DN_NT);
  const Plan p = build_plan(a, tiles, act_e, act_pref, warp_buf);
  for (int item = blockIdx.x; item < p.total; item += gridDim.x) {
    const int ai = find_act(act_pref, p.n_act, item);
    const int e = act_e[ai];
    const int local = item - act_pref[ai];
    const int off = a.offsets[e];
    const int cnt = a.offsets[e + 1] - off;
    const int nrc = ceil_div(cnt, EX_MR);
    const int tile = local / nrc, rc = local - tile * nrc;
    const int p0 = off + rc * EX_MR;
    const int rows = min(EX_MR, cnt - rc * EX_MR);
    const int MRr = pow2_rows(rows);
    for (int i = threadIdx.x; i < MRr * a.I; i += EX_THREADS) {
      const int r = i / a.I, n = i - r * a.I;
      as[r * astride + swz<EPL>(n)] = r < rows ? a.A[(size_t)(p0 + r) * a.I + n] : 0.0f;
    }
    __syncthreads();
    const uint8_t* rec = a.pool + (uint64_t)a.slot_of[e] * a.S;
    const int h_base = tile * DN_NT;
    if (ONE) {
      for (int r = 0; r < rows; ++r)
        down_rows<WT, 1, EX_UNR_ONE>(a, as + r * astride, astride, rec, h_base, p0 + r, 1);
    } else {
      switch (MRr) {
        case 1: down_rows<WT, 1>(a, as, astride, rec, h_base, p0, rows); break;
        case 2: down_rows<WT, 2>(a, as, astride, rec, h_base, p0, rows); break;
        case 4: down_rows<WT, 4>(a, as, astride, rec, h_base, p0, rows); break;
        default: down_rows<WT, 8>(a, as, astride, rec, h_base, p0, rows); break;
      }
    }
    __syncthreads();
  }
  pdl_end();
}

// ------------------------------------------------------------------ layout
static int expert_layout(int wt, int H, int I, ft_expert_layout* L) {
  if (wt < FT_W_F32 || wt > FT_W_MXFP4) return FT_EINVAL;
  // K a multiple of 128 keeps every value row 16-byte aligned, covers whole
  // scale blocks (128 for fp8, 16/32 for fp4) and keeps scale rows aligned for
  // their element size, in all formats
  if (H <= 0 || I <= 0 || H % 128 || I % 128) return FT_EINVAL;
  auto al = [](uint64_t v) { return (v + 255) / 256 * 256; };
  const uint64_t HI = (uint64_t)H * I;
  const uint64_t vb = HI * fmt_bits(wt) / 8;
  uint64_t o = 0;
  L->payload_bytes = 0;
  for (int m = 0; m < 3; ++m) {
    L->off_val[m] = o;
    o = al(o + vb);
    L->payload_bytes += vb;
  }
  for (int m = 0; m < 3; ++m) {
    const int rows = m == 2 ? H : I, K = m == 2 ? I : H;
    const uint64_t sb = (uint64_t)rows * fmt_scale_row_bytes(wt, K);
    L->off_scale[m] = sb ? o : 0;
    o = al(o + sb);
    L->payload_bytes += sb;
  }
  if (wt == FT_W_NVFP4) {
    L->off_gscale = o;
    o = al(o + 12);
    L->payload_bytes += 12;
  } else {
    L->off_gscale = 0;
  }
  L->bytes = o;
  return FT_OK;
}

}  // namespace ft
