// Router logits, top-k gating, permutation by expert, and the weighted combine.
#pragma once
#include "common.cuh"

namespace ft {

// ====================================================================== router logits
// z[t][e] = sum_h x[t][h] W_r[e][h] + b[e].  The grid is (expert groups,
// row chunks of RL_RT): a CTA stages its RL_RT token rows of x in shared
// memory (fp32) and its warps sweep the experts of its group: a warp reads one
// router row with 16-byte loads and dots it with every staged row; lane
// partials are reduced with one reduce-scatter.  Few row chunks (decode) get
// many expert groups, so the router matrix is read in parallel even for one
// token; many row chunks (prefill) get few groups, so x is staged few times.
constexpr int RL_RT = 8;        // token rows per CTA (at most)
constexpr int RL_WARPS = 8;

template <typename XT>
__device__ __forceinline__ void load8(const XT* p, float (&o)[8]);

template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&o)[8]) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  o[0] = bf16lo(u.x); o[1] = bf16hi(u.x); o[2] = bf16lo(u.y); o[3] = bf16hi(u.y);
  o[4] = bf16lo(u.z); o[5] = bf16hi(u.z); o[6] = bf16lo(u.w); o[7] = bf16hi(u.w);
}

template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&o)[8]) {
  float4 a = *reinterpret_cast<const float4*>(p);
  float4 b = *reinterpret_cast<const float4*>(p + 4);
  o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w; o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}

// Stages token rows t0 .. t0+RT-1 of x (zeros past nrows) in shared memory as fp32.
template <typename XT, int RT>
__device__ __forceinline__ void stage_rows(const XT* __restrict__ x, int t0, int nrows, int H, float* xs) {
  // 8 elements (one 16-byte bf16 load or two fp32 loads) per thread step
  for (int r = 0; r < RT; ++r) {
    for (int h = threadIdx.x * 8; h < H; h += blockDim.x * 8) {
      float v[8];
      if (r < nrows) {
        load8<XT>(x + (size_t)(t0 + r) * H + h, v);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.0f;
      }
      *reinterpret_cast<float4*>(xs + r * H + h) = make_float4(v[0], v[1], v[2], v[3]);
      *reinterpret_cast<float4*>(xs + r * H + h + 4) = make_float4(v[4], v[5], v[6], v[7]);
    }
  }
}

// Logits of the staged rows for experts e0, e0 + e_step, ... (one warp per expert).
template <typename XT, int RT>
__device__ __forceinline__ void logits_of_rows(const float* xs, const XT* __restrict__ wr,
                                               const float* __restrict__ bias, int t0, int nrows, int H, int E,
                                               int e0, int e_step, float* __restrict__ z) {
  const int lane = threadIdx.x & 31;
  constexpr int U = 8;  // 256-element chunks whose weight loads are in flight together
  for (int e = e0; e < E; e += e_step) {
    float acc[RT];
#pragma unroll
    for (int r = 0; r < RT; ++r) acc[r] = 0.0f;
    const XT* w = wr + (size_t)e * H;
    for (int k0 = 0; k0 < H; k0 += 256 * U) {
      float wv[U][8];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int k = k0 + u * 256 + lane * 8;
        if (k < H) {
          load8<XT>(w + k, wv[u]);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) wv[u][i] = 0.0f;
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int k = k0 + u * 256 + lane * 8;
        if (k < H) {
#pragma unroll
          for (int r = 0; r < RT; ++r) {
            const float* xr = xs + r * H + k;
            float4 a = *reinterpret_cast<const float4*>(xr);
            float4 b = *reinterpret_cast<const float4*>(xr + 4);
            acc[r] += wv[u][0] * a.x + wv[u][1] * a.y + wv[u][2] * a.z + wv[u][3] * a.w +
                      wv[u][4] * b.x + wv[u][5] * b.y + wv[u][6] * b.z + wv[u][7] * b.w;
          }
        }
      }
    }
    warp_reduce_scatter<RT>(acc, lane);
    const int r = lane / (32 / RT);
    if ((lane % (32 / RT)) == 0 && r < nrows)
      z[(size_t)(t0 + r) * E + e] = acc[0] + (bias ? bias[e] : 0.0f);
  }
}

template <typename XT, int RT>
__global__ void __launch_bounds__(RL_WARPS * 32)
router_logits_kernel(const XT* __restrict__ x, const XT* __restrict__ wr, const float* __restrict__ bias,
                     int T, int H, int E, float* __restrict__ z) {
  extern __shared__ float xs[];  // [RT][H]
  pdl_begin();
  const int t0 = blockIdx.y * RT;
  const int nrows = min(RT, T - t0);
  stage_rows<XT, RT>(x, t0, nrows, H, xs);
  __syncthreads();
  logits_of_rows<XT, RT>(xs, wr, bias, t0, nrows, H, E, blockIdx.x * RL_WARPS + (threadIdx.x >> 5),
                         gridDim.x * RL_WARPS, z);
  pdl_end();
}

// ====================================================================== top-k gating
// One warp per token.  Lane l holds logits e = l, l+32, ...  Each of the k
// rounds takes the warp-wide maximum of (value, -index) among the experts not
// yet chosen.  Weights are a softmax over the chosen logits.
constexpr int RT_MAXK = 16;
constexpr int RT_MAXE = 1024;

__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Top-k of one token's logits z[0..E-1] by one warp; lane 0 writes idx_row and w_row.
template <int PER_LANE>
__device__ __forceinline__ void route_token(const float* __restrict__ z, int E, int k, int32_t* __restrict__ idx_row,
                                            float* __restrict__ w_row) {
  const int lane = threadIdx.x & 31;
  float v[PER_LANE];
  unsigned taken = 0;
#pragma unroll
  for (int i = 0; i < PER_LANE; ++i) {
    int e = lane + 32 * i;
    v[i] = e < E ? z[e] : -INFINITY;
    if (e >= E) taken |= 1u << i;
  }
  float sel_v[RT_MAXK];
  int sel_i[RT_MAXK];
#pragma unroll 1
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
      int e = lane + 32 * i;
      if (!(taken >> i & 1u) && better(v[i], e, bv, bi)) { bv = v[i]; bi = e; }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      float ov = __shfl_xor_sync(FT_FULL_MASK, bv, o);
      int oi = __shfl_xor_sync(FT_FULL_MASK, bi, o);
      if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    // NaN logits or all -inf: fall back to the lowest untaken index so the id stays in range
    if (bi >= E) {
      int cand = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < PER_LANE; ++i) {
        int e = lane + 32 * i;
        if (!(taken >> i & 1u) && e < cand) cand = e;
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) cand = min(cand, __shfl_xor_sync(FT_FULL_MASK, cand, o));
      bi = cand;
      bv = z[bi];
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    sel_v[j] = bv;
    sel_i[j] = bi;
  }
  if (lane == 0) {
    const float m = sel_v[0];
    float s = 0.0f;
    float ex[RT_MAXK];
#pragma unroll 1
    for (int j = 0; j < k; ++j) { ex[j] = expf(sel_v[j] - m); s += ex[j]; }
    const float inv = 1.0f / s;
#pragma unroll 1
    for (int j = 0; j < k; ++j) {
      idx_row[j] = sel_i[j];
      w_row[j] = ex[j] * inv;
    }
  }
}

template <int PER_LANE>
__global__ void __launch_bounds__(256)
route_kernel(const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ idx_out,
             float* __restrict__ w_out) {
  pdl_begin();
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  route_token<PER_LANE>(logits + (size_t)t * E, E, k, idx_out + (size_t)t * k, w_out + (size_t)t * k);
  pdl_end();
}

// ====================================================================== permutation
// One CTA.  Pass 1: per-expert counts with shared-memory atomics, exclusive
// scan into offsets.  Pass 2: assignments in tiles of blockDim; inside a warp,
// __match_any_sync groups equal experts and the rank is the number of equal
// lanes below; across warps a per-(warp, expert) count table is scanned in warp
// order, continuing from the previous tiles.  Positions therefore follow the
// assignment order a = t*k + j within each expert (stable).
constexpr int PM_THREADS = 1024;
constexpr int PM_WARPS = PM_THREADS / 32;
constexpr int PM_MAXE = 512;

__global__ void __launch_bounds__(PM_THREADS)
permute_kernel(const int32_t* __restrict__ idx, int n, int E, int32_t* __restrict__ counts,
               int32_t* __restrict__ offsets, int32_t* __restrict__ perm, int32_t* __restrict__ inv) {
  extern __shared__ int32_t pm_smem[];
  pdl_begin();
  int32_t* cnt = pm_smem;                    // [E]
  int32_t* base = cnt + E;                // [E] running position per expert (absolute)
  int32_t* wc = base + E;                 // [PM_WARPS][E]
  __shared__ int32_t warp_tot[PM_WARPS];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < E; e += PM_THREADS) cnt[e] = 0;
  for (int i = tid; i < PM_WARPS * E; i += PM_THREADS) wc[i] = 0;
  __syncthreads();
  for (int a = tid; a < n; a += PM_THREADS) {
    int e = idx[a];
    if ((unsigned)e < (unsigned)E) atomicAdd(&cnt[e], 1);
    else record_error(FT_DERR_EXPERT_INDEX);
  }
  __syncthreads();
  // exclusive scan of cnt (E <= 512): each thread sums a strided chunk, then warp scans
  {
    const int per = ceil_div(E, PM_THREADS);
    int local = 0;
    for (int i = 0; i < per; ++i) {
      int e = tid * per + i;
      if (e < E) local += cnt[e];
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(FT_FULL_MASK, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int w = warp_tot[lane];
      int wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(FT_FULL_MASK, wi, o);
        if (lane >= o) wi += y;
      }
      warp_tot[lane] = wi - w;
    }
    __syncthreads();
    int run = warp_tot[warp] + incl - local;
    for (int i = 0; i < per; ++i) {
      int e = tid * per + i;
      if (e < E) {
        base[e] = run;
        offsets[e] = run;
        counts[e] = cnt[e];
        run += cnt[e];
      }
    }
    if (tid == 0) offsets[E] = n;
  }
  __syncthreads();
  for (int t0 = 0; t0 < n; t0 += PM_THREADS) {
    const int a = t0 + tid;
    int e = a < n ? idx[a] : -1;
    if ((unsigned)e >= (unsigned)E) e = -1;
    const unsigned peers = __match_any_sync(FT_FULL_MASK, e);
    const int rank = __popc(peers & ((1u << lane) - 1));
    const int leader = __ffs(peers) - 1;
    if (e >= 0 && lane == leader) wc[warp * E + e] = __popc(peers);
    __syncthreads();
    for (int ex = tid; ex < E; ex += PM_THREADS) {
      int run = base[ex];
#pragma unroll 4
      for (int w = 0; w < PM_WARPS; ++w) {
        int c = wc[w * E + ex];
        wc[w * E + ex] = run;
        run += c;
      }
      base[ex] = run;
    }
    __syncthreads();
    if (e >= 0) {
      const int pos = wc[warp * E + e] + rank;
      perm[pos] = a;
      inv[a] = pos;
    }
    __syncthreads();
    // the scan above wrote every (w, ex) entry: reset the whole table for the next tile
    for (int i = tid; i < PM_WARPS * E; i += PM_THREADS) wc[i] = 0;
    __syncthreads();
  }
  pdl_end();
}

// ====================================================================== fused routing (decode batches)
// Router logits, top-k and the permutation of a small batch (T <= RF_MAXT) in
// one launch: a cluster of RF_CL CTAs.  Each CTA computes the logits of its
// share of the experts for every token (the same per-expert arithmetic as
// router_logits_kernel, so the logits are bit-identical) and writes them out;
// after a cluster barrier (release/acquire at cluster scope, so the other
// CTAs' logits are visible) CTA 0 routes every token (one warp per token, as
// route_kernel) and builds counts, offsets, perm and inv for the T*k
// assignments: the rank of an assignment within its expert is the number of
// earlier assignments to the same expert, so perm is stable.
constexpr int RF_CL = 8;
constexpr int RF_MAXT = 16;
constexpr int RF_WARPS = 16;
constexpr int RF_THREADS = RF_WARPS * 32;

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <typename XT, int RT, int PER_LANE>
__global__ void __launch_bounds__(RF_THREADS)
route_fused_kernel(const XT* __restrict__ x, const XT* __restrict__ wr, const float* __restrict__ bias, int T,
                   int H, int E, int k, float* __restrict__ z, int32_t* __restrict__ idx_out,
                   float* __restrict__ w_out, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                   int32_t* __restrict__ perm, int32_t* __restrict__ inv) {
  extern __shared__ float xs[];                      // [RT][H]
  __shared__ int32_t s_cnt[RT_MAXE + 1];
  __shared__ int32_t s_idx[RF_MAXT * RT_MAXK];
  __shared__ int32_t s_wsum[RF_WARPS];
  pdl_begin();
  const int rank = (int)cluster_ctarank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int t0 = 0; t0 < T; t0 += RT) {
    const int nrows = min(RT, T - t0);
    stage_rows<XT, RT>(x, t0, nrows, H, xs);
    __syncthreads();
    logits_of_rows<XT, RT>(xs, wr, bias, t0, nrows, H, E, rank * RF_WARPS + warp, RF_CL * RF_WARPS, z);
    __syncthreads();
  }
  __threadfence();
  cluster_sync_all();
  if (rank != 0) return;
  // top-k per token
  for (int t = warp; t < T; t += RF_WARPS)
    route_token<PER_LANE>(z + (size_t)t * E, E, k, idx_out + (size_t)t * k, w_out + (size_t)t * k);
  for (int e = threadIdx.x; e <= E; e += RF_THREADS) s_cnt[e] = 0;
  __syncthreads();
  // permutation of the n = T*k assignments
  const int n = T * k;
  for (int a = threadIdx.x; a < n; a += RF_THREADS) {
    int e = idx_out[a];
    if ((unsigned)e >= (unsigned)E) {
      record_error(FT_DERR_EXPERT_INDEX);
      e = -1;
    } else {
      atomicAdd(&s_cnt[e], 1);
    }
    s_idx[a] = e;
  }
  __syncthreads();
  // exclusive scan of the counts: each thread a run of consecutive experts
  const int per = ceil_div(E, RF_THREADS);
  int local = 0;
  for (int i = 0; i < per; ++i) {
    const int e = threadIdx.x * per + i;
    if (e < E) local += s_cnt[e];
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(FT_FULL_MASK, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_wsum[warp] = incl;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += s_wsum[w];
  int run = before + incl - local;
  __syncthreads();                                   // every count is read before it is replaced by its offset
  for (int i = 0; i < per; ++i) {
    const int e = threadIdx.x * per + i;
    if (e < E) {
      const int c = s_cnt[e];
      counts[e] = c;
      offsets[e] = run;
      s_cnt[e] = run;
      run += c;
    }
  }
  if (threadIdx.x == 0) offsets[E] = n;
  __syncthreads();
  for (int a = threadIdx.x; a < n; a += RF_THREADS) {
    const int e = s_idx[a];
    if (e < 0) continue;
    int r = 0;
    for (int b = 0; b < a; ++b) r += s_idx[b] == e;
    const int pos = s_cnt[e] + r;
    perm[pos] = a;
    inv[a] = pos;
  }
  pdl_end();
}

// ====================================================================== combine
// out[t][h] = sum_j w[t][j] y[inv[t*k+j]][h] (+ P[t][h]); assignments of
// experts flagged external are skipped.  CB threads per CTA cover CB float4
// columns of one token; every assignment's index loads are issued before the
// row loads, so a token costs two dependent memory round trips.  The sum order
// is fixed (j ascending, then P).
constexpr int CB_THREADS = 64;

__global__ void __launch_bounds__(CB_THREADS)
combine_kernel(const float* __restrict__ y, const int32_t* __restrict__ inv, const int32_t* __restrict__ idx,
               const float* __restrict__ w, const int32_t* __restrict__ ext, const float* __restrict__ P,
               int T, int k, int H, int E, float* __restrict__ out) {
  pdl_begin();
  const int t = blockIdx.y;
  const int h4 = blockIdx.x * blockDim.x + threadIdx.x;
  if (h4 * 4 >= H) return;
  const int nrows = T * k;
  int row[RT_MAXK];
  float wj[RT_MAXK];
#pragma unroll
  for (int j = 0; j < RT_MAXK; ++j) {
    row[j] = -1;
    wj[j] = 0.0f;
    if (j < k) {
      const int a = t * k + j;
      const int e = idx[a];
      const int rr = inv[a];
      if ((unsigned)e >= (unsigned)E) {
        record_error(FT_DERR_EXPERT_INDEX);
      } else if (!(ext && ext[e])) {
        if ((unsigned)rr >= (unsigned)nrows) record_error(FT_DERR_ROW_INDEX);
        else { row[j] = rr; wj[j] = w[a]; }
      }
    }
  }
  float4 v[RT_MAXK];
#pragma unroll
  for (int j = 0; j < RT_MAXK; ++j)
    if (row[j] >= 0) v[j] = reinterpret_cast<const float4*>(y + (size_t)row[j] * H)[h4];
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 0; j < RT_MAXK; ++j) {
    if (row[j] >= 0) {
      acc.x += wj[j] * v[j].x; acc.y += wj[j] * v[j].y; acc.z += wj[j] * v[j].z; acc.w += wj[j] * v[j].w;
    }
  }
  if (P) {
    float4 p = reinterpret_cast<const float4*>(P + (size_t)t * H)[h4];
    acc.x += p.x; acc.y += p.y; acc.z += p.z; acc.w += p.w;
  }
  reinterpret_cast<float4*>(out + (size_t)t * H)[h4] = acc;
  pdl_end();
}

}  // namespace ft
