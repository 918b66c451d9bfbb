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
// The logits are read through L2: other CTAs of the same launch may have written them.
template <int PER_LANE>
__device__ __forceinline__ void route_token(const float* z, int E, int k, int32_t* __restrict__ idx_row,
                                            float* __restrict__ w_row) {
  const int lane = threadIdx.x & 31;
  float v[PER_LANE];
  unsigned taken = 0;
#pragma unroll
  for (int i = 0; i < PER_LANE; ++i) {
    int e = lane + 32 * i;
    v[i] = e < E ? __ldcg(z + e) : -INFINITY;
    if (e >= E) taken |= 1u << i;
  }
  float my_v = 0.0f;  // lane j keeps the j-th choice
  int my_i = 0;
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
      bv = __ldcg(z + bi);
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == j) {
      my_v = bv;
      my_i = bi;
    }
  }
  // softmax over the chosen logits; the sum runs in choice order
  const float m = __shfl_sync(FT_FULL_MASK, my_v, 0);
  const float ex = lane < k ? expf(my_v - m) : 0.0f;
  float s = 0.0f;
#pragma unroll 1
  for (int j = 0; j < k; ++j) s += __shfl_sync(FT_FULL_MASK, ex, j);
  const float inv = 1.0f / s;
  if (lane < k) {
    idx_row[lane] = my_i;
    w_row[lane] = ex * inv;
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
// Stable grouping of the n = T*k assignments by expert, by one CTA of W warps.
// Pass 1: per-expert counts with shared-memory atomics, exclusive scan into
// offsets.  Pass 2: assignments in tiles of 32*W; inside a warp,
// __match_any_sync groups equal experts and the rank is the number of equal
// lanes below; across warps a per-(warp, expert) count table is scanned in warp
// order, continuing from the previous tiles.  Positions therefore follow the
// assignment order a = t*k + j within each expert (stable), which makes the
// result unique.  idx is read through L2 (it may have been written by other
// CTAs of the same launch).  tab holds (2 + W) * E ints of shared memory.
constexpr int PM_THREADS = 1024;
constexpr int PM_WARPS = PM_THREADS / 32;
constexpr int PM_MAXE = 512;

template <int W>
__device__ __forceinline__ void permute_block(const int32_t* idx, int n, int E, int32_t* __restrict__ counts,
                                              int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                                              int32_t* __restrict__ inv, int32_t* tab, int32_t* warp_tot) {
  static_assert(W >= 1 && W <= 32, "one warp scans the warp totals");
  constexpr int NT = W * 32;
  int32_t* cnt = tab;                     // [E]
  int32_t* base = cnt + E;                // [E] running position per expert (absolute)
  int32_t* wc = base + E;                 // [W][E]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < E; e += NT) cnt[e] = 0;
  for (int i = tid; i < W * E; i += NT) wc[i] = 0;
  __syncthreads();
  for (int a = tid; a < n; a += NT) {
    const int e = __ldcg(idx + a);
    if ((unsigned)e < (unsigned)E) atomicAdd(&cnt[e], 1);
    else record_error(FT_DERR_EXPERT_INDEX);
  }
  __syncthreads();
  // exclusive scan of cnt: each thread sums a run of consecutive experts, then warp scans
  {
    const int per = ceil_div(E, NT);
    int local = 0;
    for (int i = 0; i < per; ++i) {
      const int e = tid * per + i;
      if (e < E) local += cnt[e];
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(FT_FULL_MASK, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int w = lane < W ? warp_tot[lane] : 0;
      int wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(FT_FULL_MASK, wi, o);
        if (lane >= o) wi += y;
      }
      if (lane < W) warp_tot[lane] = wi - w;
    }
    __syncthreads();
    int run = warp_tot[warp] + incl - local;
    for (int i = 0; i < per; ++i) {
      const int e = tid * per + i;
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
  for (int t0 = 0; t0 < n; t0 += NT) {
    const int a = t0 + tid;
    int e = a < n ? __ldcg(idx + a) : -1;
    if ((unsigned)e >= (unsigned)E) e = -1;
    const unsigned peers = __match_any_sync(FT_FULL_MASK, e);
    const int rank = __popc(peers & ((1u << lane) - 1));
    const int leader = __ffs(peers) - 1;
    if (e >= 0 && lane == leader) wc[warp * E + e] = __popc(peers);
    __syncthreads();
    for (int ex = tid; ex < E; ex += NT) {
      int run = base[ex];
#pragma unroll 4
      for (int w = 0; w < W; ++w) {
        const int c = wc[w * E + ex];
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
    for (int i = tid; i < W * E; i += NT) wc[i] = 0;
    __syncthreads();
  }
}

__global__ void __launch_bounds__(PM_THREADS)
permute_kernel(const int32_t* __restrict__ idx, int n, int E, int32_t* __restrict__ counts,
               int32_t* __restrict__ offsets, int32_t* __restrict__ perm, int32_t* __restrict__ inv) {
  extern __shared__ int32_t pm_smem[];       // [(2 + PM_WARPS) * E]
  __shared__ int32_t warp_tot[PM_WARPS];
  pdl_begin();
  permute_block<PM_WARPS>(idx, n, E, counts, offsets, perm, inv, pm_smem, warp_tot);
  pdl_end();
}

// ====================================================================== fused routing (decode batches)
// Router logits, top-k and the permutation of a small batch (T <= RW_MAXT) in
// one launch over the grid of router_logits_kernel (expert groups x row
// chunks), so the router matrix is read by many SMs at once:
//   1. each CTA computes the logits of its RT rows for its experts (the same
//      per-expert arithmetic as router_logits_kernel: bit-identical logits);
//   2. the CTA that completes a row chunk (the last of its expert groups to
//      arrive on the chunk's counter) routes the chunk's rows, one warp each;
//   3. the CTA that routes the last chunk (the last arrival on the batch
//      counter) groups all T*k assignments (permute_block).
// Arrival counters live in a caller-owned, zero-initialised device array; the
// last arrival on a counter puts it back to zero, so every call finds them
// zeroed.  Nothing waits: a CTA that is not last simply exits.
constexpr int RW_MAXT = 64;
constexpr int RW_WARPS = RL_WARPS;
constexpr int RW_THREADS = RW_WARPS * 32;

// Counts this CTA's arrival on *ctr once all its threads' earlier global writes
// are done, and tells whether it arrived last of n.  The last arrival puts the
// counter back to zero and afterwards sees every other arrival's writes (read
// them through L2).  An arrival number past n means the counter was not zero
// at launch: recorded, never last.
__device__ __forceinline__ bool last_arrival(uint32_t* ctr, uint32_t n, int* s_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t before = atomicAdd(ctr, 1u);
    const bool last = before == n - 1;
    if (before >= n) record_error(FT_DERR_TABLE);
    if (last) {
      atomicExch(ctr, 0u);
      __threadfence();
    }
    *s_flag = last;
  }
  __syncthreads();
  return *s_flag != 0;
}

template <typename XT, int RT, int PER_LANE>
__global__ void __launch_bounds__(RW_THREADS)
route_grid_kernel(const XT* __restrict__ x, const XT* __restrict__ wr, const float* __restrict__ bias, int T,
                  int H, int E, int k, float* z, int32_t* idx_out, float* w_out, int32_t* __restrict__ counts,
                  int32_t* __restrict__ offsets, int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                  uint32_t* __restrict__ arrivals) {
  extern __shared__ float xs[];  // [RT][H] staged rows; the grouping tables of the last CTA afterwards
  __shared__ int s_flag;
  __shared__ int32_t s_wtot[RW_WARPS];
  pdl_begin();
  const int warp = threadIdx.x >> 5;
  const int chunk = blockIdx.y;
  const int t0 = chunk * RT;
  const int nrows = min(RT, T - t0);
  stage_rows<XT, RT>(x, t0, nrows, H, xs);
  __syncthreads();
  logits_of_rows<XT, RT>(xs, wr, bias, t0, nrows, H, E, blockIdx.x * RW_WARPS + warp, gridDim.x * RW_WARPS, z);
  if (!last_arrival(arrivals + 1 + chunk, gridDim.x, &s_flag)) {
    pdl_end();
    return;
  }
  for (int r = warp; r < nrows; r += RW_WARPS) {
    const int t = t0 + r;
    route_token<PER_LANE>(z + (size_t)t * E, E, k, idx_out + (size_t)t * k, w_out + (size_t)t * k);
  }
  if (!last_arrival(arrivals, gridDim.y, &s_flag)) {
    pdl_end();
    return;
  }
  permute_block<RW_WARPS>(idx_out, T * k, E, counts, offsets, perm, inv, reinterpret_cast<int32_t*>(xs), s_wtot);
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
