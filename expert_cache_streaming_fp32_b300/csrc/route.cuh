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

// Stages token rows t0 .. t0+RT-1 of x (zeros past nrows) in shared memory,
// in x's own type (bf16 rows stay bf16: half the shared-memory reads of fp32).
// Each thread loads its 16-byte piece of every row before storing any.
template <typename XT, int RT>
__device__ __forceinline__ void stage_rows(const XT* __restrict__ x, int t0, int nrows, int H, XT* xs) {
  constexpr int V = 16 / (int)sizeof(XT);
  for (int h = threadIdx.x * V; h < H; h += blockDim.x * V) {
    uint4 v[RT];
#pragma unroll
    for (int r = 0; r < RT; ++r)
      v[r] = r < nrows ? *reinterpret_cast<const uint4*>(x + (size_t)(t0 + r) * H + h) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int r = 0; r < RT; ++r) *reinterpret_cast<uint4*>(xs + r * H + h) = v[r];
  }
}

// Eight consecutive staged elements as fp32 (exact for both types).
template <typename XT>
__device__ __forceinline__ void staged8(const XT* p, float (&o)[8]) {
  load8<XT>(p, o);
}

// Logits of the staged rows for experts e0, e0 + e_step, ... (one warp per expert).
template <typename XT, int RT>
__device__ __forceinline__ void logits_of_rows(const XT* xs, const XT* __restrict__ wr,
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
            float a[8];
            staged8<XT>(xs + r * H + k, a);
            acc[r] += wv[u][0] * a[0] + wv[u][1] * a[1] + wv[u][2] * a[2] + wv[u][3] * a[3] +
                      wv[u][4] * a[4] + wv[u][5] * a[5] + wv[u][6] * a[6] + wv[u][7] * a[7];
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
  extern __shared__ __align__(16) unsigned char rl_smem[];
  XT* xs = reinterpret_cast<XT*>(rl_smem);  // [RT][H]
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
// rounds takes, among the experts not yet chosen, the largest logit, ties to
// the smaller expert id.  Logits are compared as order-preserving 32-bit keys
// (-0 taken as +0, so equal logits have equal keys); a round is two warp
// reductions: the largest key, then the smallest id holding it.  NaN logits
// are never preferred; a round that finds only NaN left takes the smallest
// id not yet chosen, so every id stays in range.  Weights are a softmax over
// the chosen logits, summed in choice order.
constexpr int RT_MAXK = 16;
constexpr int RT_MAXE = 1024;

// 0 for NaN, else a key whose unsigned order is the order of the values (> 0).
__device__ __forceinline__ uint32_t logit_key(float v) {
  if (v != v) return 0u;
  const uint32_t b = __float_as_uint(v == 0.0f ? 0.0f : v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Top-k of one token's logits z[0..E-1] by one warp; lanes 0..k-1 write idx_row and w_row
// (and the ids to idx_shared too, when given).  The logits are read through L2: other
// CTAs of the same launch may have written them.
template <int PER_LANE>
__device__ __forceinline__ void route_token(const float* z, int E, int k, int32_t* __restrict__ idx_row,
                                            float* __restrict__ w_row, int32_t* idx_shared = nullptr) {
  const int lane = threadIdx.x & 31;
  float v[PER_LANE];
  uint32_t key[PER_LANE];
  unsigned taken = 0;
#pragma unroll
  for (int i = 0; i < PER_LANE; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? __ldcg(z + e) : -INFINITY;
    key[i] = e < E ? logit_key(v[i]) : 0u;
    if (e >= E) taken |= 1u << i;
  }
  float my_v = 0.0f;  // lane j keeps the j-th choice
  int my_i = 0;
#pragma unroll 1
  for (int j = 0; j < k; ++j) {
    // this lane's candidate: its largest untaken key, the smaller id on ties
    uint32_t bk = 0;
    int bi = 0x7fffffff;
    float bv = 0.0f;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
      if (!(taken >> i & 1u) && key[i] > bk) {
        bk = key[i];
        bi = lane + 32 * i;
        bv = v[i];
      }
    }
    const uint32_t m = __reduce_max_sync(FT_FULL_MASK, bk);
    int win;
    float wv;
    if (m != 0u) {
      win = (int)__reduce_min_sync(FT_FULL_MASK, bk == m ? (uint32_t)bi : 0x7fffffffu);
      wv = __shfl_sync(FT_FULL_MASK, bv, win & 31);
    } else {
      // only NaN left: the smallest id not yet chosen
      uint32_t cand = 0x7fffffffu;
#pragma unroll
      for (int i = 0; i < PER_LANE; ++i)
        if (!(taken >> i & 1u)) cand = min(cand, (uint32_t)(lane + 32 * i));
      win = (int)__reduce_min_sync(FT_FULL_MASK, cand);
      wv = __ldcg(z + win);
    }
    if ((win & 31) == lane) taken |= 1u << (win >> 5);
    if (lane == j) {
      my_v = wv;
      my_i = win;
    }
  }
  // softmax over the chosen logits; the sum runs in choice order
  const float mx = __shfl_sync(FT_FULL_MASK, my_v, 0);
  const float ex = lane < k ? expf(my_v - mx) : 0.0f;
  float part[RT_MAXK];
#pragma unroll
  for (int j = 0; j < RT_MAXK; ++j) part[j] = __shfl_sync(FT_FULL_MASK, ex, j);
  float sum = 0.0f;
#pragma unroll
  for (int j = 0; j < RT_MAXK; ++j)
    if (j < k) sum += part[j];
  const float inv = 1.0f / sum;
  if (lane < k) {
    idx_row[lane] = my_i;
    w_row[lane] = ex * inv;
    if (idx_shared) idx_shared[lane] = my_i;
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
// result unique.  idx is in shared memory (IDX_SHARED) or global memory, read
// through L2 (other CTAs of the same launch may have written it).  tab holds
// (2 + W) * E ints of shared memory.
constexpr int PM_THREADS = 1024;
constexpr int PM_WARPS = PM_THREADS / 32;
constexpr int PM_MAXE = 512;

template <int W, bool IDX_SHARED = false>
__device__ __forceinline__ int load_id(const int32_t* idx, int a) {
  return IDX_SHARED ? idx[a] : __ldcg(idx + a);
}

template <int W, bool IDX_SHARED = false>
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
    const int e = load_id<W, IDX_SHARED>(idx, a);
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
    int e = a < n ? load_id<W, IDX_SHARED>(idx, a) : -1;
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

// The same grouping for n <= 32 assignments by one warp: lane a holds the
// expert of assignment a (anything for a >= n).  Equal experts are grouped with
// __match_any_sync (the rank is the number of equal lanes below); the counts
// go through cnt (E ints of shared memory), which the warp scans in place.
__device__ __forceinline__ void permute_warp(int e_a, int n, int E, int32_t* __restrict__ counts,
                                             int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                                             int32_t* __restrict__ inv, int32_t* cnt) {
  const int lane = threadIdx.x & 31;
  for (int e = lane; e < E; e += 32) cnt[e] = 0;
  bool valid = lane < n;
  if (valid && (unsigned)e_a >= (unsigned)E) {
    record_error(FT_DERR_EXPERT_INDEX);
    valid = false;
  }
  const unsigned peers = __match_any_sync(FT_FULL_MASK, valid ? e_a : -1);
  const int rank = __popc(peers & ((1u << lane) - 1));
  __syncwarp();
  if (valid && rank == 0) cnt[e_a] = __popc(peers);
  __syncwarp();
  // exclusive scan: each lane a run of consecutive experts
  const int per = ceil_div(E, 32);
  int local = 0;
  for (int i = 0; i < per; ++i) {
    const int e = lane * per + i;
    if (e < E) local += cnt[e];
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(FT_FULL_MASK, incl, o);
    if (lane >= o) incl += y;
  }
  int run = incl - local;
  for (int i = 0; i < per; ++i) {
    const int e = lane * per + i;
    if (e < E) {
      const int c = cnt[e];
      counts[e] = c;
      offsets[e] = run;
      cnt[e] = run;
      run += c;
    }
  }
  if (lane == 0) offsets[E] = n;
  __syncwarp();
  if (valid) {
    const int pos = cnt[e_a] + rank;
    perm[pos] = lane;
    inv[lane] = pos;
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
// Router logits, top-k and the permutation of a small batch (T <= RW_MAXT, one
// chunk of rows) in one launch over the grid of router_logits_kernel, so the
// router matrix is read by many SMs at once:
//   1. each CTA computes the logits of the rows for its experts (the same
//      per-expert arithmetic as router_logits_kernel: bit-identical logits);
//   2. the CTA that arrives last on an arrival counter (after a fence) routes
//      the rows, one warp each, and groups the T*k assignments (one warp when
//      they fit in one, else the whole CTA).
// The counter lives in a caller-owned, zero-initialised device word; the last
// arrival puts it back to zero, so every call finds it zeroed.  Nothing
// waits: a CTA that is not last simply exits.  (Larger batches are faster as
// router_logits_kernel, route_kernel and permute_kernel: eight and more rows
// route in parallel over several CTAs, and the 1024-thread grouping is quicker
// than one CTA's.)
constexpr int RW_MAXT = 8;
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
                  int H, int E, int k, float* z, int32_t* __restrict__ idx_out, float* __restrict__ w_out,
                  int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                  int32_t* __restrict__ inv, uint32_t* __restrict__ arrivals) {
  static_assert(RT <= RW_MAXT, "one chunk of rows");
  extern __shared__ __align__(16) unsigned char rw_smem[];
  XT* xs = reinterpret_cast<XT*>(rw_smem);  // [RT][H] staged rows; the grouping tables of the last CTA afterwards
  __shared__ int s_flag;
  __shared__ int32_t s_wtot[RW_WARPS];
  __shared__ int32_t s_idx[RT * RT_MAXK];   // the batch's expert ids
  pdl_begin();
  const int warp = threadIdx.x >> 5;
  const int nrows = min(RT, T);
  stage_rows<XT, RT>(x, 0, nrows, H, xs);
  __syncthreads();
  logits_of_rows<XT, RT>(xs, wr, bias, 0, nrows, H, E, blockIdx.x * RW_WARPS + warp, gridDim.x * RW_WARPS, z);
  if (!last_arrival(arrivals, gridDim.x, &s_flag)) {
    pdl_end();
    return;
  }
  for (int r = warp; r < nrows; r += RW_WARPS)
    route_token<PER_LANE>(z + (size_t)r * E, E, k, idx_out + (size_t)r * k, w_out + (size_t)r * k, s_idx + r * k);
  __syncthreads();
  const int n = nrows * k;
  int32_t* tab = reinterpret_cast<int32_t*>(rw_smem);
  if (n <= 32) {
    if (warp == 0) permute_warp(threadIdx.x < n ? s_idx[threadIdx.x] : -1, n, E, counts, offsets, perm, inv, tab);
  } else {
    permute_block<RW_WARPS, true>(s_idx, n, E, counts, offsets, perm, inv, tab, s_wtot);
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
