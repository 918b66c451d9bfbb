// Shared slot-pool LRU expert cache: device tables, the per-step control kernel,
// the fixed-shape miss-fill kernel and the safe-point host operations.
#pragma once
#include <algorithm>
#include <vector>

#include "common.cuh"

struct ft_cache {
  int L, E, Lp, N, max_slots;
  uint64_t S;
  const uint8_t* host;      // pinned host pool (host address)
  const uint8_t* host_dev;  // the same memory as seen by kernels
  uint8_t* pool;
  // device tables
  int32_t* slot_of_key;     // [L*E], -1 absent
  int32_t* key_of_slot;     // [max_slots], -1 empty
  uint32_t* stamp;          // [max_slots], 0 for empty
  uint32_t* clock;          // [1]
  unsigned long long* stats;  // [5] steps, hits, fills, externals, bytes
  int32_t* fill_src;        // [E] host row
  int32_t* fill_dst;        // [E] slot
  int32_t* n_fill;          // [1]
  int fill_grid;
  cudaEvent_t ev_ctrl;      // split steps: control done on the compute stream
  cudaEvent_t ev_fill;      // split steps: fill done on the fill stream
  int pending_join;         // a split step's fill has not been joined yet
  int streaming;            // a stream handle holds the last 2E slots
  int n_full;               // capacity to restore after streaming
  int dev;
};

namespace ft {

constexpr int CC_THREADS = 1024;
constexpr int CC_WARPS = CC_THREADS / 32;
constexpr int CACHE_MAX_SLOTS = 16384;
constexpr int CACHE_MAX_E = 1024;

struct CacheDev {
  int L, E, Lp, N;
  uint64_t S;
  int32_t* slot_of_key;
  int32_t* key_of_slot;
  uint32_t* stamp;
  uint32_t* clock;
  unsigned long long* stats;
  int32_t* fill_src;
  int32_t* fill_dst;
  int32_t* n_fill;
};

// exclusive scan over the 1024 threads of the block
__device__ __forceinline__ int cc_scan(int v, int* buf, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(FT_FULL_MASK, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) buf[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = buf[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(FT_FULL_MASK, wi, o);
      if (lane >= o) wi += y;
    }
    buf[lane] = wi - w;
    if (lane == 31) buf[32] = wi;
  }
  __syncthreads();
  int r = buf[warp] + incl - v;
  total = buf[32];
  __syncthreads();
  return r;
}

// One wave of one layer step (one CTA).  Shared memory: touched flags [N]
// bytes and the victims [E].  With slot_fill (the split form) the filled
// experts' slots go there and slot_of keeps only the hits.
//
// Victims are the q slots this wave has not touched with the smallest
// (stamp, slot): empty slots hold stamp 0 and so come first, by slot; the
// others follow from least to most recently used.  They are found by q rounds
// of a block-wide minimum over the slots' keys, so no recency list is kept:
// a wave without misses touches only its hits' entries.  Each miss costs a
// whole expert over the host link, so the rounds are never the step's cost.
__global__ void __launch_bounds__(CC_THREADS)
cache_control_kernel(CacheDev d, int layer, const int32_t* __restrict__ counts, double ratio, int wave,
                     int32_t* __restrict__ slot_of, int32_t* __restrict__ slot_fill, int32_t* __restrict__ ext_flags,
                     int32_t* __restrict__ step_counts) {
  extern __shared__ __align__(16) unsigned char cc_smem[];
  __shared__ int buf[33];
  __shared__ unsigned long long s_min[CC_WARPS];
  pdl_begin();
  const int N = d.N, E = d.E;
  int32_t* s_victim = reinterpret_cast<int32_t*>(cc_smem);                   // [E]
  unsigned char* s_touched = reinterpret_cast<unsigned char*>(s_victim + E);  // [N]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  for (int s = tid; s < N; s += CC_THREADS) s_touched[s] = 0;
  // experts: thread e (E <= 1024)
  const int e = tid;
  const bool valid_e = e < E;
  const bool routed = valid_e && counts[e] > 0;
  int nU;
  const int rank = cc_scan(routed ? 1 : 0, buf, nU);
  const int w0 = wave * N;
  const bool in_wave = routed && rank >= w0 && rank < w0 + N;
  if (valid_e) {
    slot_of[e] = -1;
    if (slot_fill) slot_fill[e] = -1;
    if (wave == 0 && ext_flags) ext_flags[e] = 0;
  }
  const int nW = max(0, min(N, nU - w0));
  if (nW == 0) {
    if (tid == 0) {
      *d.n_fill = 0;
      if (step_counts) { step_counts[0] = 0; step_counts[1] = 0; step_counts[2] = 0; step_counts[3] = 0; }
    }
    pdl_end();
    return;
  }
  const uint32_t c = *d.clock + 1;
  const int key = layer * E + e;
  bool miss = false;
  if (in_wave) {
    const int s = d.slot_of_key[key];
    if (s >= 0) {
      if (s >= N || d.key_of_slot[s] != key) {
        record_error(FT_DERR_TABLE);
        miss = true;
      } else {
        d.stamp[s] = c;
        s_touched[s] = 1;
        slot_of[e] = s;
      }
    } else {
      miss = true;
    }
  }
  int m;
  const int mrank = cc_scan(miss ? 1 : 0, buf, m);  // its barriers also publish the touched flags
  const int q = qsplit_ratio(m, ratio);
  const bool fill = miss && mrank < q;
  if (miss && !fill) {
    slot_of[e] = -2;
    if (ext_flags) ext_flags[e] = 1;
  }
  if (q > 0) {
    // keys (stamp, slot) of the slots not touched by this wave; slot s = tid + i * CC_THREADS
    constexpr int MAXI = CACHE_MAX_SLOTS / CC_THREADS;
    constexpr unsigned long long kNone = ~0ull;
    unsigned long long kk[MAXI];
#pragma unroll
    for (int i = 0; i < MAXI; ++i) {
      const int s = tid + i * CC_THREADS;
      kk[i] = (s < N && !s_touched[s]) ? (((unsigned long long)d.stamp[s] << 32) | (unsigned)s) : kNone;
    }
    for (int r = 0; r < q; ++r) {
      unsigned long long best = kk[0];
#pragma unroll
      for (int i = 1; i < MAXI; ++i) best = min(best, kk[i]);
#pragma unroll
      for (int o = 16; o; o >>= 1) best = min(best, __shfl_xor_sync(FT_FULL_MASK, best, o));
      if (lane == 0) s_min[warp] = best;
      __syncthreads();
      if (warp == 0) {
        unsigned long long v = s_min[lane];
#pragma unroll
        for (int o = 16; o; o >>= 1) v = min(v, __shfl_xor_sync(FT_FULL_MASK, v, o));
        if (lane == 0) s_victim[r] = v == kNone ? -1 : (int)(v & 0xffffffffu);
      }
      __syncthreads();
      const int vs = s_victim[r];
      if (vs >= 0 && vs % CC_THREADS == tid) kk[vs / CC_THREADS] = kNone;
    }
  }
  if (fill) {
    const int v = s_victim[mrank];
    if (v < 0) {
      record_error(FT_DERR_TABLE);  // fewer free or untouched slots than fills: not reachable with nW <= N
    } else {
      const int old = d.key_of_slot[v];
      if (old >= 0) d.slot_of_key[old] = -1;
      d.key_of_slot[v] = key;
      d.slot_of_key[key] = v;
      d.stamp[v] = c;
      if (slot_fill) slot_fill[e] = v;
      else slot_of[e] = v;
      d.fill_src[mrank] = (layer % d.Lp) * E + e;
      d.fill_dst[mrank] = v;
    }
  }
  if (tid == 0) {
    *d.clock = c;
    *d.n_fill = q;
    d.stats[0] += 1;
    d.stats[1] += (unsigned long long)(nW - m);
    d.stats[2] += (unsigned long long)q;
    d.stats[3] += (unsigned long long)(m - q);
    d.stats[4] += (unsigned long long)q * d.S;
    if (step_counts) { step_counts[0] = nW; step_counts[1] = nW - m; step_counts[2] = q; step_counts[3] = m - q; }
  }
  pdl_end();
}

// One 16-byte load from the mapped pinned host pool, read-only path, with the
// L2 asked to fetch the whole 256-byte block around it. With 8 fill blocks the
// fill alone saturates the link either way; beside the hits' expert call (the
// split step) the larger requests raised 64-token decode throughput by 5% and
// left 1- to 16-token steps unchanged.
__device__ __forceinline__ uint4 ld_host_256(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Copies the filled experts host pool -> slots: one fixed-shape launch over a
// device-resident (source row, destination slot) table with a device count.
// Reads go over the host link from mapped pinned memory.
constexpr int FILL_THREADS = 256;
constexpr uint64_t FILL_CHUNK = 64 * 1024;

__global__ void __launch_bounds__(FILL_THREADS)
cache_fill_kernel(const uint8_t* __restrict__ host, uint8_t* __restrict__ pool, uint64_t S, int n_rows_host, int n_slots,
                  const int32_t* __restrict__ src, const int32_t* __restrict__ dst, const int32_t* __restrict__ n_fill) {
  pdl_begin();
  const int n = *n_fill;
  const uint64_t cpe = (S + FILL_CHUNK - 1) / FILL_CHUNK;
  const uint64_t items = (uint64_t)n * cpe;
  for (uint64_t it = blockIdx.x; it < items; it += gridDim.x) {
    const int i = (int)(it / cpe);
    const uint64_t c = it - (uint64_t)i * cpe;
    const int sr = src[i], ds = dst[i];
    if ((unsigned)sr >= (unsigned)n_rows_host || (unsigned)ds >= (unsigned)n_slots) {
      if (threadIdx.x == 0) record_error(FT_DERR_SLOT_INDEX);
      continue;
    }
    const uint64_t b = c * FILL_CHUNK;
    const uint64_t len = min(FILL_CHUNK, S - b);
    const uint4* sp = reinterpret_cast<const uint4*>(host + (uint64_t)sr * S + b);
    uint4* dp = reinterpret_cast<uint4*>(pool + (uint64_t)ds * S + b);
    const int nv = (int)(len / 16);
    constexpr int U = 4;
    for (int v0 = threadIdx.x; v0 < nv; v0 += FILL_THREADS * U) {
      uint4 t[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + u * FILL_THREADS;
        if (v < nv) t[u] = ld_host_256(sp + v);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + u * FILL_THREADS;
        if (v < nv) dp[v] = t[u];
      }
    }
  }
  pdl_end();
}

__global__ void set_buffer_slots_kernel(int32_t* slot_of, int E, int base) {
  pdl_begin();
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e < E) slot_of[e] = base + e;
  pdl_end();
}

static CacheDev cache_dev(const ft_cache* c) {
  CacheDev d;
  d.L = c->L; d.E = c->E; d.Lp = c->Lp; d.N = c->N; d.S = c->S;
  d.slot_of_key = c->slot_of_key; d.key_of_slot = c->key_of_slot; d.stamp = c->stamp;
  d.clock = c->clock; d.stats = c->stats; d.fill_src = c->fill_src; d.fill_dst = c->fill_dst; d.n_fill = c->n_fill;
  return d;
}

static size_t cache_control_smem(int N, int E) { return (size_t)E * 4 + (size_t)N; }

// ------------------------------------------------------------------ host-side table state
struct HostTables {
  std::vector<int32_t> key;     // [N]
  std::vector<uint32_t> stamp;  // [N]
  uint32_t clock = 0;
};

static int download_tables(ft_cache* c, HostTables& t) {
  FT_CHECK_CUDA(cudaDeviceSynchronize());
  t.key.resize(c->N);
  t.stamp.resize(c->N);
  if (c->N) {
    FT_CHECK_CUDA(cudaMemcpy(t.key.data(), c->key_of_slot, sizeof(int32_t) * c->N, cudaMemcpyDeviceToHost));
    FT_CHECK_CUDA(cudaMemcpy(t.stamp.data(), c->stamp, sizeof(uint32_t) * c->N, cudaMemcpyDeviceToHost));
  }
  FT_CHECK_CUDA(cudaMemcpy(&t.clock, c->clock, sizeof(uint32_t), cudaMemcpyDeviceToHost));
  return FT_OK;
}

// Writes key/stamp for slots [0, N) (N = t.key.size()) and rebuilds slot_of_key.
// Empty slots get stamp 0, which the victim search relies on.
static int upload_tables(ft_cache* c, const HostTables& t) {
  const int N = (int)t.key.size();
  std::vector<int32_t> sok((size_t)c->L * c->E, -1);
  std::vector<uint32_t> stamp(t.stamp);
  for (int s = 0; s < N; ++s) {
    if (t.key[s] >= 0) sok[t.key[s]] = s;
    else stamp[s] = 0;
  }
  if (N) {
    FT_CHECK_CUDA(cudaMemcpy(c->key_of_slot, t.key.data(), sizeof(int32_t) * N, cudaMemcpyHostToDevice));
    FT_CHECK_CUDA(cudaMemcpy(c->stamp, stamp.data(), sizeof(uint32_t) * N, cudaMemcpyHostToDevice));
  }
  FT_CHECK_CUDA(cudaMemcpy(c->slot_of_key, sok.data(), sizeof(int32_t) * sok.size(), cudaMemcpyHostToDevice));
  FT_CHECK_CUDA(cudaMemcpy(c->clock, &t.clock, sizeof(uint32_t), cudaMemcpyHostToDevice));
  c->N = N;
  return FT_OK;
}

// Safe-point rebuild to n_new slots: keep the most recent min(used, n_new)
// entries; kept entries at or above n_new move to the lowest free slots below.
static int cache_resize_impl(ft_cache* c, int n_new) {
  HostTables t;
  int st = download_tables(c, t);
  if (st) return st;
  const int N = c->N;
  std::vector<int> used;
  for (int s = 0; s < N; ++s)
    if (t.key[s] >= 0) used.push_back(s);
  std::sort(used.begin(), used.end(), [&](int a, int b) {
    return t.stamp[a] != t.stamp[b] ? t.stamp[a] > t.stamp[b] : a < b;
  });
  const int n_keep = std::min((int)used.size(), n_new);
  std::vector<char> kept(N, 0);
  for (int i = 0; i < n_keep; ++i) kept[used[i]] = 1;
  std::vector<int> movers, freeslots;
  for (int s = 0; s < N; ++s)
    if (kept[s] && s >= n_new) movers.push_back(s);
  for (int s = 0; s < std::min(N, n_new); ++s)
    if (!kept[s]) freeslots.push_back(s);
  HostTables nt;
  nt.clock = t.clock;
  nt.key.assign(n_new, -1);
  nt.stamp.assign(n_new, 0);
  for (int s = 0; s < std::min(N, n_new); ++s)
    if (kept[s]) { nt.key[s] = t.key[s]; nt.stamp[s] = t.stamp[s]; }
  for (size_t i = 0; i < movers.size(); ++i) {
    const int src = movers[i], dst = freeslots[i];
    FT_CHECK_CUDA(cudaMemcpy(c->pool + (uint64_t)dst * c->S, c->pool + (uint64_t)src * c->S, c->S,
                             cudaMemcpyDeviceToDevice));
    nt.key[dst] = t.key[src];
    nt.stamp[dst] = t.stamp[src];
  }
  st = upload_tables(c, nt);
  if (st) return st;
  FT_CHECK_CUDA(cudaDeviceSynchronize());
  return FT_OK;
}

}  // namespace ft
