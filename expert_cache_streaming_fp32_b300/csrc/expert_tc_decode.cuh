// Grouped SwiGLU expert FFN on the tcgen05 tensor cores for small batches
// (decode): the weights are the 128-row M side of the MMA and an expert's few
// token rows are the N side (16..64 columns), so no tensor-core work or shared
// memory is spent on empty token rows, and every stage carries 128 weight rows.
//
//   gate/up: tile = 64 gate rows + the same 64 up rows of one expert (128 MMA
//            rows) x up to 64 of its token rows; D[n][j] = W[n] . Xp[j]
//            Aint[j][n] = bf16(silu(G[n][j]) * U[n][j])
//   down:    tile = 128 rows of W_d x up to 64 token rows;
//            Y[j][h] = W_d[h] . Aint[j]                                (fp32)
//
// With only a few experts in a step (one decode token touches k experts),
// a tile's K range is split KS ways so that enough SMs stream weights at
// once.  Each split writes its fp32 partial tile to the workspace; the CTA
// whose split finishes last (an atomic counter per tile group, no waiting)
// adds the KS partials in split order and applies the epilogue, so the result
// does not depend on which CTA finishes last.  The finishing CTA resets the
// counter, so the counters are zero again after every launch.
//
// Roles: warp 0 TMA producer, warp 1 TMEM owner and single-thread MMA issuer,
// warps 2..5 epilogue; two 64-column fp32 accumulators.
//   bf16 weights: TMA writes the 128-byte-swizzled weight tile directly.
//   NVFP4 / MXFP4 weights: TMA stages the packed e2m1 bytes (32 per row per
//   stage); warps 6..13 expand them to bf16 in the swizzled tile, half a row
//   per thread (expand_fp4_half: hardware e2m1 -> f16 conversion and an exact
//   multiply by the block scale, e4m3 or E8M0, read SCALE_AHEAD stages ahead
//   of use).  Every e2m1 value times its block scale is a bf16 number, so the
//   expansion is exact; NVFP4's fp32 matrix scale multiplies the fp32 result
//   in the epilogue.
#pragma once
#include "expert_tc.cuh"

namespace ft {
namespace tc {

constexpr int SK_NB = 64;                          // token rows per chunk (MMA N <= 64)
constexpr int SK_MR = 128;                         // weight rows per tile (MMA M)
constexpr int SK_A_BYTES = SK_MR * BK * 2;         // 16 KiB of bf16 weights per stage
constexpr int SK_B_BYTES = SK_NB * BK * 2;         // 8 KiB of token rows (max) per stage
constexpr int SK_RAW_BYTES = SK_MR * BK / 2;       // 4 KiB of packed e2m1 weights per stage
constexpr int SK_ACC_COLS = SK_NB;
constexpr int SK_TMEM_COLS = 2 * SK_ACC_COLS;
constexpr int SK_EX_STRIDE = SK_NB + 1;            // padded row of the hand-over buffer (no bank conflicts)
constexpr int SK_EX_BYTES = 64 * SK_EX_STRIDE * 4; // gate/up: up values handed to the gate rows' threads
constexpr int SK_LUT_BYTES = LUT_BYTES;             // e4m3 byte -> bf16
constexpr int SK_MAX_SPLITS = 8;

template <int WT>
struct SkCfg {
  static constexpr bool FP4 = is_fp4(WT);
  static constexpr int THREADS = FP4 ? 192 + CVT_THREADS : 192;
  static constexpr int WARPS = THREADS / 32;
  static constexpr int STAGE_BYTES = SK_A_BYTES + SK_B_BYTES + (FP4 ? SK_RAW_BYTES : 0);
  static constexpr int STAGES = FP4 ? 6 : 8;
  static constexpr int STAGE_AREA = STAGES * STAGE_BYTES;
};

template <int WT>
__host__ __device__ constexpr size_t sk_smem_bytes(int E) {
  return 1024 + (size_t)SkCfg<WT>::STAGE_AREA + 512 + SK_EX_BYTES + SK_LUT_BYTES + (size_t)(2 * E + 2) * 4;
}

// Weight-row tiles per expert.
__host__ __device__ constexpr int sk_m_tiles(int mode, int H, int I) { return mode == GATEUP ? I / 64 : H / SK_MR; }

struct SkArgs {
  int T, k, H, I, E, pool_slots;
  int KS;                 // K splits
  int nb_box;             // token rows per TMA box (16..64; fewer when the batch is tiny)
  const int32_t* offsets;
  const int32_t* slot_of;
  const uint8_t* pool;    // slot pool (block and matrix scales of the FP4 formats)
  uint64_t S;
  uint64_t off_scale[3];
  uint64_t off_gscale;
  __nv_bfloat16* Aint;    // [T*k][I]
  float* y;               // [T*k][H]
  float* part;            // split partials [groups][KS][128][SK_NB]
  int32_t* counters;      // [groups], zero between launches
};

struct SkTile {
  int e, mt, nc, ks, group, row0, n_valid, slot;
};

__device__ __forceinline__ SkTile sk_decode(const SkArgs& a, const int* act_e, const int* act_pref, int n_act,
                                            int item) {
  int lo = 0, hi = n_act - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (act_pref[mid] <= item) lo = mid; else hi = mid - 1;
  }
  SkTile t;
  t.e = act_e[lo];
  const int local = item - act_pref[lo];
  const int off = a.offsets[t.e];
  const int cnt = a.offsets[t.e + 1] - off;
  const int n_nc = ceil_div(cnt, SK_NB);
  t.ks = local % a.KS;
  const int g = local / a.KS;
  t.nc = g % n_nc;
  t.mt = g / n_nc;
  t.group = item / a.KS;  // the KS splits of one tile are consecutive items
  t.row0 = off + t.nc * SK_NB;
  t.n_valid = min(SK_NB, cnt - t.nc * SK_NB);
  t.slot = a.slot_of[t.e];
  return t;
}

// Evaluated experts and their tile prefix (as build_tiles, with the decode tiling).
template <int MODE, int NTHREADS>
__device__ int sk_build_tiles(const SkArgs& a, int* act_e, int* act_pref, int* buf, int& n_act) {
  const int n_mt = sk_m_tiles(MODE, a.H, a.I);
  const int per = ceil_div(a.E, NTHREADS);
  const int e0 = threadIdx.x * per;
  int my_act = 0, my_tiles = 0;
  for (int i = 0; i < per; ++i) {
    const int e = e0 + i;
    if (e < a.E) {
      const int cnt = a.offsets[e + 1] - a.offsets[e];
      const int s = a.slot_of[e];
      if (cnt > 0 && s >= 0) {
        if (s >= a.pool_slots) {
          record_error(FT_DERR_SLOT_INDEX);
          continue;
        }
        my_act += 1;
        my_tiles += n_mt * ceil_div(cnt, SK_NB) * a.KS;
      }
    }
  }
  int total;
  int pos = block_scan6<NTHREADS / 32>(my_act, buf, n_act);
  int tpos = block_scan6<NTHREADS / 32>(my_tiles, buf, total);
  for (int i = 0; i < per; ++i) {
    const int e = e0 + i;
    if (e < a.E) {
      const int cnt = a.offsets[e + 1] - a.offsets[e];
      const int s = a.slot_of[e];
      if (cnt > 0 && s >= 0 && s < a.pool_slots) {
        act_e[pos] = e;
        act_pref[pos] = tpos;
        pos += 1;
        tpos += n_mt * ceil_div(cnt, SK_NB) * a.KS;
      }
    }
  }
  if (threadIdx.x == 0) act_pref[n_act] = total;
  __syncthreads();
  return total;
}

template <int MODE, int WT>
__global__ void __launch_bounds__(SkCfg<WT>::THREADS, 1)
skinny_gemm_kernel(const __grid_constant__ CUtensorMap map_w0, const __grid_constant__ CUtensorMap map_w1,
                   const __grid_constant__ CUtensorMap map_x, SkArgs a) {
  using namespace sm100;
  using C = SkCfg<WT>;
  constexpr bool FP4 = C::FP4;
  constexpr int STAGES = C::STAGES;
  constexpr int STAGE_BYTES = C::STAGE_BYTES;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t pad = (1024 - (raw_addr & 1023)) & 1023;
  unsigned char* smem = smem_raw + pad;
  const uint32_t sbase = raw_addr + pad;
  unsigned char* tail = smem + C::STAGE_AREA;
  uint64_t* bars = reinterpret_cast<uint64_t*>(tail);
  // bars: full[S], cvt[S], empty[S], tfull[2], tempty[2], drain
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 3 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_holder + 2);
  int* scan_buf = const_cast<int*>(reinterpret_cast<volatile int*>(tmem_holder + 3));  // [C::WARPS]
  float* ex = reinterpret_cast<float*>(tail + 512);                                    // [64][SK_EX_STRIDE]
  uint16_t* lut_e4m3 = reinterpret_cast<uint16_t*>(tail + 512 + SK_EX_BYTES);          // [256] bf16
  int* act_e = reinterpret_cast<int*>(tail + 512 + SK_EX_BYTES + SK_LUT_BYTES);
  int* act_pref = act_e + a.E;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto cvt_bar = [&](int s) { return smem_u32(bars + STAGES + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + 2 * STAGES + s); };
  auto tfull_bar = [&](int b) { return smem_u32(bars + 3 * STAGES + b); };
  auto tempty_bar = [&](int b) { return smem_u32(bars + 3 * STAGES + 2 + b); };
  const uint32_t drain_bar = smem_u32(bars + 3 * STAGES + 4);
  // stage s: bf16 weights (1 KiB aligned) | token rows (1 KiB aligned) | packed e2m1 weights
  auto a_off = [&](int s) { return (uint32_t)(s * STAGE_BYTES); };
  auto b_off = [&](int s) { return (uint32_t)(s * STAGE_BYTES + SK_A_BYTES); };
  auto raw_off = [&](int s) { return (uint32_t)(s * STAGE_BYTES + SK_A_BYTES + SK_B_BYTES); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(cvt_bar(s), CVT_THREADS / 32);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 4 * 32);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&map_w0);
    if (MODE == GATEUP) tma_prefetch_desc(&map_w1);
    tma_prefetch_desc(&map_x);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), SK_TMEM_COLS);
    tmem_relinquish();
  }
  if (FP4) fill_fp4_tables(lut_e4m3, C::THREADS);
  pdl_begin();  // set-up above touches no global memory; the expert list below reads the routing
  const int K = MODE == GATEUP ? a.H : a.I;
  const int nk = K / a.KS / BK;  // k-steps per split
  int n_act = 0;
  const int total = sk_build_tiles<MODE, C::THREADS>(a, act_e, act_pref, scan_buf, n_act);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const uint32_t stage_tx = (FP4 ? SK_RAW_BYTES : SK_A_BYTES) + (uint32_t)a.nb_box * BK * 2;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (elect_one()) {
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_par = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < total; item += gridDim.x) {
        const SkTile t = sk_decode(a, act_e, act_pref, n_act, item);
        const int kbase = t.ks * nk * BK;
        for (int ks = 0; ks < nk; ++ks) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1, abort_flag)) { ok = false; break; }
          const int kc = kbase + ks * BK;
          mbar_arrive_expect_tx(full_bar(stage), stage_tx);
          if (FP4) {
            // packed rows: the map's innermost unit is a byte holding two K elements
            const uint32_t sr = sbase + raw_off(stage);
            if (MODE == GATEUP) {
              tma_load_3d(sr, &map_w0, full_bar(stage), kc / 2, t.mt * 64, t.slot);
              tma_load_3d(sr + SK_RAW_BYTES / 2, &map_w1, full_bar(stage), kc / 2, t.mt * 64, t.slot);
            } else {
              tma_load_3d(sr, &map_w0, full_bar(stage), kc / 2, t.mt * SK_MR, t.slot);
            }
          } else {
            const uint32_t sa = sbase + a_off(stage);
            if (MODE == GATEUP) {
              tma_load_3d(sa, &map_w0, full_bar(stage), kc, t.mt * 64, t.slot);
              tma_load_3d(sa + SK_A_BYTES / 2, &map_w1, full_bar(stage), kc, t.mt * 64, t.slot);
            } else {
              tma_load_3d(sa, &map_w0, full_bar(stage), kc, t.mt * SK_MR, t.slot);
            }
          }
          tma_load_2d(sbase + b_off(stage), &map_x, full_bar(stage), kc, t.row0);
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok)
        for (int s = 0; s < STAGES; ++s)
          if (issued & (1u << s)) mbar_drain(full_bar(s), (last_par >> s) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (elect_one()) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, any = false;
      for (int item = blockIdx.x; ok && item < total; item += gridDim.x) {
        const SkTile t = sk_decode(a, act_e, act_pref, n_act, item);
        const uint32_t idesc = idesc_bf16(SK_MR, (t.n_valid + 15) & ~15);
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * SK_ACC_COLS;
        for (int ks = 0; ks < nk; ++ks) {
          if (!mbar_wait(FP4 ? cvt_bar(stage) : full_bar(stage), phase, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint64_t da = sdesc_k_sw128(sbase + a_off(stage));
          const uint64_t db = sdesc_k_sw128(sbase + b_off(stage));
#pragma unroll
          for (int kk = 0; kk < BK / UK; ++kk)
            mma_bf16(d, da + (uint64_t)(kk * UK * 2 / 16), db + (uint64_t)(kk * UK * 2 / 16), idesc,
                     (ks | kk) != 0 ? 1u : 0u);
          any = true;
          mma_commit(empty_bar(stage));
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        mma_commit(tfull_bar(acc));
        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
      }
      if (!ok && any) {
        mma_commit(drain_bar);
        mbar_drain(drain_bar, 0);
      }
    }
  } else if (warp >= 6) {
    // ---------------------------------------------------------------- FP4 expansion (warps 6..13)
    const int cc = threadIdx.x - 192;
    const int c = cc >> 1, half = cc & 1;  // weight row of the tile and which 32 of its 64 elements
    // (selects, not an index into the parameter array, which would copy it to local memory)
    const uint64_t off_s = MODE == GATEUP ? (c < 64 ? a.off_scale[0] : a.off_scale[1]) : a.off_scale[2];
    const int krows = MODE == GATEUP ? a.H : a.I;
    const uint64_t srow = (uint64_t)krows / (WT == FT_W_NVFP4 ? 16 : 32);  // scale bytes per matrix row
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    ScaleRing<WT> ring;
    for (int item = blockIdx.x; ok && item < total; item += gridDim.x) {
      const SkTile t = sk_decode(a, act_e, act_pref, n_act, item);
      const int m = MODE == GATEUP ? t.mt * 64 + (c & 63) : t.mt * SK_MR + c;
      const uint8_t* srow_p = a.pool + (uint64_t)t.slot * a.S + off_s + (uint64_t)m * srow;
      const int kbase = t.ks * nk * BK;
      ring.start(srow_p, kbase, nk, half);
      for (int ks = 0; ks < nk; ++ks) {
        const uint32_t sc = ring.next(srow_p, kbase, nk, ks, half);
        if (!mbar_wait(full_bar(stage), phase, abort_flag)) { ok = false; break; }
        expand_fp4_half<WT>(smem + raw_off(stage) + c * 32, half, sc, lut_e4m3, smem + a_off(stage) + c * 128, c);
        fence_proxy_async_smem();  // make the generic-proxy writes visible to the tensor core
        __syncwarp();
        if (lane == 0) mbar_arrive(cvt_bar(stage));  // one arrival per converter warp
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 2..5)
    const int q = warp & 3;
    const int r = q * 32 + lane;          // weight row within the tile = TMEM lane
    const int et = threadIdx.x - 64;      // 0..127 among the epilogue threads
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int item = blockIdx.x; item < total; item += gridDim.x) {
      const SkTile t = sk_decode(a, act_e, act_pref, n_act, item);
      if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag)) break;
      tc_fence_after();
      const int nch = ((t.n_valid + 15) & ~15) / 16;  // 16-column chunks holding results
      float v[SK_NB];
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * SK_ACC_COLS;
#pragma unroll
      for (int c = 0; c < SK_NB / 16; ++c) {
        if (c < nch) {
          uint32_t u[16];
          tmem_ld16(taddr + c * 16, u);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) v[c * 16 + j] = __uint_as_float(u[j]);
        }
      }
      tc_fence_before();
      mbar_arrive(tempty_bar(acc));  // the accumulator may take the next tile now
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }

      if (a.KS > 1) {
        // publish this split's partial; the last split of the group finishes the tile
        float* mine = a.part + ((size_t)t.group * a.KS + t.ks) * (SK_MR * SK_NB) + (size_t)r * SK_NB;
#pragma unroll
        for (int j = 0; j < SK_NB; j += 4)
          if (j < nch * 16) *reinterpret_cast<float4*>(mine + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        __threadfence();
        named_bar_sync(1, 128);
        if (et == 0) *last_flag = atomicAdd(&a.counters[t.group], 1) == a.KS - 1;
        named_bar_sync(1, 128);
        const bool last = *last_flag;
        named_bar_sync(1, 128);  // everyone has read the flag before it is written again
        if (!last) continue;
        __threadfence();
        const float* base = a.part + (size_t)t.group * a.KS * (SK_MR * SK_NB) + (size_t)r * SK_NB;
#pragma unroll
        for (int j = 0; j < SK_NB; ++j) v[j] = 0.0f;
        for (int s = 0; s < a.KS; ++s) {
          const float* ps = base + (size_t)s * (SK_MR * SK_NB);
#pragma unroll
          for (int j = 0; j < SK_NB; j += 4) {
            if (j < nch * 16) {
              const float4 w = __ldcg(reinterpret_cast<const float4*>(ps + j));
              v[j] += w.x; v[j + 1] += w.y; v[j + 2] += w.z; v[j + 3] += w.w;
            }
          }
        }
        if (et == 0) a.counters[t.group] = 0;
      }
      if (WT == FT_W_NVFP4) {
        // the matrix scale of NVFP4 multiplies the finished dot products
        const float* gs = reinterpret_cast<const float*>(a.pool + (uint64_t)t.slot * a.S + a.off_gscale);
        const float g = MODE == GATEUP ? gs[r < 64 ? 0 : 1] : gs[2];
#pragma unroll
        for (int j = 0; j < SK_NB; ++j) v[j] *= g;
      }

      if (MODE == GATEUP) {
        // rows 64..127 hold U of the outputs whose G sits in rows 0..63
        if (r >= 64) {
#pragma unroll
          for (int j = 0; j < SK_NB; ++j)
            if (j < t.n_valid) ex[(r - 64) * SK_EX_STRIDE + j] = v[j];
        }
        named_bar_sync(1, 128);
        if (r < 64) {
          const int n = t.mt * 64 + r;
          __nv_bfloat16* dst = a.Aint + (size_t)t.row0 * a.I + n;
#pragma unroll
          for (int j = 0; j < SK_NB; ++j)
            if (j < t.n_valid) dst[(size_t)j * a.I] = __float2bfloat16_rn(silu(v[j]) * ex[r * SK_EX_STRIDE + j]);
        }
        named_bar_sync(1, 128);
      } else {
        const int h = t.mt * SK_MR + r;
        float* dst = a.y + (size_t)t.row0 * a.H + h;
#pragma unroll
        for (int j = 0; j < SK_NB; ++j)
          if (j < t.n_valid) dst[(size_t)j * a.H] = v[j];
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, SK_TMEM_COLS);
  }
  pdl_end();
}

}  // namespace tc
}  // namespace ft
