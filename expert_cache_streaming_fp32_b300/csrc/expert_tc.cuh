// Grouped SwiGLU expert FFN on the tcgen05 tensor cores (large batches).
//
// The gate/up and down products of every evaluated expert are dense
// contractions once an expert has tens of rows or more (prefill), so this path
// runs them as grouped GEMMs: 128-row tiles of one expert's permuted rows
// against that expert's weights, read straight from its cache slot.
//
//   gather:  Xp[p][:] = bf16(x[perm[p] / k][:])                 (rows in permuted order)
//   gate/up: Aint[p][n] = bf16(silu(Xp[p] . Wg[n]) * (Xp[p] . Wu[n]))
//   down:    Y[p][h] = Aint[p] . Wd[h]                           (fp32)
//
// One persistent kernel per product, one CTA per SM, warp-specialised:
//   warp 0      TMA producer: A tile (128 x 64 bf16) and B tile (BN x 64 bf16)
//               per stage, 128-byte swizzle, as many stages as fit in 192 KiB
//   warp 1      tensor-memory owner and MMA issuer (one thread): 4 x
//               tcgen05.mma kind::f16 (M=128, N=BN, K=16) per stage into one
//               of two BN-column fp32 accumulators
//   warps 2..5  epilogue: tcgen05.ld of the finished accumulator while the
//               next tile accumulates into the other one; results go through
//               a per-warp shared-memory transpose so that global stores are
//               whole 128-byte row segments
// BN = 256 for large batches; BN = 128 for small ones (decode), which doubles
// the number of tiles so that a handful of experts still spreads over the SMs.
// For gate/up the BN B rows are BN/2 gate rows then the same BN/2 up rows, so
// one accumulator holds G and U for the same BN/2 outputs and the SwiGLU is
// applied in registers.  Weights come through 3-D tensor maps over the whole
// slot pool (K, row, slot), so the slot is just a TMA coordinate.
//
// Rows of a tile past the end of its expert belong to the next expert (or lie
// past the last row and read as zero): their results are computed and dropped.
// Each output element is one fixed-order K reduction in the tensor core, so the
// result does not depend on the other experts of the call or on the slot.
#pragma once
#include "sm100.cuh"

namespace ft {
namespace tc {

constexpr int BM = 128;                    // rows per tile (UMMA M)
constexpr int BK = 64;                     // K per stage: 128 bytes of bf16
constexpr int UK = 16;                     // K per tcgen05.mma (kind::f16)
constexpr int THREADS = 192;
constexpr int WARPS = THREADS / 32;
constexpr int EPI_WARPS = 4;
constexpr int A_BYTES = BM * BK * 2;       // 16 KiB
constexpr int STAGE_BUDGET = 192 * 1024;   // shared memory for the operand stages
constexpr int EPI_STRIDE = 36;             // 32-bit words per staged epilogue row (32 + 4 pad)
constexpr int EPI_BYTES = EPI_WARPS * 32 * EPI_STRIDE * 4;
constexpr int MAX_E = 1024;

enum Mode { GATEUP = 0, DOWN = 1 };

constexpr int LUT_BYTES = 256 * 2;  // e4m3 byte -> bf16

__host__ __device__ constexpr bool is_fp4(int wt) { return wt == FT_W_NVFP4 || wt == FT_W_MXFP4; }

// Threads that expand FP4 rows: two per 128-row tile row (32 elements each).
constexpr int CVT_THREADS = 256;
// Stages of block scales a converter thread keeps in flight ahead of use.
constexpr int SCALE_AHEAD = 8;

// Threads that gather token rows straight from x (GA mode): one tile row
// each; every fourth issues the TMA row loads of its row and the next three.
constexpr int GATHER_THREADS = 128;

// bf16 weights: TMA writes the swizzled B tile.  NVFP4 / MXFP4: TMA stages
// the packed rows (32 bytes per row per stage) and eight more warps expand them
// (expand_fp4_half).  GA: the A tile (token rows) is gathered from x by four
// more warps with TMA tile::gather4 row loads instead of a TMA load of
// pre-gathered rows.
template <int BN, int WT = FT_W_BF16, bool GA = false>
struct Cfg {
  static_assert(BN == 128 || BN == 256, "UMMA N");
  static constexpr bool FP4 = is_fp4(WT);
  static_assert(!FP4 || BN == 128, "FP4 expansion covers 128-row weight tiles");
  static_assert(!(FP4 && GA), "one helper role per kernel");
  static constexpr int THREADS = 192 + (FP4 ? CVT_THREADS : 0) + (GA ? GATHER_THREADS : 0);
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int RAW_BYTES = FP4 ? BN * BK / 2 : 0;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + RAW_BYTES;
  static constexpr int STAGES = STAGE_BUDGET / STAGE_BYTES;  // bf16: 4 (BN 256) or 6 (BN 128); fp4 BN 128: 5
  static constexpr int ACC_COLS = BN;                        // fp32 columns per accumulator
  static constexpr int TMEM_COLS = 2 * ACC_COLS;             // double-buffered accumulators
};

// Bytes of dynamic shared memory: 1 KiB alignment slack, the stages, the
// barriers, the epilogue transpose buffers, the FP4 tables, then the expert list.
template <int BN, int WT = FT_W_BF16, bool GA = false>
__host__ __device__ constexpr size_t smem_bytes(int E) {
  return 1024 + (size_t)Cfg<BN, WT, GA>::STAGES * Cfg<BN, WT, GA>::STAGE_BYTES + 256 + EPI_BYTES + LUT_BYTES +
         (size_t)(2 * E + 2) * 4;
}

// ------------------------------------------------------------------ FP4 expansion
// Table of e4m3 byte -> bf16 bits (exact: e4m3 has 3 mantissa bits).
__device__ __forceinline__ void fill_fp4_tables(uint16_t* lut_e4m3, int nthreads) {
  for (int i = threadIdx.x; i < 256; i += nthreads) {
    __nv_bfloat16 b = __float2bfloat16_rn(e4m3_to_float((uint8_t)i));
    lut_e4m3[i] = *reinterpret_cast<uint16_t*>(&b);
  }
}

// Block scales of half a row's 64 elements at K offset kc (half = 0: elements
// 0..31, 1: 32..63): 2 e4m3 bytes (NVFP4, blocks of 16) or 1 E8M0 byte (MXFP4,
// blocks of 32).
template <int WT>
__device__ __forceinline__ uint32_t load_fp4_scales(const uint8_t* scale_row, int kc, int half) {
  if (WT == FT_W_NVFP4) return __ldg(reinterpret_cast<const uint16_t*>(scale_row + kc / 16 + 2 * half));
  return __ldg(scale_row + kc / 32 + half);
}

// Two e2m1 codes (one byte, first element in the low nibble) -> f16x2, in hardware.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(r) : "r"(byte));
  return r;
}

// bf16 bits of a block scale times 2^112 (see expand_fp4_half): e4m3 through
// the table, E8M0 b as the exponent b + 112 (b <= 142, i.e. scales up to 2^15;
// larger ones are recorded as FT_DERR_SCALE_RANGE).
template <int WT>
__device__ __forceinline__ uint32_t scale_bits_x2p112(uint32_t byte, const uint16_t* lut_e4m3) {
  if (WT == FT_W_NVFP4) return lut_e4m3[byte] + (112u << 7);
  if (byte > 142) record_error(FT_DERR_SCALE_RANGE);
  return (byte + 112u) << 7;
}

// Half a row (32 elements): 16 packed bytes -> 32 bf16 (value x block scale,
// exact) written as 4 16-byte chunks into a 128-byte-swizzled row.  Each pair
// of codes becomes f16x2 in hardware; moving an f16's bits down by three
// places reads it as a bf16 of the same sign and mantissa with the value
// scaled by 2^-112 (zero stays zero), and the multiply by the block scale
// times 2^112 restores it.  Every step is exact: e2m1 values have one
// mantissa bit, and value x scale fits bf16.
template <int WT>
__device__ __forceinline__ void expand_fp4_half(const unsigned char* raw_row, int half, uint32_t sc,
                                                const uint16_t* lut_e4m3, unsigned char* dst_row, int row) {
  const uint4 p = reinterpret_cast<const uint4*>(raw_row)[half];
  const uint32_t packed[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {  // 8 elements (one 16-byte chunk) per step
    const int j = half * 4 + jj;
    const uint32_t sbyte = WT == FT_W_NVFP4 ? (sc >> (8 * (jj >> 1))) & 0xff : sc & 0xff;
    const uint32_t sbits = scale_bits_x2p112<WT>(sbyte, lut_e4m3);
    const uint32_t s2 = sbits | (sbits << 16);
    const __nv_bfloat162 sv = *reinterpret_cast<const __nv_bfloat162*>(&s2);
    uint32_t o[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t h = e2m1x2_to_f16x2((packed[jj] >> (8 * b)) & 0xff);
      const uint32_t v = ((h >> 3) & 0x0fff0fffu) | (h & 0x80008000u);
      __nv_bfloat162 w = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&v), sv);
      o[b] = *reinterpret_cast<uint32_t*>(&w);
    }
    *reinterpret_cast<uint4*>(dst_row + ((j ^ (row & 7)) * 16)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Ring of block scales loaded SCALE_AHEAD stages before they are needed, so
// their memory latency stays off the per-stage critical path.
template <int WT>
struct ScaleRing {
  uint32_t v[SCALE_AHEAD];
  __device__ __forceinline__ void start(const uint8_t* row, int kbase, int nk, int half) {
#pragma unroll
    for (int i = 0; i < SCALE_AHEAD; ++i) v[i] = i < nk ? load_fp4_scales<WT>(row, kbase + i * BK, half) : 0u;
  }
  // scales of stage ks; loads those of stage ks + SCALE_AHEAD
  __device__ __forceinline__ uint32_t next(const uint8_t* row, int kbase, int nk, int ks, int half) {
    const uint32_t cur = v[0];
#pragma unroll
    for (int i = 0; i < SCALE_AHEAD - 1; ++i) v[i] = v[i + 1];
    const int kn = ks + SCALE_AHEAD;
    v[SCALE_AHEAD - 1] = kn < nk ? load_fp4_scales<WT>(row, kbase + kn * BK, half) : 0u;
    return cur;
  }
};

struct Args {
  int T, k, H, I, E, pool_slots;
  const int32_t* offsets;
  const int32_t* slot_of;
  const uint8_t* pool;       // slot pool (block and matrix scales of the FP4 formats)
  uint64_t off_scale[3];
  uint64_t off_gscale;
  uint64_t S;
  const __nv_bfloat16* x;    // [T][H] (GA: token rows are gathered from here)
  const int32_t* perm;       // [T*k] (GA)
  __nv_bfloat16* Aint;       // [T*k][I]
  float* y;                  // [T*k][H]
};

// ------------------------------------------------------------------ expert list
// act_e[i] = i-th evaluated expert (rows > 0, valid slot) in ascending id;
// act_pref[i] = its first tile index; act_pref[n_act] = total tiles.
// Exclusive scan over the NW warps of the block; buf holds NW ints.
template <int NW = WARPS>
__device__ __forceinline__ int block_scan6(int v, int* buf, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(FT_FULL_MASK, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) buf[warp] = incl;
  __syncthreads();
  int before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    const int b = buf[w];
    before += w < warp ? b : 0;
    tot += b;
  }
  __syncthreads();
  total = tot;
  return before + incl - v;
}

template <int NTHREADS>
__device__ int build_tiles(const Args& a, int n_tiles_n, int* act_e, int* act_pref, int* buf, int& n_act) {
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
        my_tiles += n_tiles_n * ceil_div(cnt, BM);
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
        tpos += n_tiles_n * ceil_div(cnt, BM);
      }
    }
  }
  if (threadIdx.x == 0) act_pref[n_act] = total;
  __syncthreads();
  return total;
}

struct Tile {
  int e, nt, mt, row0, cnt, slot;
};

// Tiles of one expert are ordered n-tile major, m-tile minor, so CTAs that run
// at the same time share the same weight tile through L2.
__device__ __forceinline__ Tile decode_tile(const Args& a, const int* act_e, const int* act_pref, int n_act,
                                            int item) {
  int lo = 0, hi = n_act - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (act_pref[mid] <= item) lo = mid; else hi = mid - 1;
  }
  Tile t;
  t.e = act_e[lo];
  const int local = item - act_pref[lo];
  const int off = a.offsets[t.e];
  t.cnt = a.offsets[t.e + 1] - off;
  const int n_mt = ceil_div(t.cnt, BM);
  t.nt = local / n_mt;
  t.mt = local - t.nt * n_mt;
  t.row0 = off + t.mt * BM;
  t.slot = a.slot_of[t.e];
  return t;
}

// ------------------------------------------------------------------ the kernel
template <int MODE, int BN, int WT, bool GA>
__global__ void __launch_bounds__(Cfg<BN, WT, GA>::THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b0,
                    const __grid_constant__ CUtensorMap map_b1, Args a) {
  using namespace sm100;
  using C = Cfg<BN, WT, GA>;
  constexpr bool FP4 = C::FP4;
  constexpr int STAGES = C::STAGES;
  constexpr int STAGE_BYTES = C::STAGE_BYTES;
  constexpr int B_BYTES = C::B_BYTES;
  constexpr int RAW_BYTES = C::RAW_BYTES;
  constexpr int ACC_COLS = C::ACC_COLS;
  constexpr int TMEM_COLS = C::TMEM_COLS;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // 1 KiB-aligned stage buffers (the 128-byte swizzle pattern repeats every 1 KiB)
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t pad = (1024 - (raw_addr & 1023)) & 1023;
  unsigned char* smem = smem_raw + pad;
  const uint32_t sbase = raw_addr + pad;
  unsigned char* tail = smem + (size_t)STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(tail);
  // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], drain, cvt[STAGES]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 3 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* scan_buf = const_cast<int*>(reinterpret_cast<volatile int*>(tmem_holder + 2));  // [C::THREADS / 32]
  uint32_t* epi_buf = reinterpret_cast<uint32_t*>(tail + 256);
  uint16_t* lut_e4m3 = reinterpret_cast<uint16_t*>(tail + 256 + EPI_BYTES);
  int* act_e = reinterpret_cast<int*>(tail + 256 + EPI_BYTES + LUT_BYTES);
  int* act_pref = act_e + a.E;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + STAGES + s); };
  auto tfull_bar = [&](int b) { return smem_u32(bars + 2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return smem_u32(bars + 2 * STAGES + 2 + b); };
  const uint32_t drain_bar = smem_u32(bars + 2 * STAGES + 4);
  auto cvt_bar = [&](int s) { return smem_u32(bars + 2 * STAGES + 5 + s); };
  // stage s: token rows (A) | bf16 weight rows (B) | packed e2m1 rows (FP4)
  auto raw_off = [&](int s) { return (uint32_t)(s * STAGE_BYTES + A_BYTES + B_BYTES); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // one arrival (the producer's, expecting the A and B bytes); in GA mode the
      // gather warps' row loads count their bytes on the same barrier
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(cvt_bar(s), CVT_THREADS / 32);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 4 * 32);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&map_a);
    tma_prefetch_desc(&map_b0);
    if (MODE == GATEUP) tma_prefetch_desc(&map_b1);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), TMEM_COLS);
    tmem_relinquish();
  }
  if (FP4) fill_fp4_tables(lut_e4m3, C::THREADS);
  pdl_begin();  // set-up above touches no global memory; the expert list below reads the routing
  const int n_tiles_n = MODE == GATEUP ? a.I / (BN / 2) : ceil_div(a.H, BN);
  const int K = MODE == GATEUP ? a.H : a.I;
  const int nk = K / BK;
  int n_act = 0;
  const int total = build_tiles<C::THREADS>(a, n_tiles_n, act_e, act_pref, scan_buf, n_act);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (elect_one()) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, last_par = 0;  // per stage: a load was issued / parity of its phase
      bool ok = true;
      for (int item = blockIdx.x; ok && item < total; item += gridDim.x) {
        const Tile t = decode_tile(a, act_e, act_pref, n_act, item);
        for (int ks = 0; ks < nk; ++ks) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1, abort_flag)) { ok = false; break; }
          const uint32_t sa = sbase + stage * STAGE_BYTES;
          // FP4: the packed rows go to the staging area, the map's unit is a byte of two elements
          const uint32_t sb = FP4 ? sbase + raw_off(stage) : sa + A_BYTES;
          const int kb = FP4 ? ks * BK / 2 : ks * BK;
          const uint32_t half = FP4 ? RAW_BYTES / 2 : B_BYTES / 2;
          mbar_arrive_expect_tx(full_bar(stage), A_BYTES + (FP4 ? RAW_BYTES : B_BYTES));
          if (!GA) tma_load_2d(sa, &map_a, full_bar(stage), ks * BK, t.row0);
          if (MODE == GATEUP) {
            tma_load_3d(sb, &map_b0, full_bar(stage), kb, t.nt * (BN / 2), t.slot);
            tma_load_3d(sb + half, &map_b1, full_bar(stage), kb, t.nt * (BN / 2), t.slot);
          } else {
            tma_load_3d(sb, &map_b0, full_bar(stage), kb, t.nt * BN, t.slot);
          }
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok) {
        // wind down: let every load already issued land before the CTA exits
        for (int s = 0; s < STAGES; ++s)
          if (issued & (1u << s)) mbar_drain(full_bar(s), (last_par >> s) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (elect_one()) {
      constexpr uint32_t idesc = idesc_bf16(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, any = false;
      for (int item = blockIdx.x; ok && item < total; item += gridDim.x) {
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * ACC_COLS;
        for (int ks = 0; ks < nk; ++ks) {
          if (!mbar_wait(FP4 ? cvt_bar(stage) : full_bar(stage), phase, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = sbase + stage * STAGE_BYTES;
          const uint64_t da = sdesc_k_sw128(sa);
          const uint64_t db = sdesc_k_sw128(sa + A_BYTES);
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
        // wind down: wait until every MMA issued so far has finished with TMEM and smem
        mma_commit(drain_bar);
        mbar_drain(drain_bar, 0);
      }
    }
  } else if (GA && warp >= 6) {
    // ---------------------------------------------------------------- token-row gather (warps 6..9)
    // Thread g holds the token of tile row g; per stage, every fourth lane
    // loads its row and the next three with one TMA tile::gather4 (64 columns
    // of 4 rows of x) into the 128-byte-swizzled A tile.  The bytes count on
    // the stage's full barrier, whose expected total the producer sets.
    const int g = threadIdx.x - 192;
    const long long Tk = (long long)a.T * a.k;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, last_par = 0;  // per stage: a row load was issued / parity of its phase
    for (int item = blockIdx.x; item < total; item += gridDim.x) {
      const Tile t = decode_tile(a, act_e, act_pref, n_act, item);
      const long long p = min((long long)t.row0 + g, Tk - 1);  // rows past the end: any valid row
      int tok = a.perm[p] / a.k;
      if ((unsigned)tok >= (unsigned)a.T) {
        record_error(FT_DERR_ROW_INDEX);
        tok = 0;
      }
      const int t1 = __shfl_down_sync(FT_FULL_MASK, tok, 1);
      const int t2 = __shfl_down_sync(FT_FULL_MASK, tok, 2);
      const int t3 = __shfl_down_sync(FT_FULL_MASK, tok, 3);
      bool ok = true;
      for (int ks = 0; ks < nk; ++ks) {
        if (!mbar_wait(empty_bar(stage), phase ^ 1, abort_flag)) { ok = false; break; }
        if ((lane & 3) == 0) {
          tma_gather4(sbase + stage * STAGE_BYTES + g * 128, &map_a, full_bar(stage), ks * BK, tok, t1, t2, t3);
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
        }
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
    }
    // after an abort, wait (bounded) for the row loads still in flight before the block exits
    if (*abort_flag)
      for (int s = 0; s < STAGES; ++s)
        if (issued & (1u << s)) mbar_drain(full_bar(s), (last_par >> s) & 1);
  } else if (FP4 && warp >= 6) {
    // ---------------------------------------------------------------- FP4 expansion (warps 6..13)
    const int c = threadIdx.x - 192;
    const int row = c >> 1, half = c & 1;  // B-tile row and which 32 of its 64 elements
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    ScaleRing<WT> ring;
    for (int item = blockIdx.x; ok && item < total; item += gridDim.x) {
      const Tile t = decode_tile(a, act_e, act_pref, n_act, item);
      // matrix row of B-tile row `row`; selects, not a parameter-array index
      const bool up = MODE == GATEUP && row >= BN / 2;
      const int m = MODE == GATEUP ? t.nt * (BN / 2) + (row % (BN / 2)) : t.nt * BN + row;
      const uint64_t off_s = MODE == GATEUP ? (up ? a.off_scale[1] : a.off_scale[0]) : a.off_scale[2];
      const uint8_t* srow_p =
          a.pool + (uint64_t)t.slot * a.S + off_s + (uint64_t)m * (uint64_t)(K / (WT == FT_W_NVFP4 ? 16 : 32));
      ring.start(srow_p, 0, nk, half);
      for (int ks = 0; ks < nk; ++ks) {
        const uint32_t sc = ring.next(srow_p, 0, nk, ks, half);
        if (!mbar_wait(full_bar(stage), phase, abort_flag)) { ok = false; break; }
        expand_fp4_half<WT>(smem + raw_off(stage) + row * 32, half, sc, lut_e4m3,
                            smem + stage * STAGE_BYTES + A_BYTES + row * 128, row);
        fence_proxy_async_smem();  // make the generic-proxy writes visible to the tensor core
        __syncwarp();
        if (lane == 0) mbar_arrive(cvt_bar(stage));  // one arrival per converter warp
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 2..5)
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    uint32_t* buf = epi_buf + (warp - 2) * 32 * EPI_STRIDE;  // this warp's 32 x 32 transpose buffer
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int item = blockIdx.x; item < total; item += gridDim.x) {
      const Tile t = decode_tile(a, act_e, act_pref, n_act, item);
      if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag)) break;
      tc_fence_after();
      const int rbase = t.mt * BM + q * 32;   // expert-local row of this warp's first lane
      const size_t pbase = (size_t)t.row0 + q * 32;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * ACC_COLS;
      // NVFP4: the fp32 matrix scales multiply the finished dot products
      float gs_g = 1.0f, gs_u = 1.0f, gs_d = 1.0f;
      if (WT == FT_W_NVFP4) {
        const float* gs = reinterpret_cast<const float*>(a.pool + (uint64_t)t.slot * a.S + a.off_gscale);
        gs_g = gs[0]; gs_u = gs[1]; gs_d = gs[2];
      }
      if (MODE == GATEUP) {
        // lane = row: 32 outputs silu(g) * u as bf16 (64 bytes), staged, then
        // written as 16-byte pieces, 4 lanes per row, 8 rows per instruction
#pragma unroll 1
        for (int c = 0; c < (BN / 2) / 32; ++c) {
          uint32_t g[32], u[32];
          tmem_ld32(taddr + c * 32, g);
          tmem_ld32(taddr + BN / 2 + c * 32, u);
          tmem_ld_wait();
          uint32_t* row = buf + lane * EPI_STRIDE;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float a0 = silu(__uint_as_float(g[2 * j]) * gs_g) * (__uint_as_float(u[2 * j]) * gs_u);
            const float a1 = silu(__uint_as_float(g[2 * j + 1]) * gs_g) * (__uint_as_float(u[2 * j + 1]) * gs_u);
            __nv_bfloat162 h2 = __floats2bfloat162_rn(a0, a1);
            row[j] = *reinterpret_cast<uint32_t*>(&h2);
          }
          __syncwarp();
          const int col = t.nt * (BN / 2) + c * 32;
#pragma unroll
          for (int it = 0; it < 4; ++it) {
            const int r = it * 8 + (lane >> 2), piece = lane & 3;
            if (rbase + r < t.cnt) {
              const uint4 v = *reinterpret_cast<const uint4*>(buf + r * EPI_STRIDE + piece * 4);
              *reinterpret_cast<uint4*>(a.Aint + (pbase + r) * a.I + col + piece * 8) = v;
            }
          }
          __syncwarp();
        }
      } else {
        // lane = row: 32 fp32 outputs (128 bytes), staged, then written as
        // 16-byte pieces, 8 lanes per row, 4 rows per instruction
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(taddr + c * 32, v);
          tmem_ld_wait();
          uint4* row = reinterpret_cast<uint4*>(buf + lane * EPI_STRIDE);
          if (WT == FT_W_NVFP4) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * gs_d);
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) row[j] = make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          __syncwarp();
          const int col = t.nt * BN + c * 32;
          if (col < a.H) {
#pragma unroll
            for (int it = 0; it < 8; ++it) {
              const int r = it * 4 + (lane >> 3), piece = lane & 7;
              if (rbase + r < t.cnt) {
                const uint4 w = *reinterpret_cast<const uint4*>(buf + r * EPI_STRIDE + piece * 4);
                *reinterpret_cast<uint4*>(a.y + (pbase + r) * a.H + col + piece * 4) = w;
              }
            }
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      mbar_arrive(tempty_bar(acc));
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
  pdl_end();
}

// ------------------------------------------------------------------ gather
// Xp[p][:] = bf16(x[perm[p] / k][:]); 16 bytes of output per thread step.
// Also clears the split counters of the decode kernels that follow it.
template <typename XT>
__global__ void __launch_bounds__(256)
gather_rows_kernel(const XT* __restrict__ x, const int32_t* __restrict__ perm, int T, int k, int H, int n_rows,
                   __nv_bfloat16* __restrict__ xp, int32_t* __restrict__ zero, int n_zero) {
  pdl_begin();
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  for (long long i = tid; i < n_zero; i += (long long)gridDim.x * blockDim.x) zero[i] = 0;
  const int vpr = H / 8;  // 16-byte output vectors per row
  const long long n = (long long)n_rows * vpr;
  for (long long i = tid; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int p = (int)(i / vpr), v = (int)(i - (long long)p * vpr);
    const int t = perm[p] / k;
    uint4 o = make_uint4(0, 0, 0, 0);
    if ((unsigned)t < (unsigned)T) {
      if constexpr (sizeof(XT) == 2) {
        o = __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * H) + v);
      } else {
        const float4* s = reinterpret_cast<const float4*>(x + (size_t)t * H) + 2 * v;
        const float4 f0 = __ldg(s), f1 = __ldg(s + 1);
        __nv_bfloat162 b0 = __floats2bfloat162_rn(f0.x, f0.y), b1 = __floats2bfloat162_rn(f0.z, f0.w);
        __nv_bfloat162 b2 = __floats2bfloat162_rn(f1.x, f1.y), b3 = __floats2bfloat162_rn(f1.z, f1.w);
        o = make_uint4(*reinterpret_cast<uint32_t*>(&b0), *reinterpret_cast<uint32_t*>(&b1),
                       *reinterpret_cast<uint32_t*>(&b2), *reinterpret_cast<uint32_t*>(&b3));
      }
    } else {
      record_error(FT_DERR_ROW_INDEX);
    }
    reinterpret_cast<uint4*>(xp + (size_t)p * H)[v] = o;
  }
  pdl_end();
}

}  // namespace tc
}  // namespace ft
