// Grouped SwiGLU expert FFN for small batches (decode) with NVFP4 / MXFP4
// weights on the block-scaled FP4 tensor cores (tcgen05.mma kind::mxf4nvf4):
// the packed e2m1 weights go from the slot pool to the tensor core as they
// are, with their block scales, so no instruction is spent per weight.
//
// The other operand must be FP4 too.  The token rows are quantised once per
// call (quant_rows_kernel) and the intermediate silu(G)*U in the gate/up
// epilogue, each block of K elements on its own:
//   NVFP4 weights: blocks of 16, scale e4m3(amax / 6) (round to nearest even,
//                  saturated), values e2m1(v / scale) (nearest even, saturated)
//   MXFP4 weights: blocks of 32, scale 2^(floor(log2 amax) - 2) as E8M0,
//                  values e2m1(v / scale)
// in fp32 arithmetic with the hardware conversions.  NVFP4's fp32 matrix scale
// multiplies the fp32 results.
//
// Tiling as the bf16 small-batch kernel (expert_tc_decode.cuh): 128 weight
// rows (M) x up to 64 of an expert's token rows (N), K split when few experts
// are routed, the last split finishing the tile.  A stage carries 256 K
// elements: 128 bytes per row of weights and of tokens, plus the block scales
// of both rearranged into 512-byte atoms (32 rows x 16 bytes; tile row
// r = r0 + 32j keeps its four scales of one MMA at bytes 16 r0 + 4j) that
// tcgen05.cp copies to tensor memory, where the MMA reads them.
//
// Roles: warp 0 TMA producer (weights and token rows), warp 1 TMEM owner and
// MMA issuer, warps 2..5 epilogue, warps 6..7 build the scale atoms of each
// stage from the slot pool's scale rows and the token rows' scales.
#pragma once
#include "expert_tc_decode.cuh"

namespace ft {
namespace tc {

constexpr int BS_BK = 256;                           // K elements per stage (128 bytes of e2m1 per row)
constexpr int BS_A_BYTES = SK_MR * BS_BK / 2;        // 16 KiB of weights per stage
constexpr int BS_B_BYTES = SK_NB * BS_BK / 2;        // 8 KiB of token rows (max) per stage
constexpr int BS_ATOM = 512;
constexpr int BS_SF_BYTES = 8 * BS_ATOM;             // 4 atoms for the weights, 4 for the tokens
constexpr int BS_STAGE_BYTES = BS_A_BYTES + BS_B_BYTES + BS_SF_BYTES;
constexpr int BS_STAGES = 7;
constexpr int BS_THREADS = 256;
constexpr int BS_SF_COLS = 32;                       // tensor-memory columns of one stage's scales
constexpr int BS_SC_COL0 = 2 * SK_ACC_COLS;          // scales after the two accumulators
constexpr int BS_TMEM_COLS = 512;                    // 128 + 7 x 32 = 352, rounded up to a power of two

__host__ __device__ constexpr size_t bs_smem_bytes(int E) {
  return 1024 + (size_t)BS_STAGES * BS_STAGE_BYTES + 512 + SK_EX_BYTES + (size_t)(2 * E + 2) * 4;
}

// ------------------------------------------------------------------ FP4 quantisation (fp32, hardware conversions)
__device__ __forceinline__ uint32_t cvt_e4m3_byte(float v) {  // round to nearest even, saturated at 448
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return r & 0xffu;
}

// Two values -> one byte of e2m1 codes, the first in the low nibble.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Scale byte of a block with absolute maximum amax: e4m3(amax / 6) for NVFP4,
// the E8M0 exponent floor(log2 amax) - 2 (+127) for MXFP4; and the factor that
// maps the block's values to the e2m1 range (1 / scale, or 0 for an all-zero
// NVFP4 block).
template <int WT>
__device__ __forceinline__ uint32_t block_scale(float amax, float& inv) {
  if (WT == FT_W_NVFP4) {
    const uint32_t b = cvt_e4m3_byte(__fdiv_rn(amax, 6.0f));
    const float s = e4m3_to_float((uint8_t)b);
    inv = s > 0.0f ? s : 0.0f;  // divided by below (0: the block stays zero)
    return b;
  }
  int e = (int)((__float_as_uint(amax) >> 23) & 0xffu) - 127 - 2;  // floor(log2 amax) - 2 (amax normal)
  e = max(-127, min(126, e));
  inv = __uint_as_float((uint32_t)(127 - e) << 23);                // 2^-e, exact
  return (uint32_t)(e + 127);
}

template <int WT>
__device__ __forceinline__ float to_e2m1_range(float v, float inv) {
  if (WT == FT_W_NVFP4) return inv > 0.0f ? __fdiv_rn(v, inv) : 0.0f;
  return v * inv;
}

// Token rows in permuted order, quantised: xq[p][K/2] e2m1 bytes and xs[p][K/blk]
// scale bytes for row p = assignment perm[p] (token perm[p] / k; perm NULL: row
// p of x).  One thread per block of 16 (NVFP4) or 32 (MXFP4) elements.  Also
// clears the split counters.
template <typename XT, int WT>
__global__ void __launch_bounds__(256)
quant_rows_kernel(const XT* __restrict__ x, const int32_t* __restrict__ perm, int T, int k, int K, int Tk,
                  uint8_t* __restrict__ xq, uint8_t* __restrict__ xs, int32_t* __restrict__ zero, int n_zero) {
  pdl_begin();
  constexpr int BLK = WT == FT_W_NVFP4 ? 16 : 32;
  const int nb = K / BLK;
  const long long total = (long long)Tk * nb;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    const int p = (int)(i / nb), b = (int)(i % nb);
    const int a = perm ? perm[p] : p;  // no permutation: row p of x
    if ((unsigned)a >= (unsigned)(T * k)) {
      record_error(FT_DERR_ROW_INDEX);
      continue;
    }
    const XT* src = x + (size_t)(a / k) * K + (size_t)b * BLK;
    float v[BLK];
#pragma unroll
    for (int j = 0; j < BLK; j += 8) load8<XT>(src + j, *reinterpret_cast<float(*)[8]>(v + j));
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < BLK; ++j) amax = fmaxf(amax, fabsf(v[j]));
    float inv;
    xs[(size_t)p * nb + b] = (uint8_t)block_scale<WT>(amax, inv);
    uint32_t w[BLK / 8];
#pragma unroll
    for (int j = 0; j < BLK / 8; ++j) {
      uint32_t word = 0;
#pragma unroll
      for (int h = 0; h < 4; ++h)
        word |= cvt_e2m1x2(to_e2m1_range<WT>(v[8 * j + 2 * h], inv), to_e2m1_range<WT>(v[8 * j + 2 * h + 1], inv))
                << (8 * h);
      w[j] = word;
    }
    uint8_t* dst = xq + (size_t)p * (K / 2) + (size_t)b * (BLK / 2);
    if (BLK == 16) *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    else *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_zero; i += gridDim.x * blockDim.x) zero[i] = 0;
  pdl_end();
}

struct BsArgs {
  int T, k, H, I, E, pool_slots;
  int KS;
  int nb_box;
  const int32_t* offsets;
  const int32_t* slot_of;
  const uint8_t* pool;
  uint64_t S;
  uint64_t off_scale[3];
  uint64_t off_gscale;
  const uint8_t* bscale;  // scales of the token-side operand: [T*k][K/blk] (x for gate/up, the intermediate for down)
  uint8_t* Aq;            // gate/up output: quantised intermediate [T*k][I/2]
  uint8_t* As;            //                 and its scales [T*k][I/blk]
  float* y;               // down output [T*k][H]
  float* part;
  int32_t* counters;
};

__device__ __forceinline__ SkArgs bs_as_sk(const BsArgs& b) {
  SkArgs a;
  a.T = b.T; a.k = b.k; a.H = b.H; a.I = b.I; a.E = b.E; a.pool_slots = b.pool_slots; a.KS = b.KS;
  a.nb_box = b.nb_box; a.offsets = b.offsets; a.slot_of = b.slot_of; a.pool = b.pool; a.S = b.S;
  for (int m = 0; m < 3; ++m) a.off_scale[m] = b.off_scale[m];
  a.off_gscale = b.off_gscale;
  a.Aint = nullptr; a.y = b.y; a.part = b.part; a.counters = b.counters;
  return a;
}

template <int MODE, int WT>
__global__ void __launch_bounds__(BS_THREADS, 1)
bs_skinny_kernel(const __grid_constant__ CUtensorMap map_w0, const __grid_constant__ CUtensorMap map_w1,
                 const __grid_constant__ CUtensorMap map_x, BsArgs ba) {
  using namespace sm100;
  constexpr bool MX = WT == FT_W_MXFP4;
  constexpr int BLK = MX ? 32 : 16;
  constexpr int ATOMS = MX ? 2 : 4;          // atoms per operand per stage
  const SkArgs a = bs_as_sk(ba);
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t pad = (1024 - (raw_addr & 1023)) & 1023;
  unsigned char* smem = smem_raw + pad;
  const uint32_t sbase = raw_addr + pad;
  unsigned char* tail = smem + BS_STAGES * BS_STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(tail);
  // bars: full[S], sready[S], empty[S], tfull[2], tempty[2], drain
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 3 * BS_STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_holder + 2);
  int* scan_buf = const_cast<int*>(reinterpret_cast<volatile int*>(tmem_holder + 3));  // [BS_THREADS / 32]
  float* ex = reinterpret_cast<float*>(tail + 512);                                    // [64][SK_EX_STRIDE]
  int* act_e = reinterpret_cast<int*>(tail + 512 + SK_EX_BYTES);
  int* act_pref = act_e + a.E;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto sready_bar = [&](int s) { return smem_u32(bars + BS_STAGES + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + 2 * BS_STAGES + s); };
  auto tfull_bar = [&](int b) { return smem_u32(bars + 3 * BS_STAGES + b); };
  auto tempty_bar = [&](int b) { return smem_u32(bars + 3 * BS_STAGES + 2 + b); };
  const uint32_t drain_bar = smem_u32(bars + 3 * BS_STAGES + 4);
  auto a_off = [&](int s) { return (uint32_t)(s * BS_STAGE_BYTES); };
  auto b_off = [&](int s) { return (uint32_t)(s * BS_STAGE_BYTES + BS_A_BYTES); };
  auto sf_off = [&](int s) { return (uint32_t)(s * BS_STAGE_BYTES + BS_A_BYTES + BS_B_BYTES); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < BS_STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(sready_bar(s), 2);  // the two scale warps
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
    tmem_alloc(smem_u32(tmem_holder), BS_TMEM_COLS);
    tmem_relinquish();
  }
  pdl_begin();  // set-up above touches no global memory; the expert list below reads the routing
  const int K = MODE == GATEUP ? a.H : a.I;
  const int nk = K / a.KS / BS_BK;  // stages per split
  int n_act = 0;
  const int total = sk_build_tiles<MODE, BS_THREADS>(a, act_e, act_pref, scan_buf, n_act);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const uint32_t stage_tx = BS_A_BYTES + (uint32_t)a.nb_box * (BS_BK / 2);

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (elect_one()) {
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_par = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < total; item += gridDim.x) {
        const SkTile t = sk_decode(a, act_e, act_pref, n_act, item);
        const int kbase = t.ks * nk * BS_BK;
        for (int ks = 0; ks < nk; ++ks) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1, abort_flag)) { ok = false; break; }
          const int kb = (kbase + ks * BS_BK) / 2;  // byte coordinate along K
          mbar_arrive_expect_tx(full_bar(stage), stage_tx);
          const uint32_t sa = sbase + a_off(stage);
          if (MODE == GATEUP) {
            tma_load_3d(sa, &map_w0, full_bar(stage), kb, t.mt * 64, t.slot);
            tma_load_3d(sa + BS_A_BYTES / 2, &map_w1, full_bar(stage), kb, t.mt * 64, t.slot);
          } else {
            tma_load_3d(sa, &map_w0, full_bar(stage), kb, t.mt * SK_MR, t.slot);
          }
          tma_load_2d(sbase + b_off(stage), &map_x, full_bar(stage), kb, t.row0);
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == BS_STAGES) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok)
        for (int s = 0; s < BS_STAGES; ++s)
          if (issued & (1u << s)) mbar_drain(full_bar(s), (last_par >> s) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- scale copies and MMA issuer
    if (elect_one()) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, any = false;
      for (int item = blockIdx.x; ok && item < total; item += gridDim.x) {
        const SkTile t = sk_decode(a, act_e, act_pref, n_act, item);
        const int n16 = (t.n_valid + 15) & ~15;
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * SK_ACC_COLS;
        for (int ks = 0; ks < nk; ++ks) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag)) { ok = false; break; }
          if (!mbar_wait(sready_bar(stage), phase, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sc = tmem_base + BS_SC_COL0 + stage * BS_SF_COLS;  // 16 columns weights, 16 tokens
          const uint32_t sf = sbase + sf_off(stage);
#pragma unroll
          for (int j = 0; j < ATOMS; ++j) {
            tmem_cp_scale_atom(sc + 4 * j, sdesc_rows16(sf + j * BS_ATOM));
            tmem_cp_scale_atom(sc + 16 + 4 * j, sdesc_rows16(sf + (4 + j) * BS_ATOM));
          }
          const uint64_t da = sdesc_k_sw128(sbase + a_off(stage));
          const uint64_t db = sdesc_k_sw128(sbase + b_off(stage));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {  // 4 MMAs of K = 64: 32 bytes each along the 128-byte row
            const uint32_t acc_in = (ks | kk) != 0 ? 1u : 0u;
            if (MX) {
              const uint32_t idesc = idesc_fp4_bs(SK_MR, n16, true, 2u * (kk & 1));
              mma_fp4_bs<true>(d, da + (uint64_t)(kk * 2), db + (uint64_t)(kk * 2), idesc, sc + 4 * (kk >> 1),
                               sc + 16 + 4 * (kk >> 1), acc_in);
            } else {
              const uint32_t idesc = idesc_fp4_bs(SK_MR, n16, false, 0);
              mma_fp4_bs<false>(d, da + (uint64_t)(kk * 2), db + (uint64_t)(kk * 2), idesc, sc + 4 * kk,
                                sc + 16 + 4 * kk, acc_in);
            }
          }
          any = true;
          mma_commit(empty_bar(stage));
          if (++stage == BS_STAGES) { stage = 0; phase ^= 1; }
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
    // ---------------------------------------------------------------- scale atoms (warps 6, 7)
    // Thread i (0..63) handles weight rows i and i + 64 and token row i of the tile:
    // row r's scale bytes for MMA j go to atom j, word 4 (r % 32) + r / 32.
    const int i = threadIdx.x - 192;
    const int Kr = MODE == GATEUP ? a.H : a.I;
    const uint64_t srow = (uint64_t)(Kr / BLK);          // scale bytes per matrix row
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < total; item += gridDim.x) {
      const SkTile t = sk_decode(a, act_e, act_pref, n_act, item);
      const int kbase = t.ks * nk * BS_BK;
      const uint8_t* rec = a.pool + (uint64_t)t.slot * a.S;
      for (int ks = 0; ks < nk; ++ks) {
        if (!mbar_wait(empty_bar(stage), phase ^ 1, abort_flag)) { ok = false; break; }
        const int kc = (kbase + ks * BS_BK) / BLK;       // scale index along K
        uint32_t* atoms = reinterpret_cast<uint32_t*>(smem + sf_off(stage));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int r = i + 64 * h;                      // weight row of the tile
          const uint8_t* src;
          if (MODE == GATEUP)
            src = rec + (h == 0 ? a.off_scale[0] : a.off_scale[1]) + (uint64_t)(t.mt * 64 + i) * srow + kc;
          else
            src = rec + a.off_scale[2] + (uint64_t)(t.mt * SK_MR + r) * srow + kc;
          const int w = 4 * (r & 31) + (r >> 5);
          if (MX) {
            const uint2 v = __ldg(reinterpret_cast<const uint2*>(src));
            atoms[w] = v.x;
            atoms[BS_ATOM / 4 + w] = v.y;
          } else {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(src));
            atoms[w] = v.x;
            atoms[BS_ATOM / 4 + w] = v.y;
            atoms[2 * BS_ATOM / 4 + w] = v.z;
            atoms[3 * BS_ATOM / 4 + w] = v.w;
          }
        }
        {
          // token row i (rows past the tile's last valid one get zero scales); rows 64..127 unused
          uint32_t* tatoms = atoms + 4 * BS_ATOM / 4;
          uint32_t v[4] = {0u, 0u, 0u, 0u};
          if (i < t.n_valid) {
            const uint8_t* src = ba.bscale + (size_t)(t.row0 + i) * (Kr / BLK) + kc;
            if (MX) {
              const uint2 u = *reinterpret_cast<const uint2*>(src);
              v[0] = u.x; v[1] = u.y;
            } else {
              const uint4 u = *reinterpret_cast<const uint4*>(src);
              v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
            }
          }
#pragma unroll
          for (int j = 0; j < ATOMS; ++j) {
            tatoms[j * BS_ATOM / 4 + 4 * (i & 31) + (i >> 5)] = v[j];
            tatoms[j * BS_ATOM / 4 + 4 * (i & 31) + 2 + (i >> 5)] = 0u;
          }
        }
        fence_proxy_async_smem();  // the atoms are read by tcgen05.cp (async proxy)
        __syncwarp();
        if (lane == 0) mbar_arrive(sready_bar(stage));
        if (++stage == BS_STAGES) { stage = 0; phase ^= 1; }
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
      const int nch = ((t.n_valid + 15) & ~15) / 16;
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
      mbar_arrive(tempty_bar(acc));
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }

      if (a.KS > 1) {
        float* mine = a.part + ((size_t)t.group * a.KS + t.ks) * (SK_MR * SK_NB) + (size_t)r * SK_NB;
#pragma unroll
        for (int j = 0; j < SK_NB; j += 4)
          if (j < nch * 16) *reinterpret_cast<float4*>(mine + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        __threadfence();
        named_bar_sync(1, 128);
        if (et == 0) *last_flag = atomicAdd(&a.counters[t.group], 1) == a.KS - 1;
        named_bar_sync(1, 128);
        const bool last = *last_flag;
        named_bar_sync(1, 128);
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
        const float* gs = reinterpret_cast<const float*>(a.pool + (uint64_t)t.slot * a.S + a.off_gscale);
        const float g = MODE == GATEUP ? gs[r < 64 ? 0 : 1] : gs[2];
#pragma unroll
        for (int j = 0; j < SK_NB; ++j) v[j] *= g;
      }

      if (MODE == GATEUP) {
        if (r >= 64) {
#pragma unroll
          for (int j = 0; j < SK_NB; ++j)
            if (j < t.n_valid) ex[(r - 64) * SK_EX_STRIDE + j] = v[j];
        }
        named_bar_sync(1, 128);
        if (r < 64) {
          // A = silu(G) * U for output n, quantised along n in blocks of BLK lanes
          const int n = t.mt * 64 + r;
          const int I2 = a.I / 2, nbs = a.I / BLK;
          for (int j = 0; j < SK_NB; ++j) {
            if (j >= t.n_valid) break;  // uniform across the warp
            const float av = silu(v[j]) * ex[r * SK_EX_STRIDE + j];
            float amax = fabsf(av);
#pragma unroll
            for (int o = BLK / 2; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(FT_FULL_MASK, amax, o));
            float inv;
            const uint32_t sb = block_scale<WT>(amax, inv);
            const float qv = to_e2m1_range<WT>(av, inv);
            const float qn = __shfl_down_sync(FT_FULL_MASK, qv, 1);
            const size_t row = (size_t)(t.row0 + j);
            if ((lane & 1) == 0) ba.Aq[row * I2 + n / 2] = (uint8_t)cvt_e2m1x2(qv, qn);
            if ((lane & (BLK - 1)) == 0) ba.As[row * nbs + n / BLK] = (uint8_t)sb;
          }
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
    tmem_dealloc(tmem_base, BS_TMEM_COLS);
  }
  pdl_end();
}

// ====================================================================== large batches (prefill)
// The grouped GEMM of expert_tc.cuh with FP4 weights on the block-scaled FP4
// MMA: 128 permuted token rows (M, quantised by quant_rows_kernel) x 128 weight
// rows (N: 64 gate + the same 64 up rows for gate/up, 128 rows of W_d for down)
// per tile, 256 K elements per stage, five stages.  The gate/up epilogue
// quantises the intermediate per token row (one thread per row, blocks of 16 or
// 32 along I) for the down product; down writes fp32 y.
constexpr int BG_BN = 128;
constexpr int BG_A_BYTES = BM * BS_BK / 2;        // 16 KiB of token rows
constexpr int BG_B_BYTES = BG_BN * BS_BK / 2;     // 16 KiB of weight rows
constexpr int BG_STAGE_BYTES = BG_A_BYTES + BG_B_BYTES + BS_SF_BYTES;
constexpr int BG_STAGES = 5;
constexpr int BG_THREADS = 320;                   // producer, MMA, 4 epilogue, 4 scale warps
constexpr int BG_ACC_COLS = BG_BN;
constexpr int BG_SC_COL0 = 2 * BG_ACC_COLS;
constexpr int BG_TMEM_COLS = 512;                 // 256 + 5 x 32 = 416

__host__ __device__ constexpr size_t bg_smem_bytes(int E) {
  return 1024 + (size_t)BG_STAGES * BG_STAGE_BYTES + 256 + EPI_BYTES + (size_t)(2 * E + 2) * 4;
}

template <int MODE, int WT>
__global__ void __launch_bounds__(BG_THREADS, 1)
bs_grouped_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b0,
                  const __grid_constant__ CUtensorMap map_b1, Args a, const uint8_t* __restrict__ ascale,
                  uint8_t* __restrict__ Aq, uint8_t* __restrict__ As) {
  using namespace sm100;
  constexpr bool MX = WT == FT_W_MXFP4;
  constexpr int BLK = MX ? 32 : 16;
  constexpr int ATOMS = MX ? 2 : 4;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t pad = (1024 - (raw_addr & 1023)) & 1023;
  unsigned char* smem = smem_raw + pad;
  const uint32_t sbase = raw_addr + pad;
  unsigned char* tail = smem + (size_t)BG_STAGES * BG_STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(tail);
  // bars: full[S], sready[S], empty[S], tfull[2], tempty[2], drain
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 3 * BG_STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* scan_buf = const_cast<int*>(reinterpret_cast<volatile int*>(tmem_holder + 2));  // [BG_THREADS / 32]
  uint32_t* epi_buf = reinterpret_cast<uint32_t*>(tail + 256);
  int* act_e = reinterpret_cast<int*>(tail + 256 + EPI_BYTES);
  int* act_pref = act_e + a.E;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto sready_bar = [&](int s) { return smem_u32(bars + BG_STAGES + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + 2 * BG_STAGES + s); };
  auto tfull_bar = [&](int b) { return smem_u32(bars + 3 * BG_STAGES + b); };
  auto tempty_bar = [&](int b) { return smem_u32(bars + 3 * BG_STAGES + 2 + b); };
  const uint32_t drain_bar = smem_u32(bars + 3 * BG_STAGES + 4);
  auto a_off = [&](int s) { return (uint32_t)(s * BG_STAGE_BYTES); };
  auto b_off = [&](int s) { return (uint32_t)(s * BG_STAGE_BYTES + BG_A_BYTES); };
  auto sf_off = [&](int s) { return (uint32_t)(s * BG_STAGE_BYTES + BG_A_BYTES + BG_B_BYTES); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < BG_STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(sready_bar(s), 4);  // the four scale warps
      mbar_init(empty_bar(s), 1);
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
    tmem_alloc(smem_u32(tmem_holder), BG_TMEM_COLS);
    tmem_relinquish();
  }
  pdl_begin();  // set-up above touches no global memory; the expert list below reads the routing
  const int n_tiles_n = MODE == GATEUP ? a.I / (BG_BN / 2) : ceil_div(a.H, BG_BN);
  const int K = MODE == GATEUP ? a.H : a.I;
  const int nk = K / BS_BK;
  int n_act = 0;
  const int total = build_tiles<BG_THREADS>(a, n_tiles_n, act_e, act_pref, scan_buf, n_act);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const long long Tk = (long long)a.T * a.k;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (elect_one()) {
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_par = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < total; item += gridDim.x) {
        const Tile t = decode_tile(a, act_e, act_pref, n_act, item);
        for (int ks = 0; ks < nk; ++ks) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1, abort_flag)) { ok = false; break; }
          const int kb = ks * BS_BK / 2;
          mbar_arrive_expect_tx(full_bar(stage), BG_A_BYTES + BG_B_BYTES);
          tma_load_2d(sbase + a_off(stage), &map_a, full_bar(stage), kb, t.row0);
          const uint32_t sb = sbase + b_off(stage);
          if (MODE == GATEUP) {
            tma_load_3d(sb, &map_b0, full_bar(stage), kb, t.nt * (BG_BN / 2), t.slot);
            tma_load_3d(sb + BG_B_BYTES / 2, &map_b1, full_bar(stage), kb, t.nt * (BG_BN / 2), t.slot);
          } else {
            tma_load_3d(sb, &map_b0, full_bar(stage), kb, t.nt * BG_BN, t.slot);
          }
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == BG_STAGES) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok)
        for (int s = 0; s < BG_STAGES; ++s)
          if (issued & (1u << s)) mbar_drain(full_bar(s), (last_par >> s) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- scale copies and MMA issuer
    if (elect_one()) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, any = false;
      for (int item = blockIdx.x; ok && item < total; item += gridDim.x) {
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * BG_ACC_COLS;
        for (int ks = 0; ks < nk; ++ks) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag)) { ok = false; break; }
          if (!mbar_wait(sready_bar(stage), phase, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sc = tmem_base + BG_SC_COL0 + stage * BS_SF_COLS;  // 16 columns tokens (A), 16 weights (B)
          const uint32_t sf = sbase + sf_off(stage);
#pragma unroll
          for (int j = 0; j < ATOMS; ++j) {
            tmem_cp_scale_atom(sc + 4 * j, sdesc_rows16(sf + j * BS_ATOM));
            tmem_cp_scale_atom(sc + 16 + 4 * j, sdesc_rows16(sf + (4 + j) * BS_ATOM));
          }
          const uint64_t da = sdesc_k_sw128(sbase + a_off(stage));
          const uint64_t db = sdesc_k_sw128(sbase + b_off(stage));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t acc_in = (ks | kk) != 0 ? 1u : 0u;
            if (MX)
              mma_fp4_bs<true>(d, da + (uint64_t)(kk * 2), db + (uint64_t)(kk * 2),
                               idesc_fp4_bs(BM, BG_BN, true, 2u * (kk & 1)), sc + 4 * (kk >> 1),
                               sc + 16 + 4 * (kk >> 1), acc_in);
            else
              mma_fp4_bs<false>(d, da + (uint64_t)(kk * 2), db + (uint64_t)(kk * 2),
                                idesc_fp4_bs(BM, BG_BN, false, 0), sc + 4 * kk, sc + 16 + 4 * kk, acc_in);
          }
          any = true;
          mma_commit(empty_bar(stage));
          if (++stage == BG_STAGES) { stage = 0; phase ^= 1; }
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
    // ---------------------------------------------------------------- scale atoms (warps 6..9)
    // Thread i (0..127) handles token row i (A) and weight row i (B) of the tile.
    const int i = threadIdx.x - 192;
    const uint64_t wrow = (uint64_t)(K / BLK);       // scale bytes per matrix row
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < total; item += gridDim.x) {
      const Tile t = decode_tile(a, act_e, act_pref, n_act, item);
      const uint8_t* rec = a.pool + (uint64_t)t.slot * a.S;
      const uint8_t* bsrc;
      if (MODE == GATEUP)
        bsrc = rec + (i < 64 ? a.off_scale[0] : a.off_scale[1]) + (uint64_t)(t.nt * 64 + (i & 63)) * wrow;
      else
        bsrc = rec + a.off_scale[2] + (uint64_t)(t.nt * BG_BN + i) * wrow;
      const long long arow = (long long)t.row0 + i;
      const uint8_t* asrc = arow < Tk ? ascale + (size_t)arow * wrow : nullptr;
      const int w = 4 * (i & 31) + (i >> 5);
      for (int ks = 0; ks < nk; ++ks) {
        if (!mbar_wait(empty_bar(stage), phase ^ 1, abort_flag)) { ok = false; break; }
        const int kc = ks * BS_BK / BLK;
        uint32_t* atoms = reinterpret_cast<uint32_t*>(smem + sf_off(stage));
        uint32_t va[4] = {0u, 0u, 0u, 0u}, vb[4];
        if (MX) {
          if (asrc) { const uint2 u = *reinterpret_cast<const uint2*>(asrc + kc); va[0] = u.x; va[1] = u.y; }
          const uint2 u = __ldg(reinterpret_cast<const uint2*>(bsrc + kc));
          vb[0] = u.x; vb[1] = u.y;
        } else {
          if (asrc) {
            const uint4 u = *reinterpret_cast<const uint4*>(asrc + kc);
            va[0] = u.x; va[1] = u.y; va[2] = u.z; va[3] = u.w;
          }
          const uint4 u = __ldg(reinterpret_cast<const uint4*>(bsrc + kc));
          vb[0] = u.x; vb[1] = u.y; vb[2] = u.z; vb[3] = u.w;
        }
#pragma unroll
        for (int j = 0; j < ATOMS; ++j) {
          atoms[j * BS_ATOM / 4 + w] = va[j];
          atoms[(4 + j) * BS_ATOM / 4 + w] = vb[j];
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(sready_bar(stage));
        if (++stage == BG_STAGES) { stage = 0; phase ^= 1; }
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 2..5)
    const int q = warp & 3;
    uint32_t* buf = epi_buf + (warp - 2) * 32 * EPI_STRIDE;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int item = blockIdx.x; item < total; item += gridDim.x) {
      const Tile t = decode_tile(a, act_e, act_pref, n_act, item);
      if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag)) break;
      tc_fence_after();
      const int rbase = t.mt * BM + q * 32;
      const size_t pbase = (size_t)t.row0 + q * 32;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BG_ACC_COLS;
      float gs_g = 1.0f, gs_u = 1.0f, gs_d = 1.0f;
      if (WT == FT_W_NVFP4) {
        const float* gs = reinterpret_cast<const float*>(a.pool + (uint64_t)t.slot * a.S + a.off_gscale);
        gs_g = gs[0]; gs_u = gs[1]; gs_d = gs[2];
      }
      const bool valid = rbase + lane < t.cnt;   // this lane's token row belongs to the tile's expert
      if (MODE == GATEUP) {
        // lane = token row: 32 outputs per step, quantised in blocks of BLK along I
#pragma unroll 1
        for (int c = 0; c < (BG_BN / 2) / 32; ++c) {
          uint32_t g[32], u[32];
          tmem_ld32(taddr + c * 32, g);
          tmem_ld32(taddr + BG_BN / 2 + c * 32, u);
          tmem_ld_wait();
          float av[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) av[j] = silu(__uint_as_float(g[j]) * gs_g) * (__uint_as_float(u[j]) * gs_u);
          const int n0 = t.nt * (BG_BN / 2) + c * 32;   // first output of this step
          uint32_t code[4];
          uint32_t sbytes = 0;
#pragma unroll
          for (int b = 0; b < 32 / BLK; ++b) {
            float amax = 0.0f;
#pragma unroll
            for (int j = 0; j < BLK; ++j) amax = fmaxf(amax, fabsf(av[b * BLK + j]));
            float inv;
            sbytes |= block_scale<WT>(amax, inv) << (8 * b);
#pragma unroll
            for (int j = 0; j < BLK; j += 8) {
              uint32_t word = 0;
#pragma unroll
              for (int h = 0; h < 4; ++h)
                word |= cvt_e2m1x2(to_e2m1_range<WT>(av[b * BLK + j + 2 * h], inv),
                                   to_e2m1_range<WT>(av[b * BLK + j + 2 * h + 1], inv)) << (8 * h);
              code[(b * BLK + j) / 8] = word;
            }
          }
          if (valid) {
            const size_t row = pbase + lane;
            *reinterpret_cast<uint4*>(Aq + row * (a.I / 2) + n0 / 2) = make_uint4(code[0], code[1], code[2], code[3]);
            if (MX) As[row * (a.I / 32) + n0 / 32] = (uint8_t)sbytes;
            else *reinterpret_cast<uint16_t*>(As + row * (a.I / 16) + n0 / 16) = (uint16_t)sbytes;
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < BG_BN / 32; ++c) {
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
          const int col = t.nt * BG_BN + c * 32;
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
    tmem_dealloc(tmem_base, BG_TMEM_COLS);
  }
  pdl_end();
}

}  // namespace tc
}  // namespace ft
