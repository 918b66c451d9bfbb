// libft: the exported C ABI (include/ft.h).  Single translation unit: the
// kernels live in the included .cuh files.
#include "common.cuh"
#include "host.cuh"
#include "route.cuh"
#include "expert.cuh"
#include "expert_tc.cuh"
#include "expert_tc_decode.cuh"
#include "expert_bs_decode.cuh"
#include "cache.cuh"
#include "stream.cuh"
#include "placement.cuh"
#include "cpu_experts.cuh"

#include <cudaTypedefs.h>

#include <map>
#include <mutex>
#include <new>
#include <utility>

using namespace ft;

#define FT_API extern "C" __attribute__((visibility("default")))

namespace {

int sms() { return dev_info().sms; }

template <typename K>
int occupancy_grid(K kernel, int threads, size_t smem) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  return per_sm * sms();
}

// Raises a kernel's dynamic shared-memory limit once per (device, kernel,
// size), so that steady-state calls -- and calls under stream capture -- make
// no attribute calls.
template <typename K>
int set_smem(K kernel, size_t smem) {
  if (smem <= 48 * 1024) return FT_OK;
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, size_t> done;
  int dev = 0;
  FT_CHECK_CUDA(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lock(mu);
  size_t& cur = done[{dev, reinterpret_cast<const void*>(kernel)}];
  if (smem > cur) {
    FT_CHECK_CUDA(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    cur = smem;
  }
  return FT_OK;
}

}  // namespace

FT_API const char* ft_status_str(int status) {
  switch (status) {
    case FT_OK: return "ok";
    case FT_EINVAL: return "invalid argument";
    case FT_ENOMEM: return "out of device memory";
    case FT_ECUDA: return "CUDA error";
    case FT_ETIMEOUT: return "timed out";
    case FT_ESTATE: return "call not allowed in this state";
    case FT_EUNSUPPORTED: return "unsupported configuration";
    case FT_EDEVICE: return "device-side index error";
    case FT_EIO: return "file could not be read";
    default: return "unknown status";
  }
}

FT_API int ft_version(void) { return 1; }

FT_API int ft_last_cuda_error(void) { return g_last_cuda_error; }

FT_API int ft_get_device_error(int* code) {
  FT_REQUIRE(code);
  int v = 0, zero = 0;
  FT_CHECK_CUDA(cudaDeviceSynchronize());
  FT_CHECK_CUDA(cudaMemcpyFromSymbol(&v, g_derr, sizeof(int)));
  FT_CHECK_CUDA(cudaMemcpyToSymbol(g_derr, &zero, sizeof(int)));
  *code = v;
  return v ? FT_EDEVICE : FT_OK;
}

FT_API int ft_debug_bounded_wait(int64_t limit_ns, int* completed, ft_cuda_stream s) {
  FT_REQUIRE(completed && limit_ns > 0 && limit_ns <= 2000000000ll);
  FT_LAUNCH(sm100::bounded_wait_probe_kernel, 1, 32, 0, s, (uint64_t)limit_ns, completed);
  return FT_OK;
}

FT_API int ft_debug_inject_failure(int site, int after) {
  FT_REQUIRE(site >= 1 && site < INJ_SITES);
  g_inject_after[site] = after < 0 ? -1 : after;
  return FT_OK;
}

FT_API int ft_debug_live_resources(int64_t* device_allocs, int64_t* streams_events) {
  FT_REQUIRE(device_allocs && streams_events);
  *device_allocs = g_live_dev_allocs.load();
  *streams_events = g_live_streams_events.load();
  return FT_OK;
}

FT_API int ft_debug_host_simd(int mode) { return host_simd_set(mode); }

FT_API int ft_expert_layout_get(int wtype, int hidden, int inter, ft_expert_layout* out) {
  FT_REQUIRE(out);
  return expert_layout(wtype, hidden, inter, out);
}

FT_API int ft_qsplit(int m, double bw_fill, double bw_host) {
  if (m <= 0) return 0;
  if (!(bw_host > bw_fill)) return m;
  return qsplit_ratio(m, bw_fill / bw_host);
}

// ------------------------------------------------------------------ pinned pool
FT_API int ft_host_alloc(uint64_t bytes, void** out) {
  FT_REQUIRE(out && bytes > 0);
  *out = nullptr;
  if (inject_fail(INJ_HOST_PIN)) return FT_ENOMEM;
  void* p = nullptr;
  cudaError_t e = cudaHostAlloc(&p, bytes, cudaHostAllocMapped | cudaHostAllocPortable);
  if (e != cudaSuccess) {
    cudaGetLastError();
    g_last_cuda_error = (int)e;
    return FT_ENOMEM;
  }
  *out = p;
  return FT_OK;
}

FT_API int ft_host_free(void* p) {
  if (!p) return FT_OK;
  FT_CHECK_CUDA(cudaFreeHost(p));
  return FT_OK;
}

FT_API int ft_pool_read(const char* path, uint64_t offset, void* dst, uint64_t bytes, int threads) {
  FT_REQUIRE(path && (dst || bytes == 0) && threads >= 0 && threads <= 256);
  if (bytes == 0) return FT_OK;
  if (threads == 0) threads = (int)std::min<unsigned>(64u, std::max(1u, std::thread::hardware_concurrency()));
  return pool_read(path, offset, dst, bytes, threads);
}

FT_API int ft_host_register(void* p, uint64_t bytes) {
  FT_REQUIRE(p && bytes > 0 && ((uintptr_t)p & 4095) == 0);
  if (inject_fail(INJ_HOST_PIN)) return FT_ENOMEM;
  cudaError_t e = cudaHostRegister(p, bytes, cudaHostRegisterMapped | cudaHostRegisterPortable);
  if (e != cudaSuccess) {
    cudaGetLastError();
    g_last_cuda_error = (int)e;
    return FT_ENOMEM;
  }
  return FT_OK;
}

FT_API int ft_host_unregister(void* p) {
  FT_REQUIRE(p);
  FT_CHECK_CUDA(cudaHostUnregister(p));
  return FT_OK;
}

// ------------------------------------------------------------------ router logits
FT_API int ft_router_logits(const void* x, int x_type, const void* w_router, const float* bias, int T, int H, int E,
                            float* logits, ft_cuda_stream s) {
  FT_REQUIRE(T >= 0 && H > 0 && H % 8 == 0 && E >= 1 && E <= 1024);
  FT_REQUIRE(x_type == FT_X_F32 || x_type == FT_X_BF16);
  if (T == 0) return FT_OK;
  FT_REQUIRE(x && w_router && logits);
  const int RT = T >= 8 ? 8 : T >= 4 ? 4 : T >= 2 ? 2 : 1;  // rows staged per CTA
  const size_t smem = (size_t)RT * H * (x_type == FT_X_BF16 ? 2 : 4);  // rows staged in x's type
  if (smem > 227 * 1024 || ceil_div(T, RT) > 65535) return FT_EUNSUPPORTED;
  const int chunks = ceil_div(T, RT);
  const int groups = std::max(1, std::min(ceil_div(E, RL_WARPS), ceil_div(2 * sms(), chunks)));
  dim3 grid(groups, chunks);
  cudaStream_t st = (cudaStream_t)s;
  auto go = [&](auto kernel, const auto* xx, const auto* ww) -> int {
    if (int r = set_smem(kernel, smem)) return r;
    FT_LAUNCH(kernel, grid, RL_WARPS * 32, smem, st, xx, ww, bias, T, H, E, logits);
    return FT_OK;
  };
  if (x_type == FT_X_BF16) {
    const auto* xx = (const __nv_bfloat16*)x;
    const auto* ww = (const __nv_bfloat16*)w_router;
    switch (RT) {
      case 1: return go(router_logits_kernel<__nv_bfloat16, 1>, xx, ww);
      case 2: return go(router_logits_kernel<__nv_bfloat16, 2>, xx, ww);
      case 4: return go(router_logits_kernel<__nv_bfloat16, 4>, xx, ww);
      default: return go(router_logits_kernel<__nv_bfloat16, 8>, xx, ww);
    }
  }
  const auto* xx = (const float*)x;
  const auto* ww = (const float*)w_router;
  switch (RT) {
    case 1: return go(router_logits_kernel<float, 1>, xx, ww);
    case 2: return go(router_logits_kernel<float, 2>, xx, ww);
    case 4: return go(router_logits_kernel<float, 4>, xx, ww);
    default: return go(router_logits_kernel<float, 8>, xx, ww);
  }
}

// ------------------------------------------------------------------ route
FT_API int ft_route(const float* logits, int T, int E, int k, int32_t* topk_idx, float* topk_w, ft_cuda_stream s) {
  FT_REQUIRE(T >= 0 && E >= 1 && E <= RT_MAXE && k >= 1 && k <= RT_MAXK && k <= E);
  if (T == 0) return FT_OK;
  FT_REQUIRE(logits && topk_idx && topk_w);
  const int warps = 8;
  dim3 grid(ceil_div(T, warps));
  cudaStream_t st = (cudaStream_t)s;
  const int per = ceil_div(E, 32);
  auto kr = per <= 1 ? route_kernel<1> : per <= 2 ? route_kernel<2> : per <= 4 ? route_kernel<4>
          : per <= 8 ? route_kernel<8> : per <= 16 ? route_kernel<16> : route_kernel<32>;
  FT_LAUNCH(kr, grid, warps * 32, 0, st, logits, T, E, k, topk_idx, topk_w);
  return FT_OK;
}

// ------------------------------------------------------------------ permute
FT_API int ft_permute(const int32_t* topk_idx, int T, int k, int E, int32_t* counts, int32_t* offsets, int32_t* perm,
                      int32_t* inv, ft_cuda_stream s) {
  FT_REQUIRE(T >= 0 && k >= 1 && E >= 1 && E <= PM_MAXE);
  FT_REQUIRE(counts && offsets);
  const long long n = (long long)T * k;
  FT_REQUIRE(n < (1ll << 30));
  FT_REQUIRE(n == 0 || (topk_idx && perm && inv));
  const size_t smem = (size_t)(2 * E + PM_WARPS * E) * sizeof(int32_t);
  if (int st = set_smem(permute_kernel, smem)) return st;
  FT_LAUNCH(permute_kernel, 1, PM_THREADS, smem, s, topk_idx, (int)n, E, counts, offsets, perm, inv);
  return FT_OK;
}

// ------------------------------------------------------------------ fused routing
static_assert(FT_ROUTE_ARRIVAL_WORDS >= 1, "arrival counter");

namespace {
template <typename XT, int RT>
int launch_route_grid(const XT* x, const XT* wr, const float* bias, int T, int H, int E, int k, float* z,
                      int32_t* idx, float* w, int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                      uint32_t* arrivals, cudaStream_t st) {
  // staged rows, and after them the last CTA's grouping tables
  const size_t smem = std::max((size_t)RT * H * sizeof(XT), (size_t)(2 + RW_WARPS) * E * sizeof(int32_t));
  const int groups = std::max(1, std::min(ceil_div(E, RW_WARPS), 2 * sms()));
  auto kr = E <= 256 ? route_grid_kernel<XT, RT, 8> : route_grid_kernel<XT, RT, 16>;
  if (int r = set_smem(kr, smem)) return r;
  FT_LAUNCH(kr, groups, RW_THREADS, smem, st, x, wr, bias, T, H, E, k, z, idx, w, counts, offsets, perm, inv,
            arrivals);
  return FT_OK;
}

template <typename XT>
int route_grid_rt(const void* x, const void* wr, const float* bias, int T, int H, int E, int k, float* z,
                  int32_t* idx, float* w, int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                  uint32_t* arrivals, cudaStream_t st) {
  const XT* xx = static_cast<const XT*>(x);
  const XT* ww = static_cast<const XT*>(wr);
  if (T > 4)
    return launch_route_grid<XT, 8>(xx, ww, bias, T, H, E, k, z, idx, w, counts, offsets, perm, inv, arrivals, st);
  if (T > 2)
    return launch_route_grid<XT, 4>(xx, ww, bias, T, H, E, k, z, idx, w, counts, offsets, perm, inv, arrivals, st);
  if (T == 2)
    return launch_route_grid<XT, 2>(xx, ww, bias, T, H, E, k, z, idx, w, counts, offsets, perm, inv, arrivals, st);
  return launch_route_grid<XT, 1>(xx, ww, bias, T, H, E, k, z, idx, w, counts, offsets, perm, inv, arrivals, st);
}
}  // namespace

FT_API int ft_route_fused(const void* x, int x_type, const void* w_router, const float* bias, int T, int H, int E,
                          int k, float* logits, int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                          int32_t* perm, int32_t* inv, uint32_t* arrivals, ft_cuda_stream s) {
  FT_REQUIRE(T >= 0 && H > 0 && H % 8 == 0 && E >= 1 && E <= PM_MAXE && k >= 1 && k <= RT_MAXK && k <= E);
  FT_REQUIRE(x_type == FT_X_F32 || x_type == FT_X_BF16);
  FT_REQUIRE(counts && offsets);
  if (T > 0) FT_REQUIRE(x && w_router && logits && topk_idx && topk_w && perm && inv);
  const int RT = T > 4 ? 8 : T > 2 ? 4 : T;  // rows staged by the one-launch form
  if (T == 0 || T > RW_MAXT || (size_t)RT * H * (x_type == FT_X_BF16 ? 2 : 4) > 200 * 1024) {
    // larger batches (and the empty one): the three kernels
    if (int r = ft_router_logits(x, x_type, w_router, bias, T, H, E, logits, s)) return r;
    if (int r = ft_route(logits, T, E, k, topk_idx, topk_w, s)) return r;
    return ft_permute(topk_idx, T, k, E, counts, offsets, perm, inv, s);
  }
  FT_REQUIRE(arrivals);
  cudaStream_t st = (cudaStream_t)s;
  if (x_type == FT_X_BF16)
    return route_grid_rt<__nv_bfloat16>(x, w_router, bias, T, H, E, k, logits, topk_idx, topk_w, counts, offsets,
                                        perm, inv, arrivals, st);
  return route_grid_rt<float>(x, w_router, bias, T, H, E, k, logits, topk_idx, topk_w, counts, offsets, perm, inv,
                              arrivals, st);
}

// ------------------------------------------------------------------ combine
FT_API int ft_combine(const float* y, const int32_t* inv, const int32_t* topk_idx, const float* topk_w,
                      const int32_t* ext_flags, const float* ext_partial, int T, int k, int H, int E, float* out,
                      ft_cuda_stream s) {
  FT_REQUIRE(T >= 0 && k >= 1 && H > 0 && H % 4 == 0 && E >= 1);
  if (T == 0) return FT_OK;
  FT_REQUIRE(y && inv && topk_idx && topk_w && out);
  FT_REQUIRE(T <= 65535 && k <= RT_MAXK);
  dim3 grid(ceil_div(H / 4, CB_THREADS), T);
  FT_LAUNCH(combine_kernel, grid, CB_THREADS, 0, s, y, inv, topk_idx, topk_w, ext_flags, ext_partial, T, k, H, E, out);
  return FT_OK;
}

// ------------------------------------------------------------------ expert grouped
static size_t align256(size_t v) { return (v + 255) / 256 * 256; }

// Workspace of the CUDA-core path: the fp32 intermediate [T*k][I].
static size_t ws_cuda_core(long long Tk, int inter) { return align256((size_t)Tk * inter * sizeof(float)); }
// Small-batch tensor-core tiling: K splits so that about one wave of tiles
// covers the SMs when a step has few experts (U <= T*k experts are routed).
static constexpr int kSplitTargetTiles = 148;
static int sk_splits(long long Tk, int n_mt, int K) {
  const long long est = std::min<long long>(Tk, 256) * n_mt;
  int ks = 1;
  while (ks < tc::SK_MAX_SPLITS && est * ks * 2 <= kSplitTargetTiles && (K / (ks * 2)) % tc::BK == 0 &&
         K / (ks * 2) >= 4 * tc::BK)
    ks *= 2;
  return ks;
}
// Upper bound of the tile groups (weight-row tile x token chunk) of one launch.
static long long sk_groups(long long Tk, int n_mt) { return (long long)n_mt * (Tk + Tk / tc::SK_NB + 1); }

// Workspace of the tensor-core path: gathered bf16 rows [T*k][H], the bf16
// intermediate [T*k][I], the split counters and the split partials of the
// small-batch kernels.  Every region grows (or stays) with T*k, so a
// workspace sized for a batch also serves every smaller batch.
struct TcWorkspace {
  size_t off_aint, off_counters, off_part, bytes;
  int ks_gu, ks_dn;
  long long g_gu, g_dn;
};
static TcWorkspace tc_workspace(long long Tk, int hidden, int inter) {
  TcWorkspace w{};
  const int mt_gu = tc::sk_m_tiles(tc::GATEUP, hidden, inter), mt_dn = tc::sk_m_tiles(tc::DOWN, hidden, inter);
  w.off_aint = align256((size_t)Tk * hidden * 2);
  size_t o = w.off_aint + align256((size_t)Tk * inter * 2);
  const long long Tk_small = std::min<long long>(Tk, FT_TC_WIDE_ASSIGNMENTS - 1);
  w.ks_gu = Tk < FT_TC_WIDE_ASSIGNMENTS ? sk_splits(Tk, mt_gu, hidden) : 1;
  w.ks_dn = Tk < FT_TC_WIDE_ASSIGNMENTS ? sk_splits(Tk, mt_dn, inter) : 1;
  w.g_gu = sk_groups(Tk_small, mt_gu);
  w.g_dn = sk_groups(Tk_small, mt_dn);
  w.off_counters = o;
  o += align256((size_t)(w.g_gu + w.g_dn) * 4);
  w.off_part = o;
  // splits happen only while an estimated wave of tiles is short, i.e. for
  // T*k up to kSplitTargetTiles: size the partials for the largest need there
  long long pg = 0;
  for (long long t = 1; t <= std::min<long long>(Tk, kSplitTargetTiles); ++t) {
    const int kg = sk_splits(t, mt_gu, hidden), kd = sk_splits(t, mt_dn, inter);
    if (kg > 1) pg = std::max(pg, sk_groups(t, mt_gu) * kg);
    if (kd > 1) pg = std::max(pg, sk_groups(t, mt_dn) * kd);
  }
  o += align256((size_t)pg * tc::SK_MR * tc::SK_NB * 4);
  w.bytes = o;
  return w;
}
static size_t ws_tensor_core(long long Tk, int hidden, int inter) { return tc_workspace(Tk, hidden, inter).bytes; }

// Enough for either path (the weight format, which picks the path, is not an argument here).
FT_API size_t ft_expert_grouped_workspace(int T, int k, int hidden, int inter) {
  if (T <= 0 || k <= 0 || inter <= 0 || hidden <= 0) return 256;
  const long long Tk = (long long)T * k;
  return std::max({ws_cuda_core(Tk, inter), ws_tensor_core(Tk, hidden, inter), (size_t)256});
}

namespace {

template <int WT>
int launch_expert(const ExpertArgs& a, cudaStream_t st) {
  constexpr int EPL = WFmt<WT>::EPL;
  const size_t head = ((size_t)(2 * a.E + 1) * 4 + 15) / 16 * 16;
  const size_t smem_gu = head + (size_t)EX_MR * staged_stride<EPL>(a.H) * sizeof(float);
  const size_t smem_dn = head + (size_t)EX_MR * staged_stride<EPL>(a.I) * sizeof(float);
  if (smem_gu > 227 * 1024 || smem_dn > 227 * 1024) return FT_EUNSUPPORTED;
  // one token: every expert has one row, and the kernels keep more weight loads in flight
  const bool one = a.T == 1;
  if (a.x_type == FT_X_BF16) {
    auto kg = one ? gateup_kernel<WT, __nv_bfloat16, true> : gateup_kernel<WT, __nv_bfloat16>;
    if (int s = set_smem(kg, smem_gu)) return s;
    FT_LAUNCH(kg, occupancy_grid(kg, EX_THREADS, smem_gu), EX_THREADS, smem_gu, st, a);
  } else {
    auto kg = one ? gateup_kernel<WT, float, true> : gateup_kernel<WT, float>;
    if (int s = set_smem(kg, smem_gu)) return s;
    FT_LAUNCH(kg, occupancy_grid(kg, EX_THREADS, smem_gu), EX_THREADS, smem_gu, st, a);
  }
  auto kd = one ? down_kernel<WT, true> : down_kernel<WT>;
  if (int s = set_smem(kd, smem_dn)) return s;
  FT_LAUNCH(kd, occupancy_grid(kd, EX_THREADS, smem_dn), EX_THREADS, smem_dn, st, a);
  return FT_OK;
}

// ------------------------------------------------------------------ tensor-core path
using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// Tensor map with box {box_inner, box_rows(, 1)}; dims[0] innermost.
int make_map(CUtensorMap* m, CUtensorMapDataType dtype, const void* base, int rank, const uint64_t* dims,
             const uint64_t* strides_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swz) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return FT_EUNSUPPORTED;
  cuuint64_t gd[3], gs[2];
  cuuint32_t bd[3] = {box_inner, box_rows, 1}, es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) gd[i] = dims[i];
  for (int i = 0; i < rank - 1; ++i) gs[i] = strides_bytes[i];
  CUresult r = enc(m, dtype, (cuuint32_t)rank, const_cast<void*>(base), gd, gs, bd, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FT_OK : FT_EINVAL;
}

// bf16 tensor map, 128-byte swizzle, box {64, rows(, 1)}.
int make_map_bf16(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                  uint32_t box_rows) {
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rank, dims, strides_bytes, tc::BK, box_rows,
                  CU_TENSOR_MAP_SWIZZLE_128B);
}

// Packed e2m1 values viewed as bytes (two K elements per byte), no swizzle,
// box {32 bytes = 64 elements, rows, 1}: [K/2 bytes][rows][slot].
int make_map_fp4(CUtensorMap* m, const void* base, int K, int rows, int slots, uint64_t S, uint32_t box_rows) {
  const uint64_t d[3] = {(uint64_t)K / 2, (uint64_t)rows, (uint64_t)slots}, st[2] = {(uint64_t)K / 2, S};
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, 3, d, st, tc::BK / 2, box_rows,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
}

// The tensor-core path takes bf16, NVFP4 and MXFP4 weights (H and I multiples
// of 128, which the record layout already requires).
// bf16 weights at up to FT_CC_MAX_ASSIGNMENTS assignments (one decode token) are matrix-vector
// products: the CUDA-core kernels stream them with two launches and no row gather.
bool tc_path_applies(int wtype, int T, int k, int H, int I, int E) {
  const long long Tk = (long long)T * k;
  if (wtype == FT_W_BF16 && Tk <= FT_CC_MAX_ASSIGNMENTS) return false;
  const bool fmt = wtype == FT_W_BF16 || tc::is_fp4(wtype);
  return fmt && H % 128 == 0 && I % 128 == 0 && E <= tc::MAX_E && Tk < (1ll << 28);
}

// Tile width: 256 columns from FT_TC_WIDE_ASSIGNMENTS assignments up (fewer,
// larger tiles), 128 below (twice the tiles, so a few experts still cover the SMs).
template <int BN, int WT, bool GA>
int launch_tc_gemms(const CUtensorMap& mx, const CUtensorMap& mg, const CUtensorMap& mu, const CUtensorMap& ma,
                    const CUtensorMap& md, const tc::Args& a, cudaStream_t st) {
  // gate/up gathers its token rows itself in GA mode; down reads the intermediate in permuted order
  const size_t smem = tc::smem_bytes<BN, WT, GA>(a.E), smem_d = tc::smem_bytes<BN, WT, false>(a.E);
  auto kg = tc::grouped_gemm_kernel<tc::GATEUP, BN, WT, GA>;
  auto kd = tc::grouped_gemm_kernel<tc::DOWN, BN, WT, false>;
  if (int s = set_smem(kg, smem)) return s;
  if (int s = set_smem(kd, smem_d)) return s;
  FT_LAUNCH(kg, sms(), (tc::Cfg<BN, WT, GA>::THREADS), smem, st, mx, mg, mu, a);
  FT_LAUNCH(kd, sms(), (tc::Cfg<BN, WT, false>::THREADS), smem_d, st, ma, md, md, a);
  return FT_OK;
}


// Small batches: weights on the MMA's M side, token rows on N, K split when few experts are routed.
template <int WT>
int launch_skinny_wt(const ExpertArgs& ea, const ft_expert_layout& L, const TcWorkspace& w, uint8_t* ws,
                     cudaStream_t st) {
  const long long Tk = (long long)ea.T * ea.k;
  const int H = ea.H, I = ea.I;
  __nv_bfloat16* xp = reinterpret_cast<__nv_bfloat16*>(ws);
  __nv_bfloat16* aint = reinterpret_cast<__nv_bfloat16*>(ws + w.off_aint);
  const int nb_box = (int)std::min<long long>(tc::SK_NB, (Tk + 15) / 16 * 16);
  CUtensorMap mg, mu, md, mx, ma;
  {
    const uint8_t* pool = ea.pool;
    const uint64_t dx[2] = {(uint64_t)H, (uint64_t)Tk}, sx[1] = {(uint64_t)H * 2};
    const uint64_t da[2] = {(uint64_t)I, (uint64_t)Tk}, sa[1] = {(uint64_t)I * 2};
    int r;
    if (tc::is_fp4(WT)) {
      r = make_map_fp4(&mg, pool + L.off_val[0], H, I, ea.pool_slots, ea.S, 64);
      if (!r) r = make_map_fp4(&mu, pool + L.off_val[1], H, I, ea.pool_slots, ea.S, 64);
      if (!r) r = make_map_fp4(&md, pool + L.off_val[2], I, H, ea.pool_slots, ea.S, tc::SK_MR);
    } else {
      const uint64_t dw[3] = {(uint64_t)H, (uint64_t)I, (uint64_t)ea.pool_slots}, sw[2] = {(uint64_t)H * 2, ea.S};
      const uint64_t dd[3] = {(uint64_t)I, (uint64_t)H, (uint64_t)ea.pool_slots}, sd[2] = {(uint64_t)I * 2, ea.S};
      r = make_map_bf16(&mg, pool + L.off_val[0], 3, dw, sw, 64);
      if (!r) r = make_map_bf16(&mu, pool + L.off_val[1], 3, dw, sw, 64);
      if (!r) r = make_map_bf16(&md, pool + L.off_val[2], 3, dd, sd, tc::SK_MR);
    }
    if (!r) r = make_map_bf16(&mx, xp, 2, dx, sx, nb_box);
    if (!r) r = make_map_bf16(&ma, aint, 2, da, sa, nb_box);
    if (r) return r;
  }
  tc::SkArgs a;
  a.T = ea.T; a.k = ea.k; a.H = H; a.I = I; a.E = ea.E; a.pool_slots = ea.pool_slots;
  a.nb_box = nb_box;
  a.offsets = ea.offsets; a.slot_of = ea.slot_of;
  a.pool = ea.pool; a.S = ea.S;
  for (int m = 0; m < 3; ++m) a.off_scale[m] = L.off_scale[m];
  a.off_gscale = L.off_gscale;
  a.Aint = aint; a.y = ea.y;
  a.part = reinterpret_cast<float*>(ws + w.off_part);
  int32_t* counters = reinterpret_cast<int32_t*>(ws + w.off_counters);
  const size_t smem = tc::sk_smem_bytes<WT>(ea.E);
  constexpr int NT = tc::SkCfg<WT>::THREADS;
  auto kg = tc::skinny_gemm_kernel<tc::GATEUP, WT>;
  auto kd = tc::skinny_gemm_kernel<tc::DOWN, WT>;
  if (int s = set_smem(kg, smem)) return s;
  if (int s = set_smem(kd, smem)) return s;
  a.KS = w.ks_gu;
  a.counters = counters;
  FT_LAUNCH(kg, sms(), NT, smem, st, mg, mu, mx, a);
  a.KS = w.ks_dn;
  a.counters = counters + w.g_gu;
  FT_LAUNCH(kd, sms(), NT, smem, st, md, md, ma, a);
  return FT_OK;
}

// Packed e2m1 bytes with the 128-byte swizzle, box {128 bytes = 256 elements, rows}: the
// operand tile of the block-scaled MMA.  3-D over the slot pool: [K/2 bytes][rows][slot].
int make_map_fp4_sw(CUtensorMap* m, const void* base, int K, int rows, int slots, uint64_t S, uint32_t box_rows) {
  const uint64_t d[3] = {(uint64_t)K / 2, (uint64_t)rows, (uint64_t)slots}, st[2] = {(uint64_t)K / 2, S};
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, 3, d, st, 128, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Splits of the block-scaled kernels: as sk_splits, with whole 256-element stages.
static int bs_splits(long long Tk, int n_mt, int K) {
  const long long est = std::min<long long>(Tk, 256) * n_mt;
  int ks = 1;
  while (ks < tc::SK_MAX_SPLITS && est * ks * 2 <= kSplitTargetTiles && (K / (ks * 2)) % tc::BS_BK == 0 &&
         K / (ks * 2) >= 2 * tc::BS_BK)
    ks *= 2;
  return ks;
}

std::atomic<int> g_fp4_path{FT_FP4_BLOCK_SCALED};

// Small batches of NVFP4 / MXFP4 weights on the block-scaled FP4 MMA: the token rows and the
// intermediate are quantised to the weights' format.  H and I multiples of 256.
template <int WT>
int launch_bs_skinny(const ExpertArgs& ea, const ft_expert_layout& L, const TcWorkspace& w, uint8_t* ws,
                     cudaStream_t st) {
  constexpr int BLK = WT == FT_W_NVFP4 ? 16 : 32;
  const long long Tk = (long long)ea.T * ea.k;
  const int H = ea.H, I = ea.I;
  uint8_t* xq = ws;
  uint8_t* xs = ws + align256((size_t)Tk * H / 2);
  uint8_t* aq = ws + w.off_aint;
  uint8_t* as = aq + align256((size_t)Tk * I / 2);
  int32_t* counters = reinterpret_cast<int32_t*>(ws + w.off_counters);
  const int mt_gu = tc::sk_m_tiles(tc::GATEUP, H, I), mt_dn = tc::sk_m_tiles(tc::DOWN, H, I);
  const int ks_gu = bs_splits(Tk, mt_gu, H), ks_dn = bs_splits(Tk, mt_dn, I);
  {
    const long long blocks = Tk * (H / BLK);
    const int grid = (int)std::max<long long>(1, std::min<long long>((blocks + 255) / 256, 8ll * sms()));
    const int n_zero = (int)(w.g_gu + w.g_dn);
    if (ea.x_type == FT_X_BF16)
      FT_LAUNCH((tc::quant_rows_kernel<__nv_bfloat16, WT>), grid, 256, 0, st, (const __nv_bfloat16*)ea.x, ea.perm,
                ea.T, ea.k, H, (int)Tk, xq, xs, counters, n_zero);
    else
      FT_LAUNCH((tc::quant_rows_kernel<float, WT>), grid, 256, 0, st, (const float*)ea.x, ea.perm, ea.T, ea.k, H,
                (int)Tk, xq, xs, counters, n_zero);
  }
  const int nb_box = (int)std::min<long long>(tc::SK_NB, (Tk + 15) / 16 * 16);
  CUtensorMap mg, mu, md, mx, ma;
  {
    const uint8_t* pool = ea.pool;
    int r = make_map_fp4_sw(&mg, pool + L.off_val[0], H, I, ea.pool_slots, ea.S, 64);
    if (!r) r = make_map_fp4_sw(&mu, pool + L.off_val[1], H, I, ea.pool_slots, ea.S, 64);
    if (!r) r = make_map_fp4_sw(&md, pool + L.off_val[2], I, H, ea.pool_slots, ea.S, tc::SK_MR);
    const uint64_t dx[2] = {(uint64_t)H / 2, (uint64_t)Tk}, sx[1] = {(uint64_t)H / 2};
    const uint64_t da[2] = {(uint64_t)I / 2, (uint64_t)Tk}, sa[1] = {(uint64_t)I / 2};
    if (!r) r = make_map(&mx, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, 2, dx, sx, 128, nb_box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!r) r = make_map(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, aq, 2, da, sa, 128, nb_box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (r) return r;
  }
  tc::BsArgs a;
  a.T = ea.T; a.k = ea.k; a.H = H; a.I = I; a.E = ea.E; a.pool_slots = ea.pool_slots;
  a.nb_box = nb_box;
  a.offsets = ea.offsets; a.slot_of = ea.slot_of;
  a.pool = ea.pool; a.S = ea.S;
  for (int m = 0; m < 3; ++m) a.off_scale[m] = L.off_scale[m];
  a.off_gscale = L.off_gscale;
  a.Aq = aq; a.As = as; a.y = ea.y;
  a.part = reinterpret_cast<float*>(ws + w.off_part);
  const size_t smem = tc::bs_smem_bytes(ea.E);
  auto kg = tc::bs_skinny_kernel<tc::GATEUP, WT>;
  auto kd = tc::bs_skinny_kernel<tc::DOWN, WT>;
  if (int s = set_smem(kg, smem)) return s;
  if (int s = set_smem(kd, smem)) return s;
  a.KS = ks_gu;
  a.bscale = xs;
  a.counters = counters;
  FT_LAUNCH(kg, sms(), tc::BS_THREADS, smem, st, mg, mu, mx, a);
  a.KS = ks_dn;
  a.bscale = as;
  a.counters = counters + w.g_gu;
  FT_LAUNCH(kd, sms(), tc::BS_THREADS, smem, st, md, md, ma, a);
  return FT_OK;
}

// Large batches of NVFP4 / MXFP4 weights on the block-scaled FP4 MMA (tokens on M, weights on N).
template <int WT>
int launch_bs_grouped(const ExpertArgs& ea, const ft_expert_layout& L, const TcWorkspace& w, uint8_t* ws,
                      cudaStream_t st) {
  constexpr int BLK = WT == FT_W_NVFP4 ? 16 : 32;
  const long long Tk = (long long)ea.T * ea.k;
  const int H = ea.H, I = ea.I;
  uint8_t* xq = ws;
  uint8_t* xs = ws + align256((size_t)Tk * H / 2);
  uint8_t* aq = ws + w.off_aint;
  uint8_t* as = aq + align256((size_t)Tk * I / 2);
  {
    const long long blocks = Tk * (H / BLK);
    const int grid = (int)std::max<long long>(1, std::min<long long>((blocks + 255) / 256, 8ll * sms()));
    int32_t* no_zero = nullptr;
    if (ea.x_type == FT_X_BF16)
      FT_LAUNCH((tc::quant_rows_kernel<__nv_bfloat16, WT>), grid, 256, 0, st, (const __nv_bfloat16*)ea.x, ea.perm,
                ea.T, ea.k, H, (int)Tk, xq, xs, no_zero, 0);
    else
      FT_LAUNCH((tc::quant_rows_kernel<float, WT>), grid, 256, 0, st, (const float*)ea.x, ea.perm, ea.T, ea.k, H,
                (int)Tk, xq, xs, no_zero, 0);
  }
  CUtensorMap mx, mg, mu, ma, md;
  {
    const uint8_t* pool = ea.pool;
    int r = make_map_fp4_sw(&mg, pool + L.off_val[0], H, I, ea.pool_slots, ea.S, tc::BG_BN / 2);
    if (!r) r = make_map_fp4_sw(&mu, pool + L.off_val[1], H, I, ea.pool_slots, ea.S, tc::BG_BN / 2);
    if (!r) r = make_map_fp4_sw(&md, pool + L.off_val[2], I, H, ea.pool_slots, ea.S, tc::BG_BN);
    const uint64_t dx[2] = {(uint64_t)H / 2, (uint64_t)Tk}, sx[1] = {(uint64_t)H / 2};
    const uint64_t da[2] = {(uint64_t)I / 2, (uint64_t)Tk}, sa[1] = {(uint64_t)I / 2};
    if (!r) r = make_map(&mx, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, 2, dx, sx, 128, tc::BM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!r) r = make_map(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, aq, 2, da, sa, 128, tc::BM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (r) return r;
  }
  tc::Args a;
  a.T = ea.T; a.k = ea.k; a.H = H; a.I = I; a.E = ea.E; a.pool_slots = ea.pool_slots;
  a.offsets = ea.offsets; a.slot_of = ea.slot_of; a.S = ea.S;
  a.pool = ea.pool;
  for (int m = 0; m < 3; ++m) a.off_scale[m] = L.off_scale[m];
  a.off_gscale = L.off_gscale;
  a.x = nullptr; a.perm = ea.perm; a.Aint = nullptr; a.y = ea.y;
  const size_t smem = tc::bg_smem_bytes(ea.E);
  auto kg = tc::bs_grouped_kernel<tc::GATEUP, WT>;
  auto kd = tc::bs_grouped_kernel<tc::DOWN, WT>;
  if (int s = set_smem(kg, smem)) return s;
  if (int s = set_smem(kd, smem)) return s;
  uint8_t* none = nullptr;
  FT_LAUNCH(kg, sms(), tc::BG_THREADS, smem, st, mx, mg, mu, a, (const uint8_t*)xs, aq, as);
  FT_LAUNCH(kd, sms(), tc::BG_THREADS, smem, st, ma, md, md, a, (const uint8_t*)as, none, none);
  return FT_OK;
}

int launch_expert_skinny(int wtype, const ExpertArgs& ea, const ft_expert_layout& L, const TcWorkspace& w,
                         uint8_t* ws, cudaStream_t st) {
  switch (wtype) {
    case FT_W_BF16: return launch_skinny_wt<FT_W_BF16>(ea, L, w, ws, st);
    case FT_W_NVFP4: return launch_skinny_wt<FT_W_NVFP4>(ea, L, w, ws, st);
    case FT_W_MXFP4: return launch_skinny_wt<FT_W_MXFP4>(ea, L, w, ws, st);
  }
  return FT_EINVAL;
}

int launch_expert_tc(int wtype, const ExpertArgs& ea, const ft_expert_layout& L, void* workspace, cudaStream_t st) {
  const long long Tk = (long long)ea.T * ea.k;
  const int H = ea.H, I = ea.I;
  const TcWorkspace w = tc_workspace(Tk, H, I);
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  __nv_bfloat16* xp = reinterpret_cast<__nv_bfloat16*>(ws);
  __nv_bfloat16* aint = reinterpret_cast<__nv_bfloat16*>(ws + w.off_aint);
  const bool skinny = Tk < FT_TC_WIDE_ASSIGNMENTS;
  // FP4 weights: the block-scaled FP4 MMA (unless the exact expansion is asked for)
  if (tc::is_fp4(wtype) && H % tc::BS_BK == 0 && I % tc::BS_BK == 0 && g_fp4_path.load() == FT_FP4_BLOCK_SCALED) {
    if (skinny)
      return wtype == FT_W_NVFP4 ? launch_bs_skinny<FT_W_NVFP4>(ea, L, w, ws, st)
                                 : launch_bs_skinny<FT_W_MXFP4>(ea, L, w, ws, st);
    return wtype == FT_W_NVFP4 ? launch_bs_grouped<FT_W_NVFP4>(ea, L, w, ws, st)
                               : launch_bs_grouped<FT_W_MXFP4>(ea, L, w, ws, st);
  }
  // large batches of bf16 rows with bf16 weights: the gate/up kernel gathers its rows itself
  const bool direct = !skinny && wtype == FT_W_BF16 && ea.x_type == FT_X_BF16;
  // otherwise gather the permuted rows (bf16); clear the split counters of the small-batch kernels
  if (!direct) {
    const long long vecs = Tk * (H / 8);
    const int grid = (int)std::min<long long>(ceil_div((int)std::min<long long>(vecs, 1ll << 30), 256), 8 * sms());
    int32_t* zero = skinny ? reinterpret_cast<int32_t*>(ws + w.off_counters) : nullptr;
    const int n_zero = skinny ? (int)(w.g_gu + w.g_dn) : 0;
    if (ea.x_type == FT_X_BF16)
      FT_LAUNCH(tc::gather_rows_kernel<__nv_bfloat16>, grid, 256, 0, st, (const __nv_bfloat16*)ea.x, ea.perm, ea.T,
                ea.k, H, (int)Tk, xp, zero, n_zero);
    else
      FT_LAUNCH(tc::gather_rows_kernel<float>, grid, 256, 0, st, (const float*)ea.x, ea.perm, ea.T, ea.k, H, (int)Tk,
                xp, zero, n_zero);
  }
  if (skinny) return launch_expert_skinny(wtype, ea, L, w, ws, st);
  CUtensorMap mx, mg, mu, ma, md;
  const uint8_t* pool = ea.pool;
  // bf16: 256-column weight tiles when H allows; FP4: 128 (deeper pipeline beside the staging buffers)
  const int BN = (wtype == FT_W_BF16 && H % 256 == 0) ? 256 : 128;
  {
    const uint64_t dx[2] = {(uint64_t)H, (uint64_t)Tk}, sx[1] = {(uint64_t)H * 2};
    const uint64_t da[2] = {(uint64_t)I, (uint64_t)Tk}, sa[1] = {(uint64_t)I * 2};
    // direct: a map over x itself with one-row boxes, for the kernel's tile::gather4 row loads
    const uint64_t dxd[2] = {(uint64_t)H, (uint64_t)ea.T};
    int r = direct ? make_map_bf16(&mx, ea.x, 2, dxd, sx, 1) : make_map_bf16(&mx, xp, 2, dx, sx, tc::BM);
    if (!r) r = make_map_bf16(&ma, aint, 2, da, sa, tc::BM);
    if (tc::is_fp4(wtype)) {
      if (!r) r = make_map_fp4(&mg, pool + L.off_val[0], H, I, ea.pool_slots, ea.S, BN / 2);
      if (!r) r = make_map_fp4(&mu, pool + L.off_val[1], H, I, ea.pool_slots, ea.S, BN / 2);
      if (!r) r = make_map_fp4(&md, pool + L.off_val[2], I, H, ea.pool_slots, ea.S, BN);
    } else {
      const uint64_t dw[3] = {(uint64_t)H, (uint64_t)I, (uint64_t)ea.pool_slots}, sw[2] = {(uint64_t)H * 2, ea.S};
      const uint64_t dd[3] = {(uint64_t)I, (uint64_t)H, (uint64_t)ea.pool_slots}, sd[2] = {(uint64_t)I * 2, ea.S};
      if (!r) r = make_map_bf16(&mg, pool + L.off_val[0], 3, dw, sw, BN / 2);
      if (!r) r = make_map_bf16(&mu, pool + L.off_val[1], 3, dw, sw, BN / 2);
      if (!r) r = make_map_bf16(&md, pool + L.off_val[2], 3, dd, sd, BN);
    }
    if (r) return r;
  }
  tc::Args a;
  a.T = ea.T; a.k = ea.k; a.H = H; a.I = I; a.E = ea.E; a.pool_slots = ea.pool_slots;
  a.offsets = ea.offsets; a.slot_of = ea.slot_of; a.S = ea.S;
  a.pool = ea.pool;
  for (int m = 0; m < 3; ++m) a.off_scale[m] = L.off_scale[m];
  a.off_gscale = L.off_gscale;
  a.x = reinterpret_cast<const __nv_bfloat16*>(ea.x);
  a.perm = ea.perm;
  a.Aint = aint; a.y = ea.y;
  switch (wtype) {
    case FT_W_BF16:
      if (direct) return BN == 256 ? launch_tc_gemms<256, FT_W_BF16, true>(mx, mg, mu, ma, md, a, st)
                                   : launch_tc_gemms<128, FT_W_BF16, true>(mx, mg, mu, ma, md, a, st);
      return BN == 256 ? launch_tc_gemms<256, FT_W_BF16, false>(mx, mg, mu, ma, md, a, st)
                       : launch_tc_gemms<128, FT_W_BF16, false>(mx, mg, mu, ma, md, a, st);
    case FT_W_NVFP4: return launch_tc_gemms<128, FT_W_NVFP4, false>(mx, mg, mu, ma, md, a, st);
    case FT_W_MXFP4: return launch_tc_gemms<128, FT_W_MXFP4, false>(mx, mg, mu, ma, md, a, st);
  }
  return FT_EINVAL;
}

}  // namespace

FT_API int ft_debug_quant_fp4(const void* x, int x_type, int rows, int K, int wtype, uint8_t* q, uint8_t* scales,
                              ft_cuda_stream s) {
  FT_REQUIRE(rows >= 0 && K > 0 && (wtype == FT_W_NVFP4 || wtype == FT_W_MXFP4) && K % 32 == 0);
  FT_REQUIRE(x_type == FT_X_F32 || x_type == FT_X_BF16);
  if (rows == 0) return FT_OK;
  FT_REQUIRE(x && q && scales);
  const int blk = wtype == FT_W_NVFP4 ? 16 : 32;
  const long long blocks = (long long)rows * (K / blk);
  const int grid = (int)std::max<long long>(1, std::min<long long>((blocks + 255) / 256, 8ll * sms()));
  cudaStream_t st = (cudaStream_t)s;
  const int32_t* no_perm = nullptr;
  int32_t* no_zero = nullptr;
  if (x_type == FT_X_BF16) {
    if (wtype == FT_W_NVFP4)
      FT_LAUNCH((tc::quant_rows_kernel<__nv_bfloat16, FT_W_NVFP4>), grid, 256, 0, st, (const __nv_bfloat16*)x,
                no_perm, rows, 1, K, rows, q, scales, no_zero, 0);
    else
      FT_LAUNCH((tc::quant_rows_kernel<__nv_bfloat16, FT_W_MXFP4>), grid, 256, 0, st, (const __nv_bfloat16*)x,
                no_perm, rows, 1, K, rows, q, scales, no_zero, 0);
  } else {
    if (wtype == FT_W_NVFP4)
      FT_LAUNCH((tc::quant_rows_kernel<float, FT_W_NVFP4>), grid, 256, 0, st, (const float*)x, no_perm, rows, 1, K,
                rows, q, scales, no_zero, 0);
    else
      FT_LAUNCH((tc::quant_rows_kernel<float, FT_W_MXFP4>), grid, 256, 0, st, (const float*)x, no_perm, rows, 1, K,
                rows, q, scales, no_zero, 0);
  }
  return FT_OK;
}

FT_API int ft_expert_set_fp4_path(int path) {
  FT_REQUIRE(path == FT_FP4_BLOCK_SCALED || path == FT_FP4_EXPAND_BF16);
  g_fp4_path = path;
  return FT_OK;
}

FT_API int ft_expert_grouped(const void* x, int x_type, int T, int k, int hidden, int inter, int E, int wtype,
                             const int32_t* perm, const int32_t* offsets, const int32_t* slot_of,
                             const void* slot_pool, uint64_t slot_bytes, int pool_slots, float* y, void* workspace,
                             size_t workspace_bytes, ft_cuda_stream s) {
  FT_REQUIRE(T >= 0 && k >= 1 && E >= 1 && E <= 1024 && pool_slots >= 1);
  FT_REQUIRE(x_type == FT_X_F32 || x_type == FT_X_BF16);
  ft_expert_layout L;
  if (expert_layout(wtype, hidden, inter, &L) != FT_OK) return FT_EINVAL;
  FT_REQUIRE(slot_bytes >= L.bytes && slot_bytes % 256 == 0);
  if (T == 0) return FT_OK;
  FT_REQUIRE(x && perm && offsets && slot_of && slot_pool && y && workspace);
  FT_REQUIRE(workspace_bytes >= ft_expert_grouped_workspace(T, k, hidden, inter));
  FT_REQUIRE(((uintptr_t)workspace & 255) == 0 && ((uintptr_t)slot_pool & 255) == 0);
  ExpertArgs a;
  a.x = x; a.x_type = x_type; a.T = T; a.k = k; a.H = hidden; a.I = inter; a.E = E; a.pool_slots = pool_slots;
  a.perm = perm; a.offsets = offsets; a.slot_of = slot_of; a.pool = (const uint8_t*)slot_pool; a.S = slot_bytes;
  for (int m = 0; m < 3; ++m) { a.off_val[m] = L.off_val[m]; a.off_scale[m] = L.off_scale[m]; }
  a.off_gscale = L.off_gscale;
  a.A = (float*)workspace;
  a.y = y;
  cudaStream_t st = (cudaStream_t)s;
  if (tc_path_applies(wtype, T, k, hidden, inter, E)) return launch_expert_tc(wtype, a, L, workspace, st);
  switch (wtype) {
    case FT_W_F32: return launch_expert<FT_W_F32>(a, st);
    case FT_W_BF16: return launch_expert<FT_W_BF16>(a, st);
    case FT_W_FP8E4M3: return launch_expert<FT_W_FP8E4M3>(a, st);
    case FT_W_NVFP4: return launch_expert<FT_W_NVFP4>(a, st);
    case FT_W_MXFP4: return launch_expert<FT_W_MXFP4>(a, st);
  }
  return FT_EINVAL;
}

// ------------------------------------------------------------------ cache
FT_API int ft_cache_create(const ft_cache_config* cfg, ft_cache** out) {
  FT_REQUIRE(cfg && out);
  *out = nullptr;
  FT_REQUIRE(cfg->n_layers >= 1 && cfg->n_experts >= 1 && cfg->n_experts <= CACHE_MAX_E);
  FT_REQUIRE(cfg->n_phys_layers >= 1 && cfg->n_phys_layers <= cfg->n_layers);
  FT_REQUIRE(cfg->max_slots >= 1 && cfg->max_slots <= CACHE_MAX_SLOTS);
  FT_REQUIRE(cfg->n_slots >= 1 && cfg->n_slots <= cfg->max_slots);
  FT_REQUIRE(cfg->slot_bytes > 0 && cfg->slot_bytes % 256 == 0);
  FT_REQUIRE(cfg->host_pool && cfg->slot_pool);
  FT_REQUIRE((long long)cfg->n_layers * cfg->n_experts < (1ll << 30));
  void* hd = nullptr;
  cudaError_t e = cudaHostGetDevicePointer(&hd, const_cast<void*>(cfg->host_pool), 0);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FT_EINVAL;  // not mapped pinned memory
  }
  ft_cache* c = new (std::nothrow) ft_cache();
  if (!c) return FT_ENOMEM;
  c->L = cfg->n_layers; c->E = cfg->n_experts; c->Lp = cfg->n_phys_layers; c->N = cfg->n_slots;
  c->max_slots = cfg->max_slots; c->S = cfg->slot_bytes;
  c->host = (const uint8_t*)cfg->host_pool; c->host_dev = (const uint8_t*)hd; c->pool = (uint8_t*)cfg->slot_pool;
  cudaGetDevice(&c->dev);
  const size_t nk = (size_t)c->L * c->E;
  auto dm = [](auto** p, size_t n) { return dev_malloc(reinterpret_cast<void**>(p), n) == cudaSuccess; };
  bool ok = dm(&c->slot_of_key, nk * 4) && dm(&c->key_of_slot, (size_t)c->max_slots * 4) &&
            dm(&c->stamp, (size_t)c->max_slots * 4) &&
            dm(&c->clock, 4) && dm(&c->stats, 5 * 8) && dm(&c->fill_src, (size_t)c->E * 4) &&
            dm(&c->fill_dst, (size_t)c->E * 4) && dm(&c->n_fill, 4);
  if (!ok) {
    cudaGetLastError();
    ft_cache_destroy(c);
    return FT_ENOMEM;
  }
  int st = FT_OK;
  if (cudaMemset(c->stats, 0, 5 * 8) != cudaSuccess || cudaMemset(c->n_fill, 0, 4) != cudaSuccess) st = FT_ECUDA;
  HostTables t;
  t.key.assign(c->N, -1);
  t.stamp.assign(c->N, 0);
  t.clock = 0;
  if (!st) st = upload_tables(c, t);
  if (!st) st = set_smem(cache_control_kernel, cache_control_smem(c->max_slots, c->E));
  // The fill may run beside the expert kernels (split steps), which need most of
  // the shared memory: ask for the largest shared-memory carveout so that an SM
  // running fill blocks need not drain to take an expert block.
  if (!st && cudaFuncSetAttribute(cache_fill_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess)
    st = FT_ECUDA;
  if (!st) {
    cudaError_t e2 = make_event(&c->ev_ctrl);
    if (e2 == cudaSuccess) e2 = make_event(&c->ev_fill);
    if (e2 != cudaSuccess) st = cuda_status(e2);
  }
  if (!st && cudaDeviceSynchronize() != cudaSuccess) st = FT_ECUDA;
  if (st) {
    ft_cache_destroy(c);
    return st;
  }
  // 32 blocks of 256 threads, 4 x 16 B reads in flight per thread (512 KiB).
  // A fill running alone holds the link's SM-copy rate (51 GB/s) from 8 blocks
  // up; reads beyond that queue in the memory system and hold up the HBM reads
  // of expert kernels running beside the fill (64-token expert calls took 1.6x
  // as long beside 8 fill blocks, 2.6x beside 32, 3.3x beside 148).  Inside a
  // split decode step the fill is the longer branch, and more blocks finish it
  // sooner: 64-token decode of the 40-layer bf16 stack at 6895 / 7523 / 7821
  // tokens/s with 8 / 16 / 32 blocks, 16-token decode within 1% (measured on
  // B300).
  c->fill_grid = 32;
  *out = c;
  return FT_OK;
}

FT_API int ft_cache_destroy(ft_cache* c) {
  if (!c) return FT_OK;
  dev_free(c->slot_of_key); dev_free(c->key_of_slot); dev_free(c->stamp);
  dev_free(c->clock); dev_free(c->stats); dev_free(c->fill_src); dev_free(c->fill_dst); dev_free(c->n_fill);
  drop_event(c->ev_ctrl);
  drop_event(c->ev_fill);
  delete c;
  return FT_OK;
}

FT_API int ft_cache_n_waves(const ft_cache* c) {
  if (!c) return 0;
  return ceil_div(c->E, c->N);
}

FT_API int ft_cache_step(ft_cache* c, int layer, const int32_t* counts, double fill_ratio, int wave, int32_t* slot_of,
                         int32_t* ext_flags, int32_t* step_counts, ft_cuda_stream s) {
  FT_REQUIRE(c && counts && slot_of);
  FT_REQUIRE(layer >= 0 && layer < c->L && wave >= 0 && wave < ceil_div(c->E, c->N));
  FT_REQUIRE(fill_ratio > 0.0);
  if (c->streaming || c->pending_join) return FT_ESTATE;
  cudaStream_t st = (cudaStream_t)s;
  const size_t smem = cache_control_smem(c->N, c->E);
  FT_LAUNCH(cache_control_kernel, 1, CC_THREADS, smem, st, cache_dev(c), layer, counts, fill_ratio, wave, slot_of,
            (int32_t*)nullptr, ext_flags, step_counts);
  FT_LAUNCH(cache_fill_kernel, c->fill_grid, FILL_THREADS, 0, st, (const uint8_t*)c->host_dev, c->pool, c->S,
            c->Lp * c->E, c->max_slots, (const int32_t*)c->fill_src, (const int32_t*)c->fill_dst,
            (const int32_t*)c->n_fill);
  return FT_OK;
}

FT_API int ft_cache_step_split(ft_cache* c, int layer, const int32_t* counts, double fill_ratio, int wave,
                               int32_t* slot_hit, int32_t* slot_fill, int32_t* ext_flags, int32_t* step_counts,
                               ft_cuda_stream s, ft_cuda_stream fill_s) {
  FT_REQUIRE(c && counts && slot_hit && slot_fill && slot_hit != slot_fill);
  FT_REQUIRE(layer >= 0 && layer < c->L && wave >= 0 && wave < ceil_div(c->E, c->N));
  FT_REQUIRE(fill_ratio > 0.0);
  if (c->streaming || c->pending_join) return FT_ESTATE;
  cudaStream_t st = (cudaStream_t)s, fs = (cudaStream_t)fill_s;
  const size_t smem = cache_control_smem(c->N, c->E);
  FT_LAUNCH(cache_control_kernel, 1, CC_THREADS, smem, st, cache_dev(c), layer, counts, fill_ratio, wave, slot_hit,
            slot_fill, ext_flags, step_counts);
  if (fs == st) {
    FT_LAUNCH(cache_fill_kernel, c->fill_grid, FILL_THREADS, 0, st, (const uint8_t*)c->host_dev, c->pool, c->S,
              c->Lp * c->E, c->max_slots, (const int32_t*)c->fill_src, (const int32_t*)c->fill_dst,
              (const int32_t*)c->n_fill);
    return FT_OK;
  }
  // fork: the fill stream starts after the control launch; a plain launch there
  // (its only predecessor that matters is the control kernel on the other stream)
  FT_CHECK_CUDA(cudaEventRecord(c->ev_ctrl, st));
  FT_CHECK_CUDA(cudaStreamWaitEvent(fs, c->ev_ctrl, 0));
  cache_fill_kernel<<<c->fill_grid, FILL_THREADS, 0, fs>>>((const uint8_t*)c->host_dev, c->pool, c->S,
                                                            c->Lp * c->E, c->max_slots, (const int32_t*)c->fill_src,
                                                            (const int32_t*)c->fill_dst, (const int32_t*)c->n_fill);
  FT_CHECK_CUDA(cudaGetLastError());
  FT_CHECK_CUDA(cudaEventRecord(c->ev_fill, fs));
  c->pending_join = 1;
  return FT_OK;
}

FT_API int ft_cache_set_fill_blocks(ft_cache* c, int blocks) {
  FT_REQUIRE(c && blocks >= 1 && blocks <= 4 * sms());
  c->fill_grid = blocks;
  return FT_OK;
}

FT_API int ft_cache_fill_join(ft_cache* c, ft_cuda_stream s) {
  FT_REQUIRE(c);
  if (!c->pending_join) return FT_OK;
  FT_CHECK_CUDA(cudaStreamWaitEvent((cudaStream_t)s, c->ev_fill, 0));
  c->pending_join = 0;
  return FT_OK;
}

FT_API int ft_cache_resize(ft_cache* c, int n_slots) {
  FT_REQUIRE(c && n_slots >= 1 && n_slots <= c->max_slots);
  if (c->streaming || c->pending_join) return FT_ESTATE;
  return cache_resize_impl(c, n_slots);
}

FT_API int ft_cache_reset(ft_cache* c) {
  FT_REQUIRE(c);
  if (c->streaming || c->pending_join) return FT_ESTATE;
  FT_CHECK_CUDA(cudaDeviceSynchronize());
  HostTables t;
  t.key.assign(c->N, -1);
  t.stamp.assign(c->N, 0);
  t.clock = 0;
  if (int s = upload_tables(c, t)) return s;
  FT_CHECK_CUDA(cudaMemset(c->stats, 0, 5 * 8));
  FT_CHECK_CUDA(cudaMemset(c->n_fill, 0, 4));
  FT_CHECK_CUDA(cudaDeviceSynchronize());
  return FT_OK;
}

FT_API int ft_cache_stats(ft_cache* c, ft_cache_stats_t* out) {
  FT_REQUIRE(c && out);
  unsigned long long v[5];
  FT_CHECK_CUDA(cudaDeviceSynchronize());
  FT_CHECK_CUDA(cudaMemcpy(v, c->stats, sizeof(v), cudaMemcpyDeviceToHost));
  out->steps = v[0]; out->hits = v[1]; out->fills = v[2]; out->externals = v[3]; out->bytes_h2d = v[4];
  return FT_OK;
}

FT_API int ft_cache_export(ft_cache* c, int32_t* key_of_slot, uint32_t* stamp, int* n_slots, uint32_t* clock) {
  FT_REQUIRE(c && key_of_slot && stamp && n_slots && clock);
  HostTables t;
  if (int s = download_tables(c, t)) return s;
  for (int i = 0; i < c->N; ++i) { key_of_slot[i] = t.key[i]; stamp[i] = t.stamp[i]; }
  *n_slots = c->N;
  *clock = t.clock;
  return FT_OK;
}

// ------------------------------------------------------------------ host-side expert executor
FT_API int ft_cpu_create(int threads, ft_cpu** out) {
  FT_REQUIRE(out && threads >= 0 && threads <= 255);
  *out = nullptr;
  if (threads == 0) threads = (int)std::min<unsigned>(255u, std::max(1u, std::thread::hardware_concurrency()) - 1);
  ft_cpu* c = new (std::nothrow) ft_cpu();
  if (!c) return FT_ENOMEM;
  c->n_threads = threads + 1;
  try {
    for (int i = 0; i < threads; ++i) c->workers.emplace_back(cpu_worker, c);
  } catch (...) {
    ft_cpu_destroy(c);
    return FT_ENOMEM;
  }
  *out = c;
  return FT_OK;
}

FT_API int ft_cpu_destroy(ft_cpu* c) {
  if (!c) return FT_OK;
  {
    std::lock_guard<std::mutex> lk(c->mu);
    c->stop.store(true, std::memory_order_release);
  }
  c->cv.notify_all();
  for (auto& t : c->workers) t.join();
  delete c;
  return FT_OK;
}

FT_API int ft_cpu_experts(ft_cpu* c, const ft_cpu_job* job) {
  FT_REQUIRE(c && job);
  return cpu_experts_run(c, *job);
}

static void CUDART_CB cpu_host_fn(void* p) {
  ft_cpu_job_rec* r = static_cast<ft_cpu_job_rec*>(p);
  const int st = cpu_experts_run(r->cpu, r->job);
  if (st) {
    int zero = 0;
    r->cpu->status.compare_exchange_strong(zero, st);  // the first failure is kept
  }
}

FT_API int ft_cpu_experts_enqueue(ft_cpu* c, const ft_cpu_job* job, ft_cuda_stream s) {
  FT_REQUIRE(c && job);
  ft_expert_layout L;
  if (expert_layout(job->wtype, job->hidden, job->inter, &L) != FT_OK) return FT_EINVAL;
  FT_REQUIRE(job->host_pool && job->x && job->topk_idx && job->topk_w && job->ext_flags && job->partial);
  FT_REQUIRE(job->T >= 0 && job->k >= 1 && job->n_experts >= 1 && job->slot_bytes >= L.bytes);
  std::unique_ptr<ft_cpu_job_rec> r(new (std::nothrow) ft_cpu_job_rec{c, *job});
  if (!r) return FT_ENOMEM;
  FT_CHECK_CUDA(cudaLaunchHostFunc((cudaStream_t)s, cpu_host_fn, r.get()));
  std::lock_guard<std::mutex> lk(c->run_mu);
  c->jobs.push_back(std::move(r));
  return FT_OK;
}

FT_API int ft_cpu_status(ft_cpu* c) {
  FT_REQUIRE(c);
  return c->status.exchange(0);
}

// ------------------------------------------------------------------ placement replay
FT_API int ft_placement_replay(int policy, int n_layers, int n_experts, int capacity, const int32_t* prefill_counts,
                               const int32_t* trace, int n_steps, int width, uint64_t* accesses, uint64_t* misses) {
  FT_REQUIRE(accesses && misses && n_layers >= 1 && n_experts >= 1 && n_steps >= 0 && width >= 1);
  const long long keys = (long long)n_layers * n_experts;
  FT_REQUIRE(keys < (1ll << 30) && capacity >= 1 && capacity <= keys);
  FT_REQUIRE(trace || n_steps == 0);
  uint64_t acc = 0, miss = 0;
  if (policy == FT_PLACE_GLOBAL_LRU) {
    FT_REQUIRE(capacity >= n_experts);
    replay_lru(n_layers, n_experts, capacity, trace, n_steps, width, acc, miss);
  } else if (policy == FT_PLACE_PREFILL_HOT || policy == FT_PLACE_STATIC_SPLIT) {
    std::vector<char> resident((size_t)keys, 0);
    if (policy == FT_PLACE_STATIC_SPLIT) {
      for (int k = 0; k < capacity; ++k) resident[k] = 1;
    } else {
      FT_REQUIRE(prefill_counts);
      std::vector<int> order;
      for (int k = 0; k < keys; ++k)
        if (prefill_counts[k] > 0) order.push_back(k);
      std::stable_sort(order.begin(), order.end(),
                       [&](int a, int b) { return prefill_counts[a] > prefill_counts[b]; });
      for (size_t i = 0; i < order.size() && (int)i < capacity; ++i) resident[order[i]] = 1;
    }
    replay_fixed(n_layers, n_experts, resident, trace, n_steps, width, acc, miss);
  } else {
    return FT_EINVAL;
  }
  *accesses = acc;
  *misses = miss;
  return FT_OK;
}

// ------------------------------------------------------------------ stream
// Destroys a stream handle's CUDA stream and events (those that exist) and the handle.
static void stream_release(ft_stream* st) {
  drop_stream(st->copy);
  for (int b = 0; b < 2; ++b) {
    drop_event(st->ready[b]);
    drop_event(st->freed[b]);
  }
  delete st;
}

FT_API int ft_stream_create(ft_cache* c, int serialized, ft_stream** out) {
  FT_REQUIRE(c && out);
  *out = nullptr;
  if (c->streaming || c->pending_join) return FT_ESTATE;
  if (c->N < 2 * c->E) return FT_EUNSUPPORTED;
  ft_stream* st = new (std::nothrow) ft_stream();
  if (!st) return FT_ENOMEM;
  // the stream and events first: a failure here leaves the cache untouched
  cudaError_t e = make_stream(&st->copy);
  for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
    e = make_event(&st->ready[b]);
    if (e == cudaSuccess) e = make_event(&st->freed[b]);
  }
  if (e != cudaSuccess) {
    stream_release(st);
    return cuda_status(e);
  }
  const int n_full = c->N;
  if (int s = cache_resize_impl(c, n_full - 2 * c->E)) {
    stream_release(st);
    return s;
  }
  c->n_full = n_full;
  c->streaming = 1;
  st->c = c;
  st->serialized = serialized ? 1 : 0;
  st->base = n_full - 2 * c->E;
  st->buf_layer[0] = st->buf_layer[1] = -1;
  st->freed_rec[0] = st->freed_rec[1] = false;
  st->next_buf = 0;
  st->pending_layer = -1;
  st->bytes = 0;
  st->n_hist = 0;
  *out = st;
  return FT_OK;
}

FT_API int ft_stream_layer(ft_stream* st, int layer, int next_layer, int32_t* slot_of, ft_cuda_stream compute) {
  FT_REQUIRE(st && slot_of);
  ft_cache* c = st->c;
  FT_REQUIRE(layer >= 0 && layer < c->L && next_layer >= -1 && next_layer < c->L);
  cudaStream_t cs = (cudaStream_t)compute;
  int b = buffer_of(st, layer);
  if (b < 0) {
    b = st->next_buf;
    if (int s = stream_issue_copy(st, layer, b, nullptr)) return s;
    st->next_buf = b ^ 1;
  }
  FT_CHECK_CUDA(cudaStreamWaitEvent(cs, st->ready[b], 0));
  FT_LAUNCH(set_buffer_slots_kernel, ceil_div(c->E, 256), 256, 0, cs, slot_of, c->E, st->base + b * c->E);
  st->pending_layer = -1;
  if (next_layer >= 0 && buffer_of(st, next_layer) < 0) {
    const int nb = b ^ 1;
    if (!st->serialized) {
      if (int s = stream_issue_copy(st, next_layer, nb, nullptr)) return s;
      st->next_buf = b;
    } else {
      st->pending_layer = next_layer;
      st->pending_buf = nb;
    }
  }
  return FT_OK;
}

FT_API int ft_stream_layer_done(ft_stream* st, int layer, ft_cuda_stream compute) {
  FT_REQUIRE(st);
  const int b = buffer_of(st, layer);
  FT_REQUIRE(b >= 0);
  cudaStream_t cs = (cudaStream_t)compute;
  FT_CHECK_CUDA(cudaEventRecord(st->freed[b], cs));
  st->freed_rec[b] = true;
  if (st->serialized && st->pending_layer >= 0) {
    const int nb = st->pending_buf;
    if (int s = stream_issue_copy(st, st->pending_layer, nb, st->freed[b])) return s;
    st->next_buf = b;
    st->pending_layer = -1;
  }
  return FT_OK;
}

FT_API int ft_stream_bytes(const ft_stream* st, uint64_t* bytes) {
  FT_REQUIRE(st && bytes);
  *bytes = st->bytes;
  return FT_OK;
}

FT_API int ft_stream_destroy(ft_stream* st) {
  if (!st) return FT_OK;
  ft_cache* c = st->c;
  cudaStreamSynchronize(st->copy);
  int s = stream_adopt(st);
  c->streaming = 0;
  stream_release(st);
  return s;
}

// ------------------------------------------------------------------ expert grouped without allocation
// A variant of ft_expert_grouped for callers that cannot allocate device
// memory.  The fp32 intermediate silu(G)*U lives in the fixed array below
// instead of a caller-supplied workspace.  Host code must not hand the array's
// name to a kernel (in host code it is a host-side stand-in); its device
// address is looked up once per device with cudaGetSymbolAddress.

static constexpr size_t kNoAllocMaxElems = (size_t)1 << 20;  // fp32 elements: 4 MiB per device
static __device__ __align__(256) float ft_noalloc_scratch[kNoAllocMaxElems];

static constexpr int kNoAllocMaxDevices = 64;
struct NoAllocAddr {
  unsigned long long ctx_id = 0;  // context the address belongs to (0: not looked up yet)
  void* addr = nullptr;
};
static NoAllocAddr g_noalloc_addr[kNoAllocMaxDevices];
static std::mutex g_noalloc_mu;

// Id of the current CUDA context (0 when it cannot be read).  The array's
// address belongs to one context: after cudaDeviceReset the next context has a
// new id and the address is looked up again.
static unsigned long long current_context_id() {
  using GetCurrentFn = CUresult (*)(CUcontext*);
  using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(p);
    cudaGetLastError();
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx && get_id(ctx, &id) == CUDA_SUCCESS) return id;
  return 0;
}

// Device address of the scratch array in the current device's context: looked
// up with cudaGetSymbolAddress on the first call in each context, then reused
// (looked up on every call if the context id cannot be read).
static int noalloc_scratch_address(void** out) {
  int d = 0;
  FT_CHECK_CUDA(cudaGetDevice(&d));
  if (d < 0 || d >= kNoAllocMaxDevices) return FT_EUNSUPPORTED;
  unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocAddr& a = g_noalloc_addr[d];
  if (ctx == 0 || a.ctx_id != ctx || !a.addr) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress((void**)&p, ft_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return cuda_status(e == cudaSuccess ? cudaErrorInvalidSymbol : e);
    }
    a.addr = p;
    a.ctx_id = ctx ? ctx : current_context_id();  // the lookup created the context if there was none
  }
  *out = a.addr;
  return FT_OK;
}

FT_API int ft_expert_grouped_noalloc(const void* x, int x_type, int T, int k, int hidden, int inter, int E, int wtype,
                                     const int32_t* perm, const int32_t* offsets, const int32_t* slot_of,
                                     const void* slot_pool, uint64_t slot_bytes, int pool_slots, float* y,
                                     ft_cuda_stream s) {
  FT_REQUIRE(T >= 0 && k >= 1 && E >= 1 && E <= 1024 && pool_slots >= 1);
  FT_REQUIRE(x_type == FT_X_F32 || x_type == FT_X_BF16);
  ft_expert_layout L;
  if (expert_layout(wtype, hidden, inter, &L) != FT_OK) return FT_EINVAL;
  FT_REQUIRE(slot_bytes >= L.bytes && slot_bytes % 256 == 0);
  // the intermediate needs T*k*inter fp32 elements; larger calls are refused
  if ((size_t)T * (size_t)k * (size_t)inter > kNoAllocMaxElems) return FT_EINVAL;
  if (T == 0) return FT_OK;
  FT_REQUIRE(x && perm && offsets && slot_of && slot_pool && y);
  FT_REQUIRE(((uintptr_t)slot_pool & 255) == 0);
  void* scratch = nullptr;
  if (int st = noalloc_scratch_address(&scratch)) return st;
  ExpertArgs a;
  a.x = x; a.x_type = x_type; a.T = T; a.k = k; a.H = hidden; a.I = inter; a.E = E; a.pool_slots = pool_slots;
  a.perm = perm; a.offsets = offsets; a.slot_of = slot_of; a.pool = (const uint8_t*)slot_pool; a.S = slot_bytes;
  for (int m = 0; m < 3; ++m) { a.off_val[m] = L.off_val[m]; a.off_scale[m] = L.off_scale[m]; }
  a.off_gscale = L.off_gscale;
  a.A = (float*)scratch;  // every element the down pass reads is written by the gate/up pass of this call
  a.y = y;
  cudaStream_t st = (cudaStream_t)s;
  switch (wtype) {
    case FT_W_F32: return launch_expert<FT_W_F32>(a, st);
    case FT_W_BF16: return launch_expert<FT_W_BF16>(a, st);
    case FT_W_FP8E4M3: return launch_expert<FT_W_FP8E4M3>(a, st);
    case FT_W_NVFP4: return launch_expert<FT_W_NVFP4>(a, st);
    case FT_W_MXFP4: return launch_expert<FT_W_MXFP4>(a, st);
  }
  return FT_EINVAL;
}
