// Shared helpers of libft: status plumbing, the device error word, bf16/fp8/fp4
// decoding, warp reductions.  Part of the single translation unit ft.cu.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_fp4.h>
#include <stdint.h>
#include <stddef.h>

#include <utility>

#include "../../include/ft.h"

#define FT_FULL_MASK 0xffffffffu

namespace ft {

// ------------------------------------------------------------------ host status
static thread_local int g_last_cuda_error = 0;

static inline int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return FT_OK;
  g_last_cuda_error = (int)e;
  return FT_ECUDA;
}

#define FT_CHECK_CUDA(call)                                 \
  do {                                                      \
    cudaError_t _e = (call);                                \
    if (_e != cudaSuccess) return ::ft::cuda_status(_e);    \
  } while (0)

#define FT_CHECK_LAUNCH() FT_CHECK_CUDA(cudaGetLastError())

#define FT_REQUIRE(cond)          \
  do {                            \
    if (!(cond)) return FT_EINVAL; \
  } while (0)

// ------------------------------------------------------------------ device error word
// First error wins; kernels skip the offending access after recording it.
__device__ int g_derr = 0;

__device__ __forceinline__ void record_error(int code) { atomicCAS(&g_derr, 0, code); }

// ------------------------------------------------------------------ dependent launches
// Every kernel of the library is launched with programmatic stream
// serialization.  It runs its set-up that touches no global memory (barrier
// init, TMEM allocation, tensor-map prefetch), then waits (griddepcontrol.wait)
// until the kernel before it on the stream has completed and its memory is
// visible.  It lets the next kernel launch (griddepcontrol.launch_dependents)
// only when its own work is done: a dependent launched earlier would hold SM
// slots and shared memory while it waits, which the rest of a multi-wave grid
// (or the other kernels of a split step) needs.
__device__ __forceinline__ void pdl_begin() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void pdl_end() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
static inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

#define FT_LAUNCH(kernel, grid, block, smem, stream, ...) \
  FT_CHECK_CUDA(::ft::launch_pdl(kernel, dim3(grid), dim3(block), (size_t)(smem), (cudaStream_t)(stream), __VA_ARGS__))

// ------------------------------------------------------------------ numeric helpers
__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ float silu(float g) { return g / (1.0f + __expf(-g)); }

// Two e4m3 bytes (low byte = first element) -> two floats.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t v) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)v, __NV_E4M3);
  __half2 hh = *reinterpret_cast<__half2*>(&h);
  return __half22float2(hh);
}

__device__ __forceinline__ float e4m3_to_float(uint8_t v) {
  __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)v, __NV_E4M3);
  return __half2float(*reinterpret_cast<__half*>(&h));
}

// One byte of two e2m1 codes (element 2i in the low nibble) -> two floats.
__device__ __forceinline__ float2 e2m1x2_to_float2(uint8_t v) {
  __half2_raw h = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)v, __NV_E2M1);
  __half2 hh = *reinterpret_cast<__half2*>(&h);
  return __half22float2(hh);
}

// E8M0 scale byte -> 2^(b-127) (b = 255, NaN, is not produced by the writers).
__device__ __forceinline__ float e8m0_to_float(uint8_t b) {
  return b == 0 ? __uint_as_float(0x00400000u) : __uint_as_float((uint32_t)b << 23);
}

// ------------------------------------------------------------------ warp reductions
// Reduce V values (V a power of two <= 32) across the warp so that afterwards
// lane l holds in v[0] the warp total of value index l / (32 / V).
// Halving exchanges move half the values per step (V - 1 shuffles in total),
// then plain butterflies finish the remaining lane bits.
template <int V>
__device__ __forceinline__ void warp_reduce_scatter(float (&v)[V], int lane) {
  static_assert(V >= 1 && V <= 32 && (V & (V - 1)) == 0, "V power of two <= 32");
#pragma unroll
  for (int n = V, off = 16; n > 1; n >>= 1, off >>= 1) {
    const bool upper = lane & off;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      float send = upper ? v[i] : v[i + n / 2];
      float keep = upper ? v[i + n / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(FT_FULL_MASK, send, off);
    }
  }
#pragma unroll
  for (int off = 16 / V; off >= 1; off >>= 1) v[0] += __shfl_xor_sync(FT_FULL_MASK, v[0], off);
}

__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Round-half-up miss split; the same rule as the host-side ft_qsplit.
__host__ __device__ __forceinline__ int qsplit_ratio(int m, double ratio) {
  if (m <= 0) return 0;
  if (ratio >= 1.0) return m;
  double q = floor((double)m * ratio + 0.5);
  int qi = (int)q;
  if (qi < 1) qi = 1;
  if (qi > m) qi = m;
  return qi;
}

// ------------------------------------------------------------------ device properties
struct DevInfo {
  int sms = 0;
  int dev = -1;
};

static inline DevInfo& dev_info() {
  static thread_local DevInfo info;
  int d = 0;
  cudaGetDevice(&d);
  if (info.dev != d) {
    cudaDeviceGetAttribute(&info.sms, cudaDevAttrMultiProcessorCount, d);
    info.dev = d;
  }
  return info;
}

}  // namespace ft
