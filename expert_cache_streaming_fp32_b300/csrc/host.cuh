// Host-side resources of libft: counted device allocations, streams and
// events of the handles, host-side failure injection for tests, and the
// read-then-pin pieces of pool setup (parallel file reads into the host pool,
// registration of an already-filled buffer).  Part of the single translation
// unit ft.cu.
#pragma once

#include <algorithm>
#include <atomic>
#include <fcntl.h>
#include <thread>
#include <unistd.h>
#include <vector>

#include "common.cuh"

namespace ft {

// ------------------------------------------------------------------ failure injection
// Each site counts down: armed with `after` = n, the next n calls at the site
// succeed and the one after fails as if the CUDA runtime had refused it; then
// the site disarms itself.  Nothing here touches the GPU: a failed call is
// simply never issued.
enum { INJ_DEVICE_ALLOC = 1, INJ_HOST_PIN = 2, INJ_STREAM_EVENT = 3, INJ_SITES = 4 };

static std::atomic<int> g_inject_after[INJ_SITES] = {{-1}, {-1}, {-1}, {-1}};

static inline bool inject_fail(int site) {
  int v = g_inject_after[site].load();
  while (v >= 0) {
    if (g_inject_after[site].compare_exchange_weak(v, v - 1)) return v == 0;
  }
  return false;
}

// ------------------------------------------------------------------ counted resources
static std::atomic<long long> g_live_dev_allocs{0};
static std::atomic<long long> g_live_streams_events{0};

static inline cudaError_t dev_malloc(void** p, size_t n) {
  *p = nullptr;
  if (inject_fail(INJ_DEVICE_ALLOC)) return cudaErrorMemoryAllocation;
  cudaError_t e = cudaMalloc(p, n);
  if (e == cudaSuccess) ++g_live_dev_allocs;
  return e;
}

template <typename T>
static inline void dev_free(T*& p) {
  if (p) {
    cudaFree(p);
    --g_live_dev_allocs;
    p = nullptr;
  }
}

static inline cudaError_t make_event(cudaEvent_t* ev) {
  *ev = nullptr;
  if (inject_fail(INJ_STREAM_EVENT)) return cudaErrorMemoryAllocation;
  cudaError_t e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  if (e == cudaSuccess) ++g_live_streams_events;
  else *ev = nullptr;
  return e;
}

static inline void drop_event(cudaEvent_t& ev) {
  if (ev) {
    cudaEventDestroy(ev);
    --g_live_streams_events;
    ev = nullptr;
  }
}

static inline cudaError_t make_stream(cudaStream_t* s) {
  *s = nullptr;
  if (inject_fail(INJ_STREAM_EVENT)) return cudaErrorMemoryAllocation;
  cudaError_t e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking);
  if (e == cudaSuccess) ++g_live_streams_events;
  else *s = nullptr;
  return e;
}

static inline void drop_stream(cudaStream_t& s) {
  if (s) {
    cudaStreamDestroy(s);
    --g_live_streams_events;
    s = nullptr;
  }
}

// ------------------------------------------------------------------ pool file reads
// Reads `bytes` from `path` at `offset` into dst with `threads` threads, each
// taking one contiguous share in pieces of at most 64 MiB.  The destination is
// ordinary (pageable) memory: the read is what first touches its pages, so
// pinning afterwards only locks pages that already hold the experts.
static int pool_read(const char* path, uint64_t offset, void* dst, uint64_t bytes, int threads) {
  const int fd = open(path, O_RDONLY | O_CLOEXEC);
  if (fd < 0) return FT_EIO;
  constexpr uint64_t kPiece = 64ull << 20;
  const uint64_t share = (bytes + threads - 1) / threads;
  std::atomic<int> failed{0};
  auto work = [&](int i) {
    const uint64_t b0 = (uint64_t)i * share, b1 = std::min<uint64_t>(bytes, b0 + share);
    for (uint64_t b = b0; b < b1 && !failed.load();) {
      const uint64_t n = std::min<uint64_t>(kPiece, b1 - b);
      const ssize_t r = pread(fd, static_cast<uint8_t*>(dst) + b, n, (off_t)(offset + b));
      if (r <= 0) {
        failed = 1;
        return;
      }
      b += (uint64_t)r;
    }
  };
  std::vector<std::thread> pool;
  for (int i = 1; i < threads; ++i) pool.emplace_back(work, i);
  work(0);
  for (auto& t : pool) t.join();
  close(fd);
  return failed.load() ? FT_EIO : FT_OK;
}

}  // namespace ft
