// Host-side expert executor: the experts left to the external path are
// evaluated from the pinned host pool by a pool of CPU threads, and their
// gate-weighted outputs summed into a per-token partial output that the GPU's
// combine adds.  Host code only; part of the single translation unit ft.cu.
#pragma once

#include <algorithm>
#include <atomic>
#include <chrono>
#include <condition_variable>
#include <cmath>
#include <cstring>
#include <functional>
#include <memory>
#include <mutex>
#include <thread>
#include <vector>

#include "common.cuh"
#include "expert.cuh"
#include "host_simd.h"

struct ft_cpu_job_rec;

struct ft_cpu {
  int n_threads = 1;
  std::vector<std::thread> workers;
  std::mutex mu;
  std::condition_variable cv, done_cv;
  const std::function<void(int)>* task = nullptr;  // the caller's, alive until busy reaches 0
  int n_tasks = 0;
  std::atomic<int> next{0};
  std::atomic<int> busy{0};                         // workers still in the current generation
  std::atomic<uint64_t> gen{0};
  std::atomic<bool> stop{false};
  std::mutex run_mu;                              // one evaluation at a time per handle
  std::atomic<int> status{0};                     // first failed status of an enqueued job
  std::vector<std::unique_ptr<ft_cpu_job_rec>> jobs;  // enqueued jobs, alive until destroy
  // scratch of one evaluation
  std::vector<float> X, Xs, A, Y;                 // Xs: X in pair-split order (vector forms, FP4)
  std::vector<int> arow_t, arow_j, rows_of;       // per external assignment: token, slot j; per (t, j): row or -1
  std::vector<int> e_begin, e_list;               // external experts and their assignment ranges
};

struct ft_cpu_job_rec {
  ft_cpu* cpu;
  ft_cpu_job job;
};

namespace ft {

// ------------------------------------------------------------------ decoding tables
// e2m1: sign, 2 exponent bits (bias 1), 1 mantissa bit; exponent 0 is 0 or 0.5.
static float e2m1_host(int c) {
  const float s = (c & 8) ? -1.0f : 1.0f;
  const int e = (c >> 1) & 3, m = c & 1;
  return e == 0 ? s * 0.5f * m : s * std::ldexp(1.0f + 0.5f * m, e - 1);
}

// e4m3 "fn": sign, 4 exponent bits (bias 7), 3 mantissa bits; S.1111.111 is NaN.
static float e4m3_host(int b) {
  const float s = (b & 0x80) ? -1.0f : 1.0f;
  const int e = (b >> 3) & 15, m = b & 7;
  if (e == 15 && m == 7) return NAN;
  return e == 0 ? s * std::ldexp(m / 8.0f, -6) : s * std::ldexp(1.0f + m / 8.0f, e - 7);
}

struct HostTables4 {
  float e2m1[16], e4m3[256], e8m0[256];
  HostTables4() {
    for (int c = 0; c < 16; ++c) e2m1[c] = e2m1_host(c);
    for (int b = 0; b < 256; ++b) {
      e4m3[b] = e4m3_host(b);
      e8m0[b] = b == 255 ? NAN : std::ldexp(1.0f, b - 127);
    }
  }
};

static const HostTables4& host_tables() {
  static HostTables4 t;
  return t;
}

// One weight row of K elements (K-major, with its scales) to fp32.
static void decode_row(int wt, const uint8_t* vals, const uint8_t* scales, float gscale, int K, float* out) {
  const HostTables4& tb = host_tables();
  switch (wt) {
    case FT_W_F32:
      std::memcpy(out, vals, (size_t)K * 4);
      return;
    case FT_W_BF16: {
      const uint16_t* v = reinterpret_cast<const uint16_t*>(vals);
      for (int i = 0; i < K; ++i) {
        const uint32_t u = (uint32_t)v[i] << 16;
        std::memcpy(out + i, &u, 4);
      }
      return;
    }
    case FT_W_FP8E4M3: {
      const float* sc = reinterpret_cast<const float*>(scales);
      for (int i = 0; i < K; ++i) out[i] = tb.e4m3[vals[i]] * sc[i >> 7];
      return;
    }
    case FT_W_NVFP4:
      for (int i = 0; i < K; i += 2) {
        const float s = tb.e4m3[scales[i >> 4]] * gscale;
        out[i] = tb.e2m1[vals[i >> 1] & 15] * s;
        out[i + 1] = tb.e2m1[vals[i >> 1] >> 4] * s;
      }
      return;
    case FT_W_MXFP4:
      for (int i = 0; i < K; i += 2) {
        const float s = tb.e8m0[scales[i >> 5]];
        out[i] = tb.e2m1[vals[i >> 1] & 15] * s;
        out[i + 1] = tb.e2m1[vals[i >> 1] >> 4] * s;
      }
      return;
  }
}

static inline float dot_f32(const float* a, const float* b, int n) {
  // eight independent partial sums (vectorisable), added in a fixed order
  float p[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  int i = 0;
  for (; i + 8 <= n; i += 8)
    for (int u = 0; u < 8; ++u) p[u] += a[i + u] * b[i + u];
  for (; i < n; ++i) p[i & 7] += a[i] * b[i];
  return ((p[0] + p[1]) + (p[2] + p[3])) + ((p[4] + p[5]) + (p[6] + p[7]));
}

// ------------------------------------------------------------------ thread pool
// Every worker takes part in every generation.  Between generations a worker
// spins on the generation counter for a while before it sleeps on the
// condition variable, so the back-to-back loops of one job find the workers
// awake: a sleeping worker costs a wake-up and a mutex hand-off per
// generation.  After a short pause-loop the spin yields its core at every
// turn, so that more threads than cores, or other threads of the process,
// still get to run.
constexpr int64_t CPU_SPIN_NS = 100000;
constexpr int CPU_PAUSE_TURNS = 512;

// Spins until pred() holds or CPU_SPIN_NS pass; returns pred().
template <typename P>
static bool cpu_spin(const P& pred) {
  const auto t0 = std::chrono::steady_clock::now();
  for (int i = 1;; ++i) {
    if (pred()) return true;
    if (i < CPU_PAUSE_TURNS) {
#if defined(__x86_64__)
      __builtin_ia32_pause();
#endif
      continue;
    }
    std::this_thread::yield();
    if (std::chrono::steady_clock::now() - t0 > std::chrono::nanoseconds(CPU_SPIN_NS)) return pred();
  }
}

static void cpu_worker(ft_cpu* c) {
  uint64_t seen = 0;
  for (;;) {
    auto woken = [&] { return c->stop.load(std::memory_order_acquire) || c->gen.load(std::memory_order_acquire) != seen; };
    if (!cpu_spin(woken)) {
      std::unique_lock<std::mutex> lk(c->mu);
      c->cv.wait(lk, woken);
    }
    if (c->stop.load(std::memory_order_acquire)) return;
    seen = c->gen.load(std::memory_order_acquire);
    const std::function<void(int)>& fn = *c->task;
    for (int i; (i = c->next.fetch_add(1)) < c->n_tasks;) fn(i);
    if (c->busy.fetch_sub(1, std::memory_order_acq_rel) == 1) {
      std::lock_guard<std::mutex> lk(c->mu);
      c->done_cv.notify_all();
    }
  }
}

// Runs fn(0 .. n-1) on the pool and the calling thread; returns when all are done.
static void cpu_parallel_for(ft_cpu* c, int n, const std::function<void(int)>& fn) {
  if (n <= 0) return;
  if (c->workers.empty() || n == 1) {
    for (int i = 0; i < n; ++i) fn(i);
    return;
  }
  c->task = &fn;
  c->n_tasks = n;
  c->next.store(0, std::memory_order_relaxed);
  c->busy.store((int)c->workers.size(), std::memory_order_relaxed);
  {
    std::lock_guard<std::mutex> lk(c->mu);          // a worker between its check and its wait holds mu
    c->gen.fetch_add(1, std::memory_order_release);
  }
  c->cv.notify_all();
  for (int i; (i = c->next.fetch_add(1)) < n;) fn(i);
  auto done = [&] { return c->busy.load(std::memory_order_acquire) == 0; };
  if (!cpu_spin(done)) {
    std::unique_lock<std::mutex> lk(c->mu);
    c->done_cv.wait(lk, done);
  }
}

// ------------------------------------------------------------------ evaluation
static int cpu_experts_run(ft_cpu* c, const ft_cpu_job& j) {
  ft_expert_layout L;
  if (expert_layout(j.wtype, j.hidden, j.inter, &L) != FT_OK) return FT_EINVAL;
  if (j.T < 0 || j.k < 1 || j.n_experts < 1 || j.phys_layer < 0 || j.slot_bytes < L.bytes) return FT_EINVAL;
  if (j.T == 0) return FT_OK;  // nothing is read or written
  if (!j.host_pool || !j.x || !j.topk_idx || !j.topk_w || !j.ext_flags || !j.partial) return FT_EINVAL;
  std::lock_guard<std::mutex> run_lock(c->run_mu);
  const int T = j.T, k = j.k, H = j.hidden, I = j.inter, E = j.n_experts;
  // external assignments, grouped by expert (ascending), tokens ascending inside
  c->e_begin.assign(E + 1, 0);
  c->rows_of.assign((size_t)T * k, -1);
  for (int a = 0; a < T * k; ++a) {
    const int e = j.topk_idx[a];
    if (e >= 0 && e < E && j.ext_flags[e]) ++c->e_begin[e + 1];
  }
  for (int e = 0; e < E; ++e) c->e_begin[e + 1] += c->e_begin[e];
  const int n_ext = c->e_begin[E];
  c->arow_t.assign(n_ext, 0);
  c->arow_j.assign(n_ext, 0);
  {
    std::vector<int> fill(c->e_begin.begin(), c->e_begin.end() - 1);
    for (int a = 0; a < T * k; ++a) {
      const int e = j.topk_idx[a];
      if (e >= 0 && e < E && j.ext_flags[e]) {
        const int r = fill[e]++;
        c->arow_t[r] = a / k;
        c->arow_j[r] = a % k;
        c->rows_of[a] = r;
      }
    }
  }
  c->e_list.clear();
  for (int e = 0; e < E; ++e)
    if (c->e_begin[e + 1] > c->e_begin[e]) c->e_list.push_back(e);
  // tokens to fp32
  c->X.resize((size_t)T * H);
  if (j.x_type == FT_X_BF16) {
    const uint16_t* xb = static_cast<const uint16_t*>(j.x);
    for (size_t i = 0; i < (size_t)T * H; ++i) {
      const uint32_t u = (uint32_t)xb[i] << 16;
      std::memcpy(&c->X[i], &u, 4);
    }
  } else if (j.x_type == FT_X_F32) {
    std::memcpy(c->X.data(), j.x, (size_t)T * H * 4);
  } else {
    return FT_EINVAL;
  }
  c->A.resize((size_t)n_ext * I);
  c->Y.resize((size_t)n_ext * H);
  const uint8_t* pool = static_cast<const uint8_t*>(j.host_pool);
  const int wt = j.wtype;
  const uint64_t vrow[3] = {(uint64_t)H * fmt_bits(wt) / 8, (uint64_t)H * fmt_bits(wt) / 8,
                            (uint64_t)I * fmt_bits(wt) / 8};
  const uint64_t srow[3] = {fmt_scale_row_bytes(wt, H), fmt_scale_row_bytes(wt, H), fmt_scale_row_bytes(wt, I)};
  auto rec = [&](int e) { return pool + ((uint64_t)j.phys_layer * E + e) * j.slot_bytes; };
  auto gscale = [&](int e, int m) {
    if (wt != FT_W_NVFP4) return 1.0f;
    float g;
    std::memcpy(&g, rec(e) + L.off_gscale + 4 * m, 4);
    return g;
  };
  constexpr int RB = 32;  // weight rows per task
  const int nE = (int)c->e_list.size();
  const int bi = (I + RB - 1) / RB, bh = (H + RB - 1) / RB;
  if (host_simd_supported()) {
    // rows decoded in registers and dotted with every token of the expert at once
    // (AVX-512 or AVX2); for FP4 weights X and the intermediate A are kept in pair-split
    // order, the order in which a row's codes unpack.
    const HostTables4& tb = host_tables();
    const float* slut = wt == FT_W_MXFP4 ? tb.e8m0 : tb.e4m3;
    const bool split = host_row_pair_split(wt);
    const float* Xr = c->X.data();
    if (split) {
      c->Xs.resize((size_t)T * H);
      for (int t = 0; t < T; ++t) split_pairs32(&c->X[(size_t)t * H], H, &c->Xs[(size_t)t * H]);
      Xr = c->Xs.data();
    }
    cpu_parallel_for(c, nE * bi, [&](int task) {
      const int e = c->e_list[task / bi], i0 = (task % bi) * RB;
      const int a0 = c->e_begin[e], n = c->e_begin[e + 1] - a0;
      const uint8_t* r = rec(e);
      thread_local std::vector<const float*> xs;
      thread_local std::vector<float> g, u;
      xs.resize(n);
      g.resize(n);
      u.resize(n);
      for (int q = 0; q < n; ++q) xs[q] = Xr + (size_t)c->arow_t[a0 + q] * H;
      for (int i = i0; i < std::min(I, i0 + RB); ++i) {
        const HostRow rg{wt, r + L.off_val[0] + i * vrow[0], r + L.off_scale[0] + i * srow[0], slut, gscale(e, 0), H};
        const HostRow ru{wt, r + L.off_val[1] + i * vrow[1], r + L.off_scale[1] + i * srow[1], slut, gscale(e, 1), H};
        host_rows(rg, xs.data(), n, g.data());
        host_rows(ru, xs.data(), n, u.data());
        const int pos = split ? (i & ~31) + ((i & 1) ? 16 : 0) + ((i & 31) >> 1) : i;
        for (int q = 0; q < n; ++q) c->A[(size_t)(a0 + q) * I + pos] = g[q] / (1.0f + std::exp(-g[q])) * u[q];
      }
    });
    cpu_parallel_for(c, nE * bh, [&](int task) {
      const int e = c->e_list[task / bh], h0 = (task % bh) * RB;
      const int a0 = c->e_begin[e], n = c->e_begin[e + 1] - a0;
      const uint8_t* r = rec(e);
      thread_local std::vector<const float*> as;
      thread_local std::vector<float> y;
      as.resize(n);
      y.resize(n);
      for (int q = 0; q < n; ++q) as[q] = &c->A[(size_t)(a0 + q) * I];
      for (int h = h0; h < std::min(H, h0 + RB); ++h) {
        const HostRow rd{wt, r + L.off_val[2] + h * vrow[2], r + L.off_scale[2] + h * srow[2], slut, gscale(e, 2), I};
        host_rows(rd, as.data(), n, y.data());
        for (int q = 0; q < n; ++q) c->Y[(size_t)(a0 + q) * H + h] = y[q];
      }
    });
  } else {
    // gate and up: A[r][i] = silu(x_t . gate_i) * (x_t . up_i)
    cpu_parallel_for(c, nE * bi, [&](int task) {
      const int e = c->e_list[task / bi], i0 = (task % bi) * RB;
      const uint8_t* r = rec(e);
      const float gg = gscale(e, 0), gu = gscale(e, 1);
      thread_local std::vector<float> wg, wu;
      wg.resize(H);
      wu.resize(H);
      for (int i = i0; i < std::min(I, i0 + RB); ++i) {
        decode_row(wt, r + L.off_val[0] + i * vrow[0], r + L.off_scale[0] + i * srow[0], gg, H, wg.data());
        decode_row(wt, r + L.off_val[1] + i * vrow[1], r + L.off_scale[1] + i * srow[1], gu, H, wu.data());
        for (int a = c->e_begin[e]; a < c->e_begin[e + 1]; ++a) {
          const float* x = &c->X[(size_t)c->arow_t[a] * H];
          const float g = dot_f32(x, wg.data(), H), u = dot_f32(x, wu.data(), H);
          c->A[(size_t)a * I + i] = g / (1.0f + std::exp(-g)) * u;
        }
      }
    });
    // down: Y[r][h] = A[r] . down_h
    cpu_parallel_for(c, nE * bh, [&](int task) {
      const int e = c->e_list[task / bh], h0 = (task % bh) * RB;
      const uint8_t* r = rec(e);
      const float gd = gscale(e, 2);
      thread_local std::vector<float> wd;
      wd.resize(I);
      for (int h = h0; h < std::min(H, h0 + RB); ++h) {
        decode_row(wt, r + L.off_val[2] + h * vrow[2], r + L.off_scale[2] + h * srow[2], gd, I, wd.data());
        for (int a = c->e_begin[e]; a < c->e_begin[e + 1]; ++a)
          c->Y[(size_t)a * H + h] = dot_f32(&c->A[(size_t)a * I], wd.data(), I);
      }
    });
  }
  // partial[t] = sum over the token's external assignments, j ascending
  cpu_parallel_for(c, T, [&](int t) {
    float* out = j.partial + (size_t)t * H;
    std::fill(out, out + H, 0.0f);
    for (int jj = 0; jj < k; ++jj) {
      const int r = c->rows_of[(size_t)t * k + jj];
      if (r < 0) continue;
      const float w = j.topk_w[(size_t)t * k + jj];
      const float* y = &c->Y[(size_t)r * H];
      for (int h = 0; h < H; ++h) out[h] += w * y[h];
    }
  });
  return FT_OK;
}

}  // namespace ft
