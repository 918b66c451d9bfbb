// Whole-layer double-buffered prefill streaming over two buffers carved from
// the cache's slot pool.
#pragma once
#include "cache.cuh"

struct ft_stream {
  ft_cache* c;
  int serialized;
  int base;                 // first buffer slot; buffer b = slots base + b*E .. + E - 1
  cudaStream_t copy;        // transfer stream
  cudaEvent_t ready[2];     // buffer b holds buf_layer[b]
  cudaEvent_t freed[2];     // compute done with buffer b
  bool freed_rec[2];
  int buf_layer[2];
  int next_buf;
  int pending_layer, pending_buf;  // serialized mode: copy to issue at layer_done
  uint64_t bytes;
  int hist_layer[2], hist_buf[2];  // last two copies issued, older first
  int n_hist;
};

namespace ft {

static int stream_issue_copy(ft_stream* st, int layer, int b, cudaEvent_t extra_wait) {
  ft_cache* c = st->c;
  if (st->freed_rec[b]) FT_CHECK_CUDA(cudaStreamWaitEvent(st->copy, st->freed[b], 0));
  if (extra_wait) FT_CHECK_CUDA(cudaStreamWaitEvent(st->copy, extra_wait, 0));
  const uint64_t bytes = (uint64_t)c->E * c->S;
  const uint8_t* src = c->host + (uint64_t)(layer % c->Lp) * bytes;
  uint8_t* dst = c->pool + (uint64_t)(st->base + b * c->E) * c->S;
  FT_CHECK_CUDA(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, st->copy));
  FT_CHECK_CUDA(cudaEventRecord(st->ready[b], st->copy));
  st->buf_layer[b] = layer;
  st->bytes += bytes;
  if (st->n_hist == 2) {
    st->hist_layer[0] = st->hist_layer[1];
    st->hist_buf[0] = st->hist_buf[1];
    st->n_hist = 1;
  }
  st->hist_layer[st->n_hist] = layer;
  st->hist_buf[st->n_hist] = b;
  st->n_hist += 1;
  return FT_OK;
}

static int buffer_of(const ft_stream* st, int layer) {
  if (st->buf_layer[0] == layer) return 0;
  if (st->buf_layer[1] == layer) return 1;
  return -1;
}

// Gives the carved slots back and adopts the experts of the last two streamed
// layers (older first, one stamp per layer, ascending expert id).
static int stream_adopt(ft_stream* st) {
  ft_cache* c = st->c;
  HostTables t;
  int s = download_tables(c, t);
  if (s) return s;
  const int E = c->E;
  const int base = st->base;
  t.key.resize(c->n_full, -1);
  t.stamp.resize(c->n_full, 0);
  std::vector<int32_t> where((size_t)c->L * E, -1);
  for (int i = 0; i < base; ++i)
    if (t.key[i] >= 0) where[t.key[i]] = i;
  for (int h = 0; h < st->n_hist; ++h) {
    const int layer = st->hist_layer[h], b = st->hist_buf[h];
    if (st->buf_layer[b] != layer) continue;  // overwritten later
    bool newer_same = false;
    for (int h2 = h + 1; h2 < st->n_hist; ++h2) newer_same |= st->hist_layer[h2] == layer;
    if (newer_same) continue;
    t.clock += 1;
    for (int e = 0; e < E; ++e) {
      const int key = layer * E + e;
      const int sb = base + b * E + e;
      if (where[key] >= 0) {
        t.stamp[where[key]] = t.clock;
      } else {
        t.key[sb] = key;
        t.stamp[sb] = t.clock;
        where[key] = sb;
      }
    }
  }
  s = upload_tables(c, t);
  if (s) return s;
  FT_CHECK_CUDA(cudaDeviceSynchronize());
  return FT_OK;
}

}  // namespace ft
