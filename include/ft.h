/*
 * ft.h -- C ABI of the expert-cache MoE layer library (libft.so, sm_103a).
 *
 * One routed-expert MoE layer evaluated over a slot-pool expert cache:
 * router logits -> top-k gating -> permutation by expert -> cache control and
 * miss fill -> grouped SwiGLU expert FFN over cache slots -> weighted combine
 * (+ an optional external partial output), plus whole-layer double-buffered
 * prefill streaming of the expert pool and the q* miss-split rule.
 *
 * Sources (page title, section):
 *   [Review]   "论文综述：FreeToken 让个人电脑跑起前沿 MoE 大模型的边缘原生服务系统"
 *              (paper.oopus.info), §2 opening, §2.2, §2.4, §2.5, §2.6, §2.7, Table 1.
 *   [Overview] "FreeToken – 边缘原生的 MoE（混合专家）模型推理服务系统"
 *              (shshi.cn), "FreeToken技术原理" items 1, 2, 4.
 *
 * Conventions for every call:
 *   - The caller owns every device and pinned-host buffer and keeps it alive
 *     until the work that uses it has finished on the stream.  The library
 *     owns only the opaque handles (ft_cache, ft_stream) and their small
 *     device tables.
 *   - "dev" pointers are CUDA device pointers on the current device; "host"
 *     pointers are ordinary host memory; "pinned" means page-locked host
 *     memory mapped into the device address space (cudaHostAlloc, or
 *     cudaHostRegister with the mapped flag).
 *   - Hot-path calls are asynchronous on the given stream (a cudaStream_t;
 *     NULL = the legacy default stream) and never synchronise the host.  The
 *     calls that synchronise say so.
 *   - Sizes are checked before any launch: a bad size or a NULL where one is
 *     not allowed returns FT_EINVAL and launches nothing.  A CUDA error returns
 *     FT_ECUDA (ft_last_cuda_error() gives the cudaError_t).
 *   - Kernels check every index they read from memory (expert ids, slots,
 *     rows).  An out-of-range index skips the access and records an error
 *     code in a device error word, read and cleared by ft_get_device_error().
 *   - Not thread-safe per handle: use one handle from one host thread.
 */
#ifndef FT_H
#define FT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* ft_cuda_stream; /* a cudaStream_t */

typedef enum {
  FT_OK = 0,
  FT_EINVAL = 1,        /* bad argument or size */
  FT_ENOMEM = 2,        /* device allocation for a handle's tables failed */
  FT_ECUDA = 3,         /* a CUDA runtime call failed */
  FT_ETIMEOUT = 4,      /* a bounded wait ran out */
  FT_ESTATE = 5,        /* call not allowed in the handle's current state */
  FT_EUNSUPPORTED = 6,  /* configuration the library does not handle */
  FT_EDEVICE = 7,       /* a kernel recorded an index error (see ft_get_device_error) */
  FT_EIO = 8            /* a file could not be opened or read to the end */
} ft_status;

/* Stored expert-weight formats ([Overview] feature table: MXFP4, NVFP4, FP8, BF16). */
typedef enum {
  FT_W_F32 = 0,      /* fp32 */
  FT_W_BF16 = 1,     /* bf16 */
  FT_W_FP8E4M3 = 2,  /* e4m3 values, one fp32 scale per 128 consecutive K elements */
  FT_W_NVFP4 = 3,    /* e2m1 values, one e4m3 scale per 16 K elements, one fp32 scale per matrix */
  FT_W_MXFP4 = 4     /* e2m1 values, one E8M0 scale per 32 K elements */
} ft_wtype;

/* Activation (x) formats. */
typedef enum { FT_X_F32 = 0, FT_X_BF16 = 1 } ft_xtype;

/* Device error codes recorded by kernels. */
enum {
  FT_DERR_NONE = 0,
  FT_DERR_EXPERT_INDEX = 1,  /* an expert id outside [0, E) */
  FT_DERR_SLOT_INDEX = 2,    /* a slot outside the pool */
  FT_DERR_ROW_INDEX = 3,     /* a permutation row outside [0, T*k) */
  FT_DERR_TABLE = 4,         /* cache tables inconsistent */
  FT_DERR_TIMEOUT = 5,       /* a kernel's bounded wait on an on-chip barrier ran out; the kernel
                                stopped early and its outputs are incomplete */
  FT_DERR_SCALE_RANGE = 6    /* an MXFP4 block scale above 2^15 (E8M0 byte > 142), beyond the range
                                of the tensor-core expansion; the affected outputs are wrong */
};

const char* ft_status_str(int status);
int ft_version(void);
int ft_last_cuda_error(void);

/* Reads and clears the device error word of the current device (synchronises
 * the device).  *code receives one of FT_DERR_*; returns FT_EDEVICE when it was
 * non-zero, FT_OK otherwise. */
int ft_get_device_error(int* code);

/* Test hook for the failure path of the kernels' bounded waits.  Launches one
 * CTA that waits on an on-chip barrier which nothing completes; after limit_ns
 * (1 .. 2e9) the wait gives up, the kernel records FT_DERR_TIMEOUT, writes 0
 * to *completed (dev int) and returns, leaving the context usable. */
int ft_debug_bounded_wait(int64_t limit_ns, int* completed, ft_cuda_stream s);

/* Host-side failure injection, for tests of the failure paths; nothing is
 * issued to the GPU for a failed call.  With after >= 0, the next `after`
 * calls at `site` succeed and the one after them fails as if the CUDA runtime
 * had refused it (the site then disarms itself); after < 0 disarms the site.
 *   FT_INJECT_DEVICE_ALLOC   device allocations of the handles' tables (ft_cache_create)
 *   FT_INJECT_HOST_PIN       pinning: ft_host_alloc, ft_host_register
 *   FT_INJECT_STREAM_EVENT   streams and events of the handles (ft_cache_create, ft_stream_create) */
enum { FT_INJECT_DEVICE_ALLOC = 1, FT_INJECT_HOST_PIN = 2, FT_INJECT_STREAM_EVENT = 3 };
int ft_debug_inject_failure(int site, int after);

/* Device allocations and streams/events currently held by the library's
 * handles (every call that fails must leave both unchanged). */
int ft_debug_live_resources(int64_t* device_allocs, int64_t* streams_events);

/* The host executor's row form (see ft_cpu_experts): mode 0 the portable row
 * decode, 1 AVX2 + FMA, 2 AVX-512F -- each where the CPU runs it, else the
 * best form below it; any other value only asks.  Returns the form in use
 * before the call (0, 1 or 2).  The default is the best form the CPU runs.
 * Process-wide; for tests and measurements that compare the forms. */
int ft_debug_host_simd(int mode);

/* ------------------------------------------------------------------------
 * Expert record layout.
 *
 * One cache slot holds every tensor of one (layer, expert) ([Review] §2
 * opening: a slot holds all tensors needed to evaluate one layer-expert pair).
 * The host pool and the device slot pool are arrays of such records; host row
 * l*E + e is expert e of physical layer l ([Review] §2.7, expert banks with the
 * flattened first dimension lE+e; here all banks of one expert are one record,
 * so one copy moves one expert and one copy moves one whole layer).
 *
 * Inside a record, K-major matrices (contraction index contiguous), each
 * section starting on a 256-byte boundary, in this order:
 *   gate values [I][H], up values [I][H], down values [H][I],
 *   then (formats with scales) gate scales, up scales, down scales,
 *   then (NVFP4) 3 fp32 matrix scales {gate, up, down}.
 * Values: f32 4 bytes, bf16 2 bytes, e4m3 1 byte, e2m1 4 bits with element 2i
 * in the low nibble of byte i.  Scales per row: fp8 [rows][K/128] fp32,
 * NVFP4 [rows][K/16] e4m3 bytes, MXFP4 [rows][K/32] E8M0 bytes.
 * The record size S is rounded up to a multiple of 256 bytes.
 * ---------------------------------------------------------------------- */
typedef struct {
  uint64_t bytes;           /* S: bytes per record (slot stride) */
  uint64_t payload_bytes;   /* bytes of weights and scales, without padding */
  uint64_t off_val[3];      /* gate, up, down values */
  uint64_t off_scale[3];    /* gate, up, down block scales (0 when the format has none) */
  uint64_t off_gscale;      /* NVFP4: 3 fp32 matrix scales (0 otherwise) */
} ft_expert_layout;

/* Fills *out for a format and shape.  H and I must be multiples of 128. */
int ft_expert_layout_get(int wtype, int hidden, int inter, ft_expert_layout* out);

/* ------------------------------------------------------------------------
 * Pinned host pool.  The full expert pool lives in page-locked host memory,
 * mapped into the device address space, so that copies and kernels can read
 * it over the host link ([Review] §2 opening: the host pool is the source of
 * truth; §2.7: the pool must be pinned for DMA).  A failed pin returns
 * FT_ENOMEM (there is no unpinned fallback).
 * ---------------------------------------------------------------------- */
int ft_host_alloc(uint64_t bytes, void** out);  /* *out = pinned, mapped, 4 KiB aligned */
int ft_host_free(void* p);

/* Read-then-pin pool setup ([Review] §2.7, fast engine start: the experts are
 * read into their final host layout first and pinned only afterwards, because
 * pinning first makes the driver fault in and zero every page of a pool of
 * tens of GB before the read writes it again).
 *
 * ft_pool_read: reads `bytes` of the file `path` from byte `offset` into host
 * memory dst (any host memory; typically a fresh page-aligned anonymous mapping
 * that the read itself faults in) with `threads` threads (1 .. 256; 0 picks
 * the hardware thread count, at most 64).  The file holds expert records in
 * the pool's row order l*E + e (one record of ft_expert_layout.bytes per row),
 * so one contiguous read fills whole layers.  FT_EIO when the file cannot be
 * opened or ends early.  Host only; no GPU is touched.
 *
 * ft_host_register: pins and maps an already-filled host buffer (p 4 KiB
 * aligned, bytes > 0) so that copies and kernels can read it over the host
 * link, as memory from ft_host_alloc.  FT_ENOMEM when pinning fails (there is
 * no unpinned fallback).  ft_host_unregister undoes it (the memory stays the
 * caller's). */
int ft_pool_read(const char* path, uint64_t offset, void* dst, uint64_t bytes, int threads);
int ft_host_register(void* p, uint64_t bytes);
int ft_host_unregister(void* p);

/* ------------------------------------------------------------------------
 * Router logits: z[t][e] = sum_h x[t][h] * W_r[h][e] + bias[e] (fp32 accumulate).
 * The gating network that picks each token's experts ([Review] §1, MoE
 * routing; the pages do not spell out the gate).
 *   x        dev [T][H], x_type
 *   w_router dev [E][H] (K-major), same type as x
 *   bias     dev [E] fp32, or NULL
 *   logits   dev [T][E] fp32 (written)
 * T >= 0, H a multiple of 8, 1 <= E <= 1024.
 * ---------------------------------------------------------------------- */
int ft_router_logits(const void* x, int x_type, const void* w_router, const float* bias,
                     int T, int H, int E, float* logits, ft_cuda_stream s);

/* ------------------------------------------------------------------------
 * ft_route: softmax over all E experts, top-k, renormalise over the k chosen.
 * Experts are ranked by descending logit (softmax is increasing in the logit);
 * equal logits go to the lower index.  Output j = 0..k-1 in rank order.
 * topk_w[t][j] = exp(z_j - z_0) / sum_{i<k} exp(z_i - z_0), which equals the
 * full softmax renormalised over the chosen k.
 *   logits   dev [T][E] fp32
 *   topk_idx dev [T][k] int32 (written)
 *   topk_w   dev [T][k] fp32 (written)
 * 1 <= k <= min(E, 16), 1 <= E <= 1024.  NaN logits give unspecified (but
 * in-range) choices.
 * ---------------------------------------------------------------------- */
int ft_route(const float* logits, int T, int E, int k, int32_t* topk_idx, float* topk_w,
             ft_cuda_stream s);

/* ------------------------------------------------------------------------
 * ft_permute: groups the T*k assignments a = t*k + j by expert for grouped
 * evaluation ([Review] §2.5: the GPU evaluates its expert set grouped by expert).
 *   topk_idx dev [T*k] int32 in [0, E)
 *   counts   dev [E]    (written) assignments per expert
 *   offsets  dev [E+1]  (written) exclusive prefix sum, offsets[E] = T*k
 *   perm     dev [T*k]  (written) perm[offsets[e] + r] = the r-th assignment
 *                       routed to e, in ascending a (stable)
 *   inv      dev [T*k]  (written) inv[perm[p]] = p
 * 1 <= E <= 512.  Deterministic.
 * ---------------------------------------------------------------------- */
int ft_permute(const int32_t* topk_idx, int T, int k, int E, int32_t* counts, int32_t* offsets,
               int32_t* perm, int32_t* inv, ft_cuda_stream s);

/* ------------------------------------------------------------------------
 * ft_route_fused: ft_router_logits, ft_route and ft_permute of one batch, with
 * the same arguments and results (the logits are bit-identical), for the
 * per-token routing and grouping of a decode step.  Batches of at most 8
 * tokens (with min(T, 8) * H * (2 for bf16 x, 4 for fp32) bytes of staged
 * rows <= 200 KiB) run as one launch over the grid of ft_router_logits: each
 * CTA computes the logits of a share of the experts; the CTA that finishes
 * last routes the tokens and groups the assignments.  Larger batches (and
 * T = 0) run the three kernels, which are faster there.
 * arrivals: device uint32[FT_ROUTE_ARRIVAL_WORDS], caller-owned, all zero
 * before the first call; every call leaves them zero again.  One call at a
 * time per array (calls in flight on several streams need one array each).
 * A nonzero word at launch is recorded as FT_DERR_TABLE, and that call's
 * outputs are not valid.  Unused (may be NULL) when the batch runs the three
 * kernels.
 * T >= 0, H a multiple of 8, 1 <= E <= 512, 1 <= k <= min(E, 16).
 * ---------------------------------------------------------------------- */
#define FT_ROUTE_ARRIVAL_WORDS 16

int ft_route_fused(const void* x, int x_type, const void* w_router, const float* bias, int T, int H, int E, int k,
                   float* logits, int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                   int32_t* perm, int32_t* inv, uint32_t* arrivals, ft_cuda_stream s);

/* ------------------------------------------------------------------------
 * ft_cache: one LRU cache of expert records shared by all MoE layers, keyed by
 * the logical (layer, expert) ([Review] §2 opening, §2.4).  The full expert
 * pool stays in pinned host memory; GPU memory changes only speed, never the
 * result ([Review] §2 opening).
 *
 * Per layer step, one kernel de-duplicates the routed experts, classifies hits
 * and misses against the residency table, takes q from the bandwidth ratio,
 * picks victims in one pass over the recency order and rewrites every routed
 * expert to a slot or to the "evaluate elsewhere" marker ([Review] §2.6,
 * device-side cache control and one-pass victim selection); a second
 * fixed-shape launch copies the q filled experts from the pinned pool into
 * their slots, driven by a device-resident (source, destination) table and a
 * device valid count ([Review] §2.6, one fused transfer).
 *
 * Rules where the pages are silent: routed experts in ascending id; the q
 * filled misses are the first q misses in ascending id; a step with more
 * unique experts than slots runs in waves of at most N experts, each wave
 * with its own recency stamp; victims are empty slots first (ascending slot),
 * then untouched slots by (stamp, slot).
 * ---------------------------------------------------------------------- */
typedef struct ft_cache ft_cache;

typedef struct {
  int n_layers;            /* logical layers L (keys are layer*E + expert) */
  int n_experts;           /* E per layer, 1..1024 */
  int n_phys_layers;       /* layers stored in the host pool; logical l reads physical l % n_phys_layers */
  int n_slots;             /* initial capacity N, 1..max_slots */
  int max_slots;           /* records the device slot pool can hold, <= 16384 */
  uint64_t slot_bytes;     /* S, from ft_expert_layout_get */
  const void* host_pool;   /* pinned [n_phys_layers*E][S]; caller-owned */
  void* slot_pool;         /* dev [max_slots][S]; caller-owned */
} ft_cache_config;

typedef struct {
  uint64_t steps, hits, fills, externals, bytes_h2d;
} ft_cache_stats_t;

/* Creates the handle and its device tables (all slots empty).  Synchronises. */
int ft_cache_create(const ft_cache_config* cfg, ft_cache** out);
int ft_cache_destroy(ft_cache* c);

/* Waves a layer step may need: ceil(E / N). */
int ft_cache_n_waves(const ft_cache* c);

/* One wave of one layer step (asynchronous on s).
 *   layer       logical layer, 0 <= layer < n_layers
 *   counts      dev [E] int32, assignments per expert (> 0 = routed)
 *   fill_ratio  B_P / B_H; q = clamp(floor(m*ratio + 0.5), 1, m) for m >= 1
 *               misses; ratio >= 1 fills every miss ([Review] §2.5)
 *   wave        0 .. ft_cache_n_waves()-1; wave w holds routed experts of
 *               rank [w*N, (w+1)*N) in ascending id; an empty wave is a no-op
 *   slot_of     dev [E] int32 (written): slot (>= 0) for this wave's experts
 *               evaluated on the GPU, -2 for this wave's experts left to the
 *               external path, -1 for every other expert
 *   ext_flags   dev [E] int32 or NULL: wave 0 clears it, every wave sets 1 for
 *               its external experts (the skip mask of ft_combine)
 *   step_counts dev [4] int32 or NULL (written): {experts in wave, hits,
 *               fills (q), externals (m - q)}
 * The fill copies are ordered on s before any later work on s. */
int ft_cache_step(ft_cache* c, int layer, const int32_t* counts, double fill_ratio, int wave,
                  int32_t* slot_of, int32_t* ext_flags, int32_t* step_counts, ft_cuda_stream s);

/* Split form of ft_cache_step: the miss fill runs on a second stream so that
 * the hits can be evaluated while the filled experts are copied ([Review]
 * §2.6: the fill is one launch after the control pass; hits need no copy).
 * Same decisions, tables, counters and step_counts as ft_cache_step.
 *   slot_hit    dev [E] int32 (written): slot for this wave's hits, -2 for its
 *               external experts, -1 for every other expert (filled ones too)
 *   slot_fill   dev [E] int32 (written): slot for this wave's filled experts,
 *               -1 for every other expert
 *   fill_s      stream of the fill copies; it waits for the control launch on
 *               s.  fill_s == s runs both on s (ft_cache_fill_join is then a no-op)
 * Reading the hit slots on s right after this call is safe: their records are
 * resident and the fill writes only victims, which are slots this wave does
 * not touch.  The filled slots may be read on s only after
 * ft_cache_fill_join(c, s), which makes s wait for the fill.  Until that join,
 * ft_cache_step, ft_cache_step_split, ft_cache_resize and ft_stream_create on
 * this handle return FT_ESTATE.  Under stream capture the join must come
 * before the capture ends (it joins fill_s back into s).
 * Passing slot_hit to ft_expert_grouped, then slot_fill after the join, gives
 * the same y as one call with ft_cache_step's slot_of (ft_expert_grouped's
 * results do not depend on which other experts a call evaluates). */
int ft_cache_step_split(ft_cache* c, int layer, const int32_t* counts, double fill_ratio, int wave,
                        int32_t* slot_hit, int32_t* slot_fill, int32_t* ext_flags, int32_t* step_counts,
                        ft_cuda_stream s, ft_cuda_stream fill_s);
int ft_cache_fill_join(ft_cache* c, ft_cuda_stream s);

/* Thread blocks of the fill launch (default 32; 256 threads, 16 KiB of host
 * reads in flight each), 1 .. 4 x the SM count; applies to later steps.  More blocks
 * keep more reads in flight over the host link; reads queued beyond what the
 * link needs also delay the device-memory reads of kernels running beside the
 * fill (the hits of a split step). */
int ft_cache_set_fill_blocks(ft_cache* c, int blocks);

/* Safe-point rebuild for a new slot budget without touching the host pool
 * ([Review] §2.7, runtime cache reconfiguration).  Keeps the min(used, N')
 * most recent entries (largest (stamp, -slot)); kept entries below N' stay,
 * kept entries at or above N' move (ascending old slot) into the lowest free
 * slots below N'.  Synchronises the device.  FT_ESTATE while a stream handle
 * holds the pool's buffers. */
int ft_cache_resize(ft_cache* c, int n_slots);

/* Cold restart at a safe point ([Review] §2.7: the engine serves its first
 * request from a cold cache, with no warm-up): every slot empty, the recency
 * clock and the counters back to zero, the capacity kept.  The handle's device
 * tables stay where they are, so CUDA graphs captured over the handle remain
 * valid.  Synchronises the device.  FT_ESTATE while a stream handle holds the
 * pool's buffers or a split step waits for its join. */
int ft_cache_reset(ft_cache* c);

/* Counters since creation or the last ft_cache_reset.  Synchronises. */
int ft_cache_stats(ft_cache* c, ft_cache_stats_t* out);

/* Copies the residency state to host arrays of at least max_slots entries:
 * key_of_slot (-1 empty, else layer*E + expert) and stamp (0 for empty);
 * *n_slots = current N, *clock = last stamp issued.  Synchronises. */
int ft_cache_export(ft_cache* c, int32_t* key_of_slot, uint32_t* stamp, int* n_slots, uint32_t* clock);

/* ------------------------------------------------------------------------
 * ft_expert_grouped: per expert e with rows and slot_of[e] >= 0,
 *   Y_e = (silu(X_e W_g[e]) * (X_e W_u[e])) W_d[e]
 * with the weights read from the expert's slot and dequantised in the kernel
 * ([Review] §2.5: grouped evaluation of the GPU expert set from cache slots).
 *   x           dev [T][H], x_type
 *   perm,offsets from ft_permute (row p of Y is assignment perm[p], token perm[p]/k)
 *   slot_of     dev [E] int32; experts with slot_of < 0 are skipped and their
 *               rows of y are left untouched
 *   slot_pool   dev [pool_slots][S] expert records of format wtype (256-aligned);
 *               a slot_of value >= pool_slots is a device error
 *   y           dev [T*k][H] fp32 (written for evaluated experts), permuted order
 *   workspace   dev, >= ft_expert_grouped_workspace(T, k, H, I) bytes, 256-aligned
 * Accumulation is fp32.  Each output element is reduced in a fixed order, so
 * results do not depend on which other experts are evaluated in the same call
 * or on the slot used.
 *
 * Two execution paths, chosen by the weight format:
 *   - bf16 (above FT_CC_MAX_ASSIGNMENTS assignments), NVFP4 and MXFP4 weights:
 *     tcgen05 tensor cores.  Below FT_TC_WIDE_ASSIGNMENTS assignments (T*k) the weights are the
 *     MMA's M side (128 weight rows) and up to 64 of an expert's token rows its
 *     N side, with the K range split when few experts are routed; from
 *     FT_TC_WIDE_ASSIGNMENTS up, 128 token rows against 128 or 256 weight rows
 *     (256 for bf16 when H is a multiple of 256).  x is rounded to bf16 (round
 *     to nearest even) for the products, the intermediate silu(G)*U is rounded
 *     to bf16 before the down product, and products accumulate in fp32.  FP4
 *     weights are expanded to bf16 in shared memory first; the expansion is
 *     exact (e2m1 value times block scale is a bf16 value), except that an
 *     MXFP4 block scale above 2^15 (E8M0 byte > 142) is beyond its range: the
 *     kernel records FT_DERR_SCALE_RANGE and those outputs are wrong.  NVFP4's
 *     fp32 matrix scale multiplies the fp32 results.
 *   - fp32 and FP8 weights, and bf16 weights at T*k <= FT_CC_MAX_ASSIGNMENTS
 *     (one decode token: each expert's product is a matrix-vector product,
 *     which the tensor cores would only pad): CUDA cores, weights streamed
 *     once per 8-row chunk of an expert's rows and dequantised in registers; x
 *     and the intermediate silu(G)*U stay in fp32.
 * ---------------------------------------------------------------------- */
#define FT_TC_WIDE_ASSIGNMENTS 2048
#define FT_CC_MAX_ASSIGNMENTS 8

/* How the tensor cores evaluate NVFP4 / MXFP4 experts, process-wide, for later
 * calls:
 *   FT_FP4_BLOCK_SCALED (default): the block-scaled FP4 MMA (kind::mxf4nvf4)
 *     reads the packed weights and their block scales directly; the token rows
 *     and the intermediate silu(G)*U are quantised to the weights' format,
 *     block by block along K in fp32 (NVFP4: blocks of 16, scale e4m3(amax/6),
 *     values e2m1(v/scale), both round to nearest even and saturating; MXFP4:
 *     blocks of 32, scale 2^(floor(log2 amax) - 2) as E8M0).  Needs H and I
 *     multiples of 256 (other shapes take the expansion).  Small batches: 128
 *     weight rows x up to 64 token rows per tile; large batches: 128 token
 *     rows x 128 weight rows.
 *   FT_FP4_EXPAND_BF16: the weights are expanded exactly to bf16 in shared
 *     memory and multiplied as bf16 (x and the intermediate rounded to bf16). */
enum { FT_FP4_BLOCK_SCALED = 0, FT_FP4_EXPAND_BF16 = 1 };
int ft_expert_set_fp4_path(int path);

/* Test hook: the activation quantiser of the block-scaled path on its own.
 * Rows of x (dev [rows][K], x_type) -> q (dev [rows][K/2] e2m1 bytes, element
 * 2i in the low nibble) and scales (dev [rows][K/16] e4m3 bytes for
 * FT_W_NVFP4, [rows][K/32] E8M0 bytes for FT_W_MXFP4).  K a multiple of 32. */
int ft_debug_quant_fp4(const void* x, int x_type, int rows, int K, int wtype, uint8_t* q, uint8_t* scales,
                       ft_cuda_stream s);
size_t ft_expert_grouped_workspace(int T, int k, int hidden, int inter);
int ft_expert_grouped(const void* x, int x_type, int T, int k, int hidden, int inter, int E,
                      int wtype, const int32_t* perm, const int32_t* offsets, const int32_t* slot_of,
                      const void* slot_pool, uint64_t slot_bytes, int pool_slots, float* y,
                      void* workspace, size_t workspace_bytes, ft_cuda_stream s);

/* ------------------------------------------------------------------------
 * ft_expert_grouped_noalloc: the grouped expert FFN with the arguments of
 * ft_expert_grouped, without the workspace.  The pages have no counterpart:
 * this entry point exists for callers that cannot call cudaMalloc -- a host
 * application that owns every device allocation through its own allocator or
 * fixed budget, or a latency-critical path where cudaMalloc's implicit device
 * synchronisation is not acceptable.  The library allocates nothing here.
 *
 * It always runs the CUDA-core kernels, for every weight format: weights
 * dequantised in registers, x and the intermediate silu(G)*U in fp32.  Where
 * ft_expert_grouped takes the tensor cores (bf16 weights above
 * FT_CC_MAX_ASSIGNMENTS assignments, NVFP4 and MXFP4 weights, with a bf16 or
 * quantised intermediate) the results therefore differ within the tolerance
 * of that rounding, not bit for bit, and this call is slower (measured on
 * B300, bf16 weights, H=2048, I=512, top-8: 0.065 against 0.041 ms at 4
 * tokens, 0.605 against 0.075 ms at 64 tokens).
 *
 * The fp32 intermediate lives in one fixed device array inside the library,
 * FT_NOALLOC_MAX_ELEMS floats (4 MiB), which every GPU that loads the library
 * holds until the process exits.  Calls with T*k*inter > FT_NOALLOC_MAX_ELEMS
 * return FT_EINVAL and launch nothing.
 *
 * The first call in each CUDA context (per device; again after a
 * cudaDeviceReset) looks up the array's device address (cudaGetSymbolAddress,
 * with that device current); make that first call before any stream capture.
 * All calls share the one array and it keeps the last call's contents
 * (nothing needs clearing: each call writes every element it reads before
 * reading it).  Calls that overlap on the GPU -- on different streams, or from
 * different host threads -- race on the array: order them.
 * ---------------------------------------------------------------------- */
#define FT_NOALLOC_MAX_ELEMS (1u << 20)
int ft_expert_grouped_noalloc(const void* x, int x_type, int T, int k, int hidden, int inter, int E,
                              int wtype, const int32_t* perm, const int32_t* offsets,
                              const int32_t* slot_of, const void* slot_pool, uint64_t slot_bytes,
                              int pool_slots, float* y, ft_cuda_stream s);

/* ------------------------------------------------------------------------
 * ft_combine: out[t] = sum_j topk_w[t][j] * y[inv[t*k+j]] + ext_partial[t],
 * skipping assignments whose expert has ext_flags != 0.  GPU and external
 * partial sums are added, keeping the MoE output exact ([Review] §2.5, the
 * exact merge).  Sum order: j = 0..k-1, then the partial.
 *   y           dev [T*k][H] fp32 (from ft_expert_grouped)
 *   inv, topk_idx, topk_w  from ft_permute / ft_route
 *   ext_flags   dev [E] int32 or NULL (no assignment skipped)
 *   ext_partial dev [T][H] fp32 or NULL
 *   out         dev [T][H] fp32 (written)
 * H a multiple of 4, 1 <= k <= 16.
 * ---------------------------------------------------------------------- */
int ft_combine(const float* y, const int32_t* inv, const int32_t* topk_idx, const float* topk_w,
               const int32_t* ext_flags, const float* ext_partial, int T, int k, int H, int E,
               float* out, ft_cuda_stream s);

/* ------------------------------------------------------------------------
 * ft_stream: whole-layer double-buffered prefill streaming ([Review] §2.2;
 * [Overview] "FreeToken技术原理" item 2).  Two whole-layer buffers (2E slots)
 * are carved from the end of the cache's slot pool (a resize to N - 2E).
 * While layer l is computed from one buffer, a transfer stream copies all of
 * layer l+1 into the other with one cudaMemcpyAsync from the pinned pool,
 * before l+1's routing is known.  Events order the copy after the compute that
 * last read the buffer, and the compute after its copy.  In serialized mode
 * the copy of l+1 starts only after layer l's compute (the ablation without the
 * second buffer's overlap).
 * ---------------------------------------------------------------------- */
typedef struct ft_stream ft_stream;

/* Carves the buffers (synchronises).  FT_EUNSUPPORTED when N < 2E: the caller
 * then runs prefill through ft_cache_step (on-demand waves). */
int ft_stream_create(ft_cache* c, int serialized, ft_stream** out);

/* Makes `compute` wait until `layer` is resident (issuing its copy first if it
 * was not prefetched), writes slot_of[e] = its buffer slot for every e (dev
 * [E] int32), and, unless serialized, issues the copy of next_layer (-1: none)
 * into the other buffer. */
int ft_stream_layer(ft_stream* st, int layer, int next_layer, int32_t* slot_of, ft_cuda_stream compute);

/* Marks the end of `layer`'s compute on `compute` (its buffer may be refilled
 * after this point); in serialized mode issues the pending next copy here. */
int ft_stream_layer_done(ft_stream* st, int layer, ft_cuda_stream compute);

/* Bytes copied host->device by this handle so far. */
int ft_stream_bytes(const ft_stream* st, uint64_t* bytes);

/* Waits for the transfer stream, gives the 2E slots back and adopts the
 * experts of the last two streamed layers into the LRU table (older layer
 * first, one stamp per layer, experts in ascending id; a key already resident
 * is refreshed and its buffer slot left empty): entries that survive prefill
 * warm decode ([Review] §2.2).  Synchronises. */
int ft_stream_destroy(ft_stream* st);

/* ------------------------------------------------------------------------
 * Host-side expert executor ([Review] §2.5: the experts of C, the misses not
 * filled into the cache, are evaluated where their weights live, from the
 * host pool, and their gate-weighted outputs form a partial sum that the GPU
 * adds to its own, so the layer output stays exact; §2.6: the CPU branch is a
 * node of the captured step).  A handle owns a pool of CPU threads.
 *
 * One job evaluates, for every token t and every j with ext_flags[topk_idx[t][j]]
 * != 0, w[t][j] * FFN_e(x[t]) from the host pool's record of (phys_layer, e),
 * and writes partial[t] = their sum over j ascending (0 where there is none).
 * Weights are decoded to fp32 row by row (every ft_wtype); x, the intermediate
 * silu(G)*U and the accumulation are fp32.  On x86-64 CPUs with AVX-512F, or
 * AVX2 and FMA, the rows are decoded in registers instead (FP4 codes through a
 * register table, one
 * scale per block; e4m3 bytes by moving their fields into place) and dotted
 * with all of an expert's tokens at once; the weights take the same values,
 * the sums run in another order (fp32 rounding differs, the results stay
 * deterministic).  Every pointer is host memory:
 *   host_pool  [n_phys_layers*E][slot_bytes] records (the cache's pinned pool)
 *   x          [T][hidden] of x_type;  topk_idx, topk_w  [T][k];
 *   ext_flags  [n_experts] (ft_cache_step's external marks);  partial [T][hidden] fp32
 * T = 0 is a no-op (the pointers may then be null).  FT_EINVAL for a null
 * pointer otherwise, T < 0, k < 1, a shape ft_expert_layout_get refuses, or
 * slot_bytes below the record size.
 * ---------------------------------------------------------------------- */
typedef struct ft_cpu ft_cpu;
typedef struct {
  const void* host_pool;
  uint64_t slot_bytes;
  int wtype, hidden, inter, n_experts, phys_layer;
  const void* x;
  int x_type, T, k;
  const int32_t* topk_idx;
  const float* topk_w;
  const int32_t* ext_flags;
  float* partial;
} ft_cpu_job;

/* threads: worker threads besides the caller (0 = hardware threads - 1, at most 255). */
int ft_cpu_create(int threads, ft_cpu** out);
/* Waits for nothing: destroy only when no enqueued job can still run. */
int ft_cpu_destroy(ft_cpu* c);
/* Runs one job now, on the calling thread and the pool. */
int ft_cpu_experts(ft_cpu* c, const ft_cpu_job* job);
/* Enqueues one job as a host function on stream s (cudaLaunchHostFunc; under
 * stream capture it becomes a host node of the graph, run at every replay).
 * The job is copied into the handle and kept until ft_cpu_destroy; its
 * pointers must stay valid for every run -- typically pinned buffers that
 * copies on s fill before the node and drain after it.  A failed run records
 * its status, which ft_cpu_status reads and clears. */
int ft_cpu_experts_enqueue(ft_cpu* c, const ft_cpu_job* job, ft_cuda_stream s);
int ft_cpu_status(ft_cpu* c);

/* ------------------------------------------------------------------------
 * Placement-policy replay (host only) ([Review] §2.4, the ablation that
 * replays routing traces under three placements of equal capacity and counts
 * the routed experts that are not in GPU memory).
 *   FT_PLACE_GLOBAL_LRU      the shared LRU of ft_cache, starting empty, every
 *                            miss filled (the cache step's victim rules);
 *                            capacity >= n_experts
 *   FT_PLACE_PREFILL_HOT     a hot set fixed at prefill time: the `capacity`
 *                            keys with the most prefill assignments
 *                            (prefill_counts, host [n_layers*n_experts]), ties
 *                            to the lower key, resident for the whole trace
 *   FT_PLACE_STATIC_SPLIT    a routing-agnostic split made at load time: keys
 *                            0 .. capacity-1 (whole layers in order) resident
 *   trace       host [n_steps][n_layers][width] int32 expert ids of each layer
 *               step's assignments (duplicates allowed, -1 = padding)
 *   accesses    (written) unique routed experts over all layer steps
 *   misses      (written) those not resident when routed
 * Keys are layer * n_experts + expert; 1 <= capacity <= n_layers*n_experts.
 * ---------------------------------------------------------------------- */
enum { FT_PLACE_GLOBAL_LRU = 0, FT_PLACE_PREFILL_HOT = 1, FT_PLACE_STATIC_SPLIT = 2 };
int ft_placement_replay(int policy, int n_layers, int n_experts, int capacity, const int32_t* prefill_counts,
                        const int32_t* trace, int n_steps, int width, uint64_t* accesses, uint64_t* misses);

/* ------------------------------------------------------------------------
 * ft_qsplit (host only, pure): q* = m B_P / B_H, rounded half up, at least 1,
 * at most m; m when B_H <= B_P; 0 when m <= 0 ([Review] §2.5, balance equation
 * and the rounding rule after it).
 * ---------------------------------------------------------------------- */
int ft_qsplit(int m, double bw_fill, double bw_host);

#ifdef __cplusplus
}
#endif
#endif /* FT_H */
