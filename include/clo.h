/*
 * clo.h -- C ABI of the CLO decode-step library for GB300 (sm_103a).
 *
 * CLO is a CPU-light KV-cache offloading system: the full K/V cache of every
 * sequence lives in pinned host memory, and each decode step attends only to the
 * top-k (10 %) tokens of each KV head, chosen by a hash-code scorer.  A head whose
 * query barely moved since its last refresh reuses its previous on-GPU selection;
 * a few "persistent" heads stay fully resident in HBM; everything else is fetched
 * from host memory by GPU loads, with no CPU thread on the data path.
 *
 * Sources (page title, section):
 *   [ABS] CLO abstract (arXiv 2511.14510v1, paper-check page): KV in CPU memory
 *         with top-k attention; features (1) head-wise approximate on-GPU cache,
 *         (2) prefetching combined with on-GPU persistent caching, (3) zero-copy
 *         transfer engine and GPU-centric synchronisation.
 *   [SYN] "CLO (2511.14510) - L3 Per-Paper Synthesis": section 2.1 (query cosine
 *         similarity > 0.8 between adjacent steps as the reuse condition; UVA
 *         polling), 2.2 (top-k = 10 %), 3.2 (HATA top-k scorer), 3.3 attack 6
 *         (s_hat_i, D_i, N_persist from profiling), 5.6 (prefetch one layer ahead),
 *         5.7 (KV produced at prefill and offloaded once).
 *
 * Conventions
 *   - Every call returns a clo_status; nothing aborts, throws or traps.  The text
 *     of the last error of the calling thread is returned by clo_last_error().
 *   - Element type is bf16 (uint16 bit patterns) for K, V, queries and the hash
 *     projection; attention outputs are fp32.
 *   - A "unit" is one (layer, sequence, kv head).  G = n_q_heads / n_kv_heads
 *     query heads share a unit (GQA).
 *   - Device pointers passed in stay owned by the caller; the library owns all
 *     memory it allocates (pinned host pool, HBM buffers) and frees it in
 *     clo_destroy().
 *   - Device-side failures (a ready-flag wait that ran out of time, an internal
 *     bounds check) are latched in a device error word and reported by the next
 *     call that synchronises with the stream: clo_sync(), clo_stats(), a
 *     host-buffer clo_decode_step(), or clo_debug_get().
 */
#ifndef CLO_H_
#define CLO_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define CLO_API __attribute__((visibility("default")))
#else
#define CLO_API
#endif

typedef struct clo_ctx clo_ctx; /* opaque */

typedef enum {
  CLO_OK = 0,
  CLO_ERR_INVALID = 1,  /* bad argument or configuration */
  CLO_ERR_OOM = 2,      /* host (pinned) or device allocation failed */
  CLO_ERR_CUDA = 3,     /* a CUDA runtime call failed */
  CLO_ERR_TIMEOUT = 4,  /* a device-side ready-flag wait gave up (bounded wait) */
  CLO_ERR_STATE = 5,    /* call not valid in the context's current state */
  CLO_ERR_CAPACITY = 6, /* append beyond max_tokens */
  CLO_ERR_DEVICE = 7    /* a device-side bounds check failed */
} clo_status;

/* Reuse decision of a unit in one step (as read back by clo_debug_get). */
enum { CLO_DEC_HIT = 0, CLO_DEC_MISS = 1, CLO_DEC_PERSIST = 2 };

typedef struct clo_config {
  int32_t n_layers;   /* L >= 1 */
  int32_t batch;      /* B >= 1 sequences */
  int32_t n_q_heads;  /* Hq, multiple of n_kv_heads, G = Hq/Hkv <= 8 */
  int32_t n_kv_heads; /* Hkv >= 1 */
  int32_t head_dim;   /* d: 64 or 128 */
  int64_t max_tokens; /* capacity per sequence (sizes the pinned host pool); <= 524288 */
  /* top-k budget: topk > 0 -> k = min(topk, N); else k = ceil(topk_ratio * N),
   * evaluated as one IEEE double product, clamped to [1, N]  ([SYN] 2.2: 10 %) */
  int64_t topk;
  double topk_ratio;
  /* hash projection R: host bf16 [L][Hkv][d][128] (row i, column j at i*128+j);
   * required; copied.  Bit j of the code of x is 1 iff the exact real value of
   * sum_i x_i R_ij is > 0 ([SYN] 3.2 names HATA as the top-k scorer). */
  const uint16_t* hash_R;
  /* reuse thresholds tau: host fp32 [L][Hkv], copied; NULL -> warm-up profiling:
   * the first warmup_steps steps reselect every unit, s_hat[l][h] = mean over the
   * batch and adjacent step pairs of cos(q_t, q_{t-1}), tau = s_hat - tau_offset,
   * and the n_persist heads with the lowest s_hat per layer become persistent
   * ([SYN] 3.3 attack 6; [SYN] 2.1 item 2). */
  const float* tau;
  /* persistent heads when tau is given: host uint8 [L][Hkv] (nonzero = resident),
   * or NULL for none ([ABS] feature (2)). */
  const uint8_t* persist_mask;
  int32_t warmup_steps; /* >= 2 when tau == NULL (default 16) */
  float tau_offset;     /* default 0.05 */
  int32_t n_persist;    /* persistent heads per layer after warm-up, < Hkv */
  int64_t wait_timeout_ns; /* bound of every device-side ready-flag wait; <= 0 -> 2 s */
  int32_t timing;          /* nonzero: record per-phase CUDA-event times (clo_stats) */
  int32_t debug_drop_flag_layer; /* fault injection: >= 0 -> the fetch of this layer
                                    never signals its ready flags; -1 = off */
  void* stream;            /* cudaStream_t to run on; NULL = the legacy default stream */
  /* online adaptive thresholds ([SYN] 5.3: online adaptation instead of offline
   * profiling only): nonzero -> after warm-up (or from the first step with fixed tau,
   * starting from s_hat = tau + tau_offset), every step updates, per (layer, kv head),
   *   s_hat = (1 - tau_ema) * s_hat + tau_ema * m,   tau = s_hat - tau_offset,
   * where m is the mean over the batch of cos(q_t, q_{t-1}) (the group's
   * concatenated queries at this step and the previous one); the new tau applies
   * from the next step.  Persistent heads stay as chosen.  0 = off (default). */
  int32_t adaptive_tau;
  double tau_ema;          /* weight of the newest step, in (0, 1]; default 1/16 */
  /* storage of the host pool ([KVO] section on quantised offloading: low-bit KV
   * crosses the link and is dequantised on the GPU): 16 (bf16, default; 0 means
   * 16), 4 or 2 bits per value.  Quantisation: per token and per K or V row,
   * groups of 64 channels, each with an fp32 scale = (max - min) / (2^bits - 1) and
   * fp32 min (+0 for a zero minimum); code q = clamp(rint((x - min) / scale), 0, 2^bits - 1) (0 if scale
   * is 0); the GPU sees bf16(fma(q, scale, min)) in the cache slots and resident
   * copies.  Key hash codes come from the keys as appended.  The host pool holds the
   * codes; the groups' (scale, min) pairs stay in HBM (8 bytes per group: 2 d / 64
   * groups per token and kv head).  Host record bytes per token and kv head (the bytes
   * a fetch moves over the link): 4 d (bf16), d (4 bits), d / 2 (2 bits). */
  int32_t kv_bits;
} clo_config;

typedef struct clo_stats_t {
  int64_t steps;             /* decode steps completed */
  int64_t units_hit;         /* cumulative unit decisions */
  int64_t units_miss;
  int64_t units_persist;
  int64_t host_bytes;        /* bytes fetched from the host pool (K and V rows) */
  int64_t hbm_bytes_alg;     /* algorithmic HBM bytes of the decode steps */
  int64_t timeouts;          /* ready-flag waits that gave up */
  int64_t last_hit, last_miss, last_persist, last_host_bytes, last_hbm_bytes_alg;
  int32_t warmup_done;       /* 1 once thresholds and persistent heads are fixed */
  /* timing != 0: CUDA-event times of the two launches of a step (decide = reuse
   * test and query hashing; fused = top-k selection of the missed and persistent
   * units, host-row fetch and sparse attention in one persistent kernel) and of the
   * whole step, for the last step and summed over the timed_steps steps since the
   * previous clo_stats call. */
  int32_t timed_steps;
  float last_ms_decide, last_ms_fused, last_ms_total;
  double sum_ms_decide, sum_ms_fused, sum_ms_total;
} clo_stats_t;

/* Fill *cfg with defaults (shapes zero; topk_ratio 0.1; warmup_steps 16;
 * tau_offset 0.05; wait 2 s; debug_drop_flag_layer -1; adaptive_tau 0, tau_ema 1/16). */
CLO_API void clo_config_default(clo_config* cfg);

/* Create a context: allocates the pinned, device-mapped host K/V pool (on a host with
 * several NUMA nodes, with its pages preferred on the node of the GPU's PCI function)
 * (L*B*Hkv*max_tokens records of K||V, 4*d bytes each, [SYN] 3.4 attack 7 sizes the
 * pool of a 512K Qwen2.5-14B context at 93.75 GB) and the HBM state (hash codes,
 * selections, cache slots, resident copies).  *out receives the context.
 * Errors: CLO_ERR_INVALID (shapes), CLO_ERR_OOM, CLO_ERR_CUDA. */
CLO_API clo_status clo_init(const clo_config* cfg, clo_ctx** out);

/* Release everything the context owns.  NULL is accepted. */
CLO_API clo_status clo_destroy(clo_ctx* ctx);

/* Offload prefill K/V once ([SYN] 5.7: KV is produced at prefill and offloaded):
 * appends n_tokens tokens of (layer, seq) at its current length.
 * k, v: bf16 [n_tokens][Hkv][d], host (src_is_device = 0) or device (1) memory,
 * copied; the caller keeps ownership and may reuse them on return.  Computes the
 * keys' 128-bit hash codes on the GPU (kept in HBM).  Synchronous.
 * Errors: CLO_ERR_INVALID, CLO_ERR_CAPACITY (length would exceed max_tokens),
 * CLO_ERR_CUDA. */
CLO_API clo_status clo_append_kv(clo_ctx* ctx, int32_t layer, int32_t seq, const void* k, const void* v,
                                 int64_t n_tokens, int32_t src_is_device);

/* Streaming growth ([SYN] 5.7: incremental offloading, the cache lookup and transfer
 * engine updated as the KV cache grows): appends one token to every (layer,
 * sequence) at its current length, asynchronously on the context's stream (no host
 * synchronisation): the K|V records go to the host pool (and to the resident copy of
 * persistent heads), the keys' hash codes are computed on the GPU, and each sequence's
 * length N and top-k count k (the same rule as at offload) advance on the device, so
 * the next clo_decode_step selects over N + 1 tokens.  A unit that reuses its
 * selection keeps it as it was.
 * k, v: bf16 [L][B][Hkv][d], device (src_is_device = 1) or host (0) memory; device
 * buffers must stay valid until the stream has consumed them, host buffers are copied.
 * Every layer of every sequence must hold the same number (>= 1) of tokens.
 * Errors: CLO_ERR_INVALID, CLO_ERR_STATE (ragged layers, no K/V, layer-by-layer
 * step in progress), CLO_ERR_CAPACITY (a sequence at max_tokens), CLO_ERR_CUDA. */
CLO_API clo_status clo_append_step(clo_ctx* ctx, const void* k, const void* v, int32_t src_is_device);

/* One decode step over all layers ([ABS]; [SYN] 2.1, 2.2):
 * q: bf16 [L][B][Hq][d]; out: fp32 [L][B][Hq][d].
 * io_on_device = 1: q and out are device pointers; the call only enqueues work on
 *   the context's stream and returns (no host synchronisation between layers or
 *   at the end); device errors surface at the next synchronising call.
 * io_on_device = 0: q and out are host pointers; the call copies q in, runs the
 *   step, copies out back and waits for it, returning device errors directly.
 * Every layer of every sequence must hold the same number of tokens (>= 1).
 * Errors: CLO_ERR_INVALID, CLO_ERR_STATE (no K/V, or ragged layers),
 * CLO_ERR_CUDA, CLO_ERR_TIMEOUT / CLO_ERR_DEVICE (host-buffer mode only). */
CLO_API clo_status clo_decode_step(clo_ctx* ctx, const void* q, float* out, int32_t io_on_device);

/* One layer of a decode step, for callers whose layer l+1 query exists only after
 * layer l's output (a model running layer by layer).  CLO prefetches one layer ahead
 * ([SYN] 5.6); here the rows of every unit's last selection stay in its on-GPU cache
 * slot between steps, so a reused unit needs no transfer at all and a unit that
 * misses needs its new query first.  The call runs the reuse test, selection, fetch
 * and attention of `layer` only, enqueued on the context's stream.
 * q: bf16 [B][Hq][d] of this layer; out: fp32 [B][Hq][d] of this layer; io_on_device
 * as for clo_decode_step.  Layers must come in order 0, 1, ..., L-1; the step (warm-up
 * counting, statistics) completes with layer L-1.  A sequence of clo_decode_layer
 * calls over all layers computes exactly what one clo_decode_step computes.
 * Errors: CLO_ERR_INVALID (null pointer, layer out of range), CLO_ERR_STATE (layer
 * out of order, no K/V, ragged layers), CLO_ERR_CUDA, CLO_ERR_TIMEOUT /
 * CLO_ERR_DEVICE (host-buffer mode only).  clo_decode_step and clo_append_kv return
 * CLO_ERR_STATE while a layer-by-layer step is in progress. */
CLO_API clo_status clo_decode_layer(clo_ctx* ctx, int32_t layer, const void* q, float* out, int32_t io_on_device);

/* Wait for all work of the context and report a latched device error, if any
 * (CLO_ERR_TIMEOUT or CLO_ERR_DEVICE); the latch is cleared once reported. */
CLO_API clo_status clo_sync(clo_ctx* ctx);

/* Counters since clo_init (synchronises; also reports a latched device error
 * after filling *out): the head-wise reuse decisions ([SYN] 2.1 item 2: reuse of
 * the on-GPU selection when adjacent-step queries are similar), the bytes the
 * fetch moved over the host link ([ABS] feature (3): the zero-copy transfer
 * engine) and the algorithmic HBM bytes, per step and cumulative. */
CLO_API clo_status clo_stats(clo_ctx* ctx, clo_stats_t* out);

/* Thread-local text of the last failed call ("" if none). */
CLO_API const char* clo_last_error(void);

/* Debug read-back of internal state (synchronises).  what selects the item;
 * dst is a host buffer of dst_bytes bytes; layer/seq/kvh select the unit where
 * the item is per unit.
 *   CLO_DBG_KEY_CODES   uint64 [N][2] hash codes of the unit's keys
 *   CLO_DBG_QUERY_CODES uint64 [G][2] query codes of the unit's last reselection
 *   CLO_DBG_IDX         int32 [k]     current selection (ascending token index)
 *   CLO_DBG_DECISION    uint8 [L][B][Hkv] decisions of the last step (unit ignored)
 *   CLO_DBG_SLOT_ROWS   bf16 [k][2][d] the unit's on-GPU cache slot (K row, V row)
 *   CLO_DBG_TAU         fp32 [L][Hkv] thresholds (after warm-up)
 *   CLO_DBG_PERSIST     uint8 [L][Hkv] persistent mask
 *   CLO_DBG_SHAT        fp64 [L][Hkv] warm-up mean similarity
 *   CLO_DBG_COS         fp32 [L][B][Hkv] cosines of the last step (NaN if none)
 *   CLO_DBG_TIMELINE    uint64 [16] %globaltimer stamps (ns) of the last step's fused
 *                       kernel, timing mode only (zeros otherwise): [0] start, [1] last
 *                       selection chunk of a missed unit done, [2] last selection chunk
 *                       of a persistent unit done, [3] first fetch chunk able to start,
 *                       [4] last fetch chunk done, [5] first attention split, [6] last
 *                       attention split done, [7] summed fetch waits on selections,
 *                       [8] summed attention waits on fetch flags, [9] summed durations
 *                       of selection chunks, [10] their number, [11] summed durations
 *                       of attention splits, [12] their number, [13] first CTA of
 *                       the step's decide kernel started, [14] its last CTA finished,
 *                       [15] summed durations of attention splits after their waits
 *   CLO_DBG_TOPK        int32 [L][B]  top-k count k of each (layer, sequence) at its
 *                       current length (the rule of clo_config.topk / topk_ratio)
 *   CLO_DBG_STEP_BYTES  uint64 [4096][2] timing mode only: cumulative {host-link bytes,
 *                       algorithmic HBM bytes} since init after step s, at row s % 4096
 *                       (written by the step's last launch; per-step bytes are the
 *                       differences of consecutive rows)
 *   CLO_DBG_POOL_NODE   int32 [1]     NUMA node the pinned pool's pages were placed on
 *                       (-1: not placed: a host with one memory node, or placement failed
 *                       and the pool came from cudaHostAlloc)
 * Errors: CLO_ERR_INVALID (item, unit or size), CLO_ERR_STATE (CLO_DBG_STEP_BYTES without
 * timing mode), CLO_ERR_CUDA. */
enum {
  CLO_DBG_KEY_CODES = 1,
  CLO_DBG_QUERY_CODES = 2,
  CLO_DBG_IDX = 3,
  CLO_DBG_DECISION = 4,
  CLO_DBG_SLOT_ROWS = 5,
  CLO_DBG_TAU = 6,
  CLO_DBG_PERSIST = 7,
  CLO_DBG_SHAT = 8,
  CLO_DBG_COS = 9,
  CLO_DBG_TIMELINE = 10,
  CLO_DBG_TOPK = 11,
  CLO_DBG_POOL_NODE = 12,
  CLO_DBG_STEP_BYTES = 13
};
CLO_API clo_status clo_debug_get(clo_ctx* ctx, int32_t what, int32_t layer, int32_t seq, int32_t kvh, void* dst,
                                 int64_t dst_bytes);

/* Change a setting after init:
 *   CLO_SET_DROP_FLAG_LAYER  fault injection: layer whose fetch never signals, or -1
 *   CLO_SET_WAIT_TIMEOUT_NS  bound of the device-side waits (> 0) */
enum { CLO_SET_DROP_FLAG_LAYER = 1, CLO_SET_WAIT_TIMEOUT_NS = 2 };
CLO_API clo_status clo_set(clo_ctx* ctx, int32_t key, int64_t value);

/* Split-K sparse decode attention that allocates nothing: the attention over a
 * selection of rows the caller provides.  The paper has no counterpart to this
 * call; it is here for callers that are not allowed to
 * allocate device memory themselves or through the library: a serving engine or
 * plugin host that plans every byte of device memory up front and hands kernels
 * only their inputs and outputs, or a latency-critical loop that cannot take the
 * device-wide stalls cudaMalloc/cudaFree may cause.
 *   q:    device bf16 [n_groups][group_size][head_dim]  (one GQA group per row)
 *   rows: device bf16 [n_groups][k][2][head_dim]         (K row then V row of each
 *         selected token, the layout of the library's cache slots); 16-byte aligned
 *   out:  device fp32 [n_groups][group_size][head_dim], written by the call
 *   out_g = sum_r softmax_r(q_g . K_r / sqrt(head_dim)) V_r over the k rows.
 * group_size <= 8, head_dim 64 or 128, k >= 1.  Work is enqueued on stream
 * (cudaStream_t, NULL = legacy default stream) and the call returns at once.
 * Scratch: one fixed array of about 8 MiB in device memory, defined in the
 * library and held by every GPU that loads it until the process exits.  Sizes
 * beyond it are rejected with CLO_ERR_INVALID: n_groups <= 4096 and
 * n_groups * ceil(k / 256) * group_size * (head_dim + 2) <= 2097152.
 * The first call on a device looks up that array's device address (once per
 * device, with that device current) and keeps it for the life of the process;
 * make the first call before any stream capture.  The kept address does not
 * survive cudaDeviceReset() or a rebuilt primary context: do not call this
 * entry point again in a process after either.  All calls share the array: calls whose work overlaps on the GPU race
 * on it, so serialise them (one stream, or events).  No cudaMalloc, cudaFree or
 * other allocating routine is called.  Errors: CLO_ERR_INVALID (null or misaligned
 * pointer, sizes), CLO_ERR_CUDA. */
CLO_API clo_status clo_sparse_attention_noalloc(const void* q, const void* rows, float* out, int32_t n_groups,
                                                int32_t group_size, int32_t head_dim, int64_t k, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* CLO_H_ */
