// Internal declarations shared by the CLO kernels and the host runtime.
//
// Data layout (all per context; unit u = (l * B + b) * Hkv + h):
//   host pool (pinned, device-mapped)  bf16 [U][Nmax][K(d) | V(d)]  record = 4*d bytes
//                                      (quantised: [U][Nmax][K codes | V codes], d*bits/4 bytes)
//   qparams    (HBM, quantised only)   float2 [U][Nmax][2d/64]      (scale, min) per group
//   codes      (HBM)                   uint4 [U][Nmax]               128-bit key codes
//   qcodes     (HBM)                   uint4 [L][B][Hq]              query codes of the step
//   qcache     (HBM)                   bf16 [U][G*d]                 query at the last refresh
//   idx        (HBM)                   int32 [U][kmax]               selection, ascending
//   unit_hist  (HBM)                   uint32 [U][nbp]               score histogram of the step
//   slots      (HBM)                   bf16 [U][kmax][K | V]         on-GPU cache of fetched rows
//   resident   (HBM)                   bf16 [L][B][P][Nmax][K | V]   persistent heads' full K/V
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "clo.h"

namespace clo {

constexpr int kMaxG = 8;
constexpr int kMaxD = 128;
constexpr int64_t kMaxTokens = 524288;

// device error word bits
constexpr uint32_t kErrFlagTimeout = 1u;   // a ready-flag wait gave up
constexpr uint32_t kErrMbarTimeout = 2u;   // a bulk-copy barrier wait gave up
constexpr uint32_t kErrBounds = 4u;        // an internal bounds check failed

// step counters (uint64 slots)
enum Counter : int {
  C_HIT = 0,
  C_MISS = 1,
  C_PERSIST = 2,
  C_HOST_BYTES = 3,
  C_HBM_BYTES = 4,
  C_TIMEOUTS = 5,
  C_NUM = 8
};
// each counter is spread over kCtrLanes addresses (by unit) to keep atomics uncontended
constexpr int kCtrLanes = 32;
__host__ __device__ inline int ctr_at(int counter, int64_t unit) {
  return counter * kCtrLanes + (int)(unit & (kCtrLanes - 1));
}

struct DevState {
  int L, B, Hq, Hkv, d, G;
  int P;                        // resident heads per layer allocated (0 = none)
  int64_t Nmax, kmax;
  const int64_t* ntok;          // [B]
  const int32_t* kcount;        // [B]
  const uint16_t* R;            // [L][Hkv][d][128]
  uint4* codes;                 // [U][Nmax]
  uint4* qcodes;                // [L][B][Hq]
  uint16_t* qcache;             // [U][G*d]
  uint8_t* qvalid;              // [U]
  float* tau;                   // [L*Hkv]
  uint8_t* persist;             // [L*Hkv]
  int32_t* persist_slot;        // [L*Hkv] resident index or -1
  double* shat_sum;             // [L*Hkv]
  double* shat;                 // [L*Hkv]
  uint8_t* decision;            // [U]
  float* cosv;                  // [U]
  int32_t* idx;                 // [U][kmax]
  uint16_t* slots;              // [U][kmax][2d]
  uint16_t* resident;           // [L][B][P][Nmax][2d]
  const uint16_t* pool;         // device view of the host pool [U][Nmax][record]
  float2* qparams;              // quantised pool: [U][Nmax][2d/64] (scale, min) per group (HBM), else null
  unsigned long long* step_ctr; // [C_NUM][kCtrLanes] this step (summed by the host)
  unsigned long long* total_ctr;// [C_NUM][kCtrLanes] since init
  uint32_t* err;                // error word
  uint32_t* unit_done;          // [U] split counters of the attention combine
  float* part;                  // attention partials [U][nsplit][G][d + 2] (one per split)
  int nsplit;                   // attention splits per unit (split_rows rows each)
  int split_rows;               // selected rows per attention split: 256 (small launches), 1024, 2048 (kmax > 8192)
  int decide_rows;              // query rows hashed per decide CTA: 32, or 16 in small launches
  int nchunk;                   // fetch chunks per unit (kChunkRows rows each)
  int fetch_rows;               // rows per fetch item: 256, 128, 64 or 32 (divides kChunkRows)
  uint32_t* ready;              // [U][nchunk] fetch-ready flag per row chunk (zeroed per step)
  int* lcnt;                    // [3L] per-layer list lengths: hit, persistent, missed (zeroed per step)
  int32_t* hit_list;            // [L][B*Hkv] units reusing their selection, per layer
  int32_t* pers_list;           // [L][B*Hkv] persistent units, per layer
  int32_t* miss_list;           // [L][B*Hkv] missed units, per layer
  unsigned* queue;              // [2] work counters: fetch, compute (zeroed per step)
  uint32_t* unit_hist;          // [U][nbp] score histogram of each unit being selected (left zeroed by its last chunk)
  int2* sel_meta;               // [U][nch] {count above T, count at T} of each selection chunk
  uint32_t* score_done;         // [U] chunks whose histogram is merged (zeroed per step)
  uint32_t* cnt_done;           // [U] chunk counts published (zeroed per step)
  uint32_t* sel_cnt;            // [U] chunks compacted (zeroed per step)
  int sel_chunk;                // tokens per selection chunk of a persistent unit
  int nch;                      // selection chunks per persistent unit = ceil(Nmax / sel_chunk)
  int sel_chunk_miss;           // tokens per selection chunk of a missed unit
  int nch_miss;                 // selection chunks per missed unit
  int nbp;                      // histogram bins per chunk, padded (>= 128*G + 1)
  unsigned long long* timeline; // [kTimelineSlots] %globaltimer stamps of the step (timing mode), or null
  int64_t wait_timeout_ns;
  int drop_flag_layer;
  uint16_t* qprev;              // [U][G*d] query of the previous step (adaptive thresholds), or null
  uint8_t* qprev_valid;         // [U]
  double* cos_sum;              // [L*Hkv] sum over the step's units of cos(q_t, q_{t-1})
  uint32_t* cos_cnt;            // [L*Hkv] number of terms in cos_sum
  int adapt_active;             // this launch updates s_hat and tau from cos_sum
  double tau_ema;               // weight of the newest step in the s_hat average
  float tau_offset;             // tau = s_hat - tau_offset
  int kv_bits;                  // host pool storage: 16 (bf16), 4 or 2
  int rec_bytes;                // bytes of one token's K|V record in the host pool
  unsigned long long* step_bytes; // [kStepHist][2] cumulative {host, HBM} bytes after each step (timing mode), or null
  int64_t step_index;           // the step this launch belongs to
  int l0, l1;                   // layers of this launch: [l0, l1)
  int q_l0;                     // layer of the first [B][Hq][d] block of the q / out buffers
};

constexpr int kMaxLayers = 256;
constexpr int kStepHist = 4096;  // steps kept by the per-step byte history (a ring)

// timeline slots of the fused step kernel (ns of %globaltimer; first = first writer)
enum Timeline : int {
  TL_START = 0,          // first CTA started
  TL_SEL_MISS_END = 1,   // last selection chunk of a missed unit finished
  TL_SEL_PERS_END = 2,   // last selection chunk of a persistent unit finished
  TL_FETCH_FIRST = 3,    // first fetch chunk could start copying
  TL_FETCH_END = 4,      // last fetch chunk released
  TL_ATT_FIRST = 5,      // first attention split started
  TL_COMP_END = 6,       // last attention split finished
  TL_FETCH_WAIT_NS = 7,  // summed waits of fetch warps on selections
  TL_ATT_WAIT_NS = 8,    // summed waits of attention groups on fetch flags
  TL_SEL_SUM_NS = 9,     // summed durations of selection chunks
  TL_SEL_ITEMS = 10,     // selection chunks run
  TL_ATT_SUM_NS = 11,    // summed durations of attention splits (waits included)
  TL_ATT_ITEMS = 12,     // attention splits run
  TL_DEC_START = 13,     // a CTA of the decide kernel started (first writer)
  TL_DEC_END = 14,       // last CTA of the decide kernel finished
  TL_ATT_RUN_NS = 15,    // summed durations of attention splits after their waits
  kTimelineSlots = 16
};
constexpr int kSelChunkMax = 16384;  // tokens per selection chunk, at most
constexpr int kSelChunkMin = 1024;   // tokens per selection chunk, at least
constexpr int kChunkRows = 256;   // selected rows per fetch chunk (one ready flag each)
constexpr int kNBPad = 1056;     // >= 128 * kMaxG + 1, multiple of 32

__host__ __device__ inline int64_t unit_of(const DevState& s, int l, int b, int h) {
  return ((int64_t)l * s.B + b) * s.Hkv + h;
}

// ---------------------------------------------------------------------------- PTX helpers
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase; on timeout sets kErrMbarTimeout and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t* err,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) {
      atomicOr(err, kErrMbarTimeout);
      return false;
    }
  }
}

// 1-D bulk copy global -> shared (TMA engine), completion counted on an mbarrier.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before later
// async-proxy (bulk copy) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add_u32(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint4 ld_nc_v4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Asks the memory system to bring [p, p + bytes) into L2 (no destination, no completion
// to wait for); p 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ---- quantised host records ---------------------------------------------------------------
// Record of one token and kv head in the host pool: [K codes | V codes]; value i of a row
// sits in 32-bit word i / (32 / BITS) at bit BITS * (i % (32 / BITS)).  One 16-byte code
// vector holds 128 / BITS values of one 64-channel group.  The groups' (scale, min) pairs
// stay in HBM (DevState::qparams, K groups then V groups per token), so a record is a
// whole number of 64-byte lines (d = 128: 128 bytes at 4 bits, 64 at 2 bits): records of
// other sizes moved 10-15 % fewer useful bytes per second over the host link.
template <int D, int BITS>
struct QRec {
  static constexpr int kCodeVecs = 2 * D * BITS / 128;  // 16-byte code vectors per record
  static constexpr int kVecsPerGroup = BITS / 2;          // 64 values per group
  static constexpr int kOutVecs = 16 / BITS;              // bf16 uint4 per code vector
  static constexpr int kBytes = kCodeVecs * 16;
  static constexpr int kGroups = 2 * D / 64;              // (scale, min) pairs per token
};

// Dequantises one 16-byte code vector: value = bf16(fma(q, scale, mn)).
template <int BITS>
__device__ __forceinline__ void dequant_vec(const uint4 p, float scale, float mn, uint4* out) {
  constexpr int PER = 32 / BITS;
  constexpr uint32_t MASK = (1u << BITS) - 1u;
  const uint32_t w[4] = {p.x, p.y, p.z, p.w};
  uint32_t o[2 * PER];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < PER; j += 2) {
      const float a = fmaf((float)((w[i] >> (BITS * j)) & MASK), scale, mn);
      const float b = fmaf((float)((w[i] >> (BITS * (j + 1))) & MASK), scale, mn);
      const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(a));
      const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(b));
      o[(i * PER + j) / 2] = lo | (hi << 16);
    }
#pragma unroll
  for (int v = 0; v < PER / 2; ++v) out[v] = make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ---------------------------------------------------------------------------- launchers
// (each returns the launch's cudaError_t)
cudaError_t launch_hash_keys(const DevState& s, int l, int b, int64_t t0, int64_t n, const uint16_t* kdev,
                             cudaStream_t st);
cudaError_t launch_decide(const DevState& s, const uint16_t* q, int64_t step, int warmup_active, cudaStream_t st);
cudaError_t launch_finish_warmup(const DevState& s, int W, float tau_offset, int n_persist, cudaStream_t st);
cudaError_t launch_step_fused(const DevState& s, const uint16_t* q, float* out, cudaStream_t st);
cudaError_t launch_resident_fill(const DevState& s, int64_t t0, int64_t t1, cudaStream_t st);
cudaError_t launch_pool_write(const DevState& s, int l, int b, int64_t t0, int64_t n, const uint16_t* kdev,
                              const uint16_t* vdev, cudaStream_t st);
cudaError_t launch_append_step(const DevState& s, const uint16_t* kdev, const uint16_t* vdev, int64_t topk,
                               double ratio, cudaStream_t st);


}  // namespace clo

namespace clo {
// Sets the thread-local text returned by clo_last_error().
void set_last_error_text(const char* msg);
}  // namespace clo
