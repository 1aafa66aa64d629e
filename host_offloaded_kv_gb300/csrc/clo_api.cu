// Host runtime of the CLO decode-step library: the C ABI declared in clo.h.
//
// One context owns a pinned, device-mapped host pool holding every sequence's
// full K/V (CLO keeps the whole KV cache in CPU memory: CLO abstract) and the HBM
// state of the decode step.  clo_decode_step() only enqueues kernels on the
// context's stream; no host synchronisation happens between layers or phases
// (GPU-centric synchronisation: CLO abstract, feature (3)).
#include <cuda_runtime.h>
#include <sys/mman.h>
#include <sys/syscall.h>
#include <unistd.h>

#include <algorithm>
#include <array>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "clo.h"
#include "clo_internal.cuh"

using namespace clo;

namespace {

thread_local std::string g_last_error;

clo_status fail(clo_status st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

#define CLO_CUDA(expr)                                                                         \
  do {                                                                                         \
    cudaError_t e_ = (expr);                                                                   \
    if (e_ != cudaSuccess) return fail(CLO_ERR_CUDA, std::string(#expr) + ": " + cudaGetErrorString(e_)); \
  } while (0)

constexpr int64_t kStageTokens = 16384;

int64_t topk_for(int64_t N, int64_t topk, double ratio) {
  if (N <= 0) return 0;
  if (topk > 0) return std::min<int64_t>(topk, N);
  int64_t k = (int64_t)std::ceil(ratio * (double)N);
  return std::max<int64_t>(1, std::min<int64_t>(k, N));
}


// ---- placement of the pinned pool ----------------------------------------------------
// On a host with several NUMA nodes the pool's pages belong on the node nearest the
// GPU (the node of its PCI function), so that the fetch's loads do not cross the
// inter-socket link.  The pool is then an anonymous mapping whose pages are preferred
// on that node, registered with CUDA as mapped, portable pinned memory; on a host with
// one memory node (or if any step fails) it is plain cudaHostAlloc memory.

// NUMA node of the device's PCI function, or -1 when unknown.
int device_numa_node(int dev) {
  char bus[64] = {0};
  if (cudaDeviceGetPCIBusId(bus, (int)sizeof(bus), dev) != cudaSuccess) return -1;
  unsigned dom = 0, b = 0, d = 0, f = 0;
  if (sscanf(bus, "%x:%x:%x.%x", &dom, &b, &d, &f) != 4) return -1;
  char path[128];
  snprintf(path, sizeof(path), "/sys/bus/pci/devices/%04x:%02x:%02x.%x/numa_node", dom, b, d, f);
  FILE* fp = fopen(path, "r");
  if (!fp) return -1;
  int node = -1;
  if (fscanf(fp, "%d", &node) != 1) node = -1;
  fclose(fp);
  return node;
}

// Number of NUMA nodes that hold memory (sysfs "has_memory" list, e.g. "0-1" or "0,2").
int memory_node_count() {
  FILE* fp = fopen("/sys/devices/system/node/has_memory", "r");
  if (!fp) return 1;
  char buf[256] = {0};
  const size_t n = fread(buf, 1, sizeof(buf) - 1, fp);
  fclose(fp);
  buf[n] = 0;
  int count = 0;
  for (char* t = buf; *t;) {
    char* end = nullptr;
    const long a = strtol(t, &end, 10);
    if (end == t) break;
    long bnd = a;
    if (*end == '-') {
      char* e2 = nullptr;
      bnd = strtol(end + 1, &e2, 10);
      end = e2;
    }
    count += (int)(bnd - a + 1);
    t = end;
    while (*t == ',' || *t == '\n' || *t == ' ') ++t;
  }
  return count > 0 ? count : 1;
}

// Pinned, device-mapped pool of `bytes` bytes with pages preferred on `node`; nullptr if
// any step fails (nothing is left allocated then).
void* alloc_pool_on_node(size_t bytes, int node) {
  void* p = mmap(nullptr, bytes, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
  if (p == MAP_FAILED) return nullptr;
  unsigned long mask[16] = {0};
  if (node < 0 || node >= (int)(sizeof(mask) * 8)) {
    munmap(p, bytes);
    return nullptr;
  }
  mask[node / 64] = 1ul << (node % 64);
  constexpr int kMpolPreferred = 1;  // MPOL_PREFERRED: that node first, others when it is full
  if (syscall(SYS_mbind, p, bytes, kMpolPreferred, mask, (unsigned long)(sizeof(mask) * 8), 0u) != 0) {
    munmap(p, bytes);
    return nullptr;
  }
  madvise(p, bytes, MADV_HUGEPAGE);  // a hint; large pages are not required
  if (cudaHostRegister(p, bytes, cudaHostRegisterMapped | cudaHostRegisterPortable) != cudaSuccess) {
    cudaGetLastError();
    munmap(p, bytes);
    return nullptr;
  }
  return p;
}
}  // namespace

struct clo_ctx {
  clo_config cfg{};
  int L = 0, B = 0, Hq = 0, Hkv = 0, d = 0, G = 0, P = 0;
  int64_t Nmax = 0, kmax = 0, U = 0;
  cudaStream_t stream = nullptr;
  uint16_t* pool_host = nullptr;
  size_t pool_bytes = 0;
  bool pool_registered = false;  // anonymous mapping registered with CUDA (else cudaHostAlloc)
  int pool_node = -1;            // NUMA node the pool's pages prefer (-1: not placed)
  DevState ds{};
  std::vector<void*> dev_allocs;
  std::vector<int64_t> ntok;  // [L*B] tokens appended per (layer, seq)
  bool ntok_dirty = true;
  int64_t* ntok_pinned = nullptr;  // [B] + k [B] staging for uploads
  int64_t step = 0;
  bool warmup_mode = false;
  int kv_bits = 16;
  int sms = 0;                   // multiprocessors of the device
  int whole_unit_min_units = 0;  // launches with at least this many units select persistent units whole
  uint16_t* kstep = nullptr;     // staging of clo_append_step's host rows
  uint16_t* vstep = nullptr;
  int next_layer = 0;  // next layer of a layer-by-layer step (0: none in progress)
  int W = 0;
  bool warmup_done = false;
  uint16_t* kstage = nullptr;
  uint16_t* vstage = nullptr;
  uint16_t* q_io = nullptr;
  float* out_io = nullptr;
  // per-step phase events (timing mode): 4 markers per step, reused after clo_stats
  std::vector<std::array<cudaEvent_t, 3>> ev_pool;
  size_t ev_used = 0;
  uint32_t epoch = 0;
  uint32_t* step_zero = nullptr;  // zeroed at the start of every step
  size_t step_zero_bytes = 0;
  unsigned long long* timeline_dev = nullptr;  // inside step_zero
  std::vector<uint8_t> persist_host;  // valid once known
  bool persist_host_valid = false;

  template <class T>
  clo_status dalloc(T** p, size_t count) {
    void* v = nullptr;
    const size_t bytes = std::max<size_t>(count * sizeof(T), 16);
    cudaError_t e = cudaMalloc(&v, bytes);
    if (e != cudaSuccess) return fail(CLO_ERR_OOM, "cudaMalloc(" + std::to_string(bytes) + "): " + cudaGetErrorString(e));
    dev_allocs.push_back(v);
    e = cudaMemset(v, 0, bytes);
    if (e != cudaSuccess) return fail(CLO_ERR_CUDA, std::string("cudaMemset: ") + cudaGetErrorString(e));
    *p = static_cast<T*>(v);
    return CLO_OK;
  }

  void release() {
    if (stream) cudaStreamSynchronize(stream);
    for (void* p : dev_allocs) cudaFree(p);
    dev_allocs.clear();
    if (pool_host) {
      if (pool_registered) {
        cudaHostUnregister(pool_host);
        munmap(pool_host, pool_bytes);
      } else {
        cudaFreeHost(pool_host);
      }
    }
    pool_host = nullptr;
    if (ntok_pinned) cudaFreeHost(ntok_pinned);
    ntok_pinned = nullptr;
    for (auto& set : ev_pool)
      for (auto& e : set) cudaEventDestroy(e);
    ev_pool.clear();
  }
};

#define CLO_TRY(expr)                 \
  do {                                \
    clo_status s_ = (expr);           \
    if (s_ != CLO_OK) return s_;      \
  } while (0)

extern "C" {

CLO_API void clo_config_default(clo_config* cfg) {
  if (!cfg) return;
  std::memset(cfg, 0, sizeof(*cfg));
  cfg->topk_ratio = 0.1;
  cfg->warmup_steps = 16;
  cfg->tau_offset = 0.05f;
  cfg->wait_timeout_ns = 2000000000LL;
  cfg->debug_drop_flag_layer = -1;
  cfg->tau_ema = 0.0625;
}

CLO_API const char* clo_last_error(void) { return g_last_error.c_str(); }

static clo_status init_impl(const clo_config* cfg, clo_ctx* c) {
  c->cfg = *cfg;
  c->L = cfg->n_layers;
  c->B = cfg->batch;
  c->Hq = cfg->n_q_heads;
  c->Hkv = cfg->n_kv_heads;
  c->d = cfg->head_dim;
  if (c->L < 1 || c->B < 1 || c->Hkv < 1 || c->Hq < 1 || c->Hq % c->Hkv != 0)
    return fail(CLO_ERR_INVALID, "shapes: need L, B, Hkv >= 1 and Hq a multiple of Hkv");
  c->G = c->Hq / c->Hkv;
  if (c->G > kMaxG) return fail(CLO_ERR_INVALID, "GQA group Hq/Hkv must be <= 8");
  if (c->d != 64 && c->d != 128) return fail(CLO_ERR_INVALID, "head_dim must be 64 or 128");
  if (cfg->max_tokens < 1 || cfg->max_tokens > kMaxTokens)
    return fail(CLO_ERR_INVALID, "max_tokens must be in [1, 524288]");
  if (!cfg->hash_R) return fail(CLO_ERR_INVALID, "hash_R (bf16 [L][Hkv][d][128]) is required");
  if (cfg->topk < 0) return fail(CLO_ERR_INVALID, "topk must be >= 0");
  if (cfg->topk == 0 && !(cfg->topk_ratio > 0.0 && cfg->topk_ratio <= 1.0))
    return fail(CLO_ERR_INVALID, "topk_ratio must be in (0, 1] when topk == 0");
  c->kv_bits = cfg->kv_bits == 0 ? 16 : cfg->kv_bits;
  if (c->kv_bits != 16 && c->kv_bits != 4 && c->kv_bits != 2)
    return fail(CLO_ERR_INVALID, "kv_bits must be 16, 4 or 2");
  if (cfg->adaptive_tau && !(cfg->tau_ema > 0.0 && cfg->tau_ema <= 1.0))
    return fail(CLO_ERR_INVALID, "tau_ema must be in (0, 1] with adaptive_tau");
  c->warmup_mode = cfg->tau == nullptr;
  if (c->warmup_mode) {
    if (cfg->warmup_steps < 2) return fail(CLO_ERR_INVALID, "warmup_steps must be >= 2 when tau is NULL");
    if (cfg->n_persist < 0 || cfg->n_persist >= c->Hkv)
      return fail(CLO_ERR_INVALID, "n_persist must be in [0, n_kv_heads)");
    if (cfg->persist_mask) return fail(CLO_ERR_INVALID, "persist_mask is only used with fixed tau");
    c->W = cfg->warmup_steps;
    c->P = cfg->n_persist;
  } else {
    int pmax = 0;
    if (cfg->persist_mask) {
      for (int l = 0; l < c->L; ++l) {
        int n = 0;
        for (int h = 0; h < c->Hkv; ++h) n += cfg->persist_mask[l * c->Hkv + h] ? 1 : 0;
        pmax = std::max(pmax, n);
      }
    }
    c->P = pmax;
    c->warmup_done = true;
  }
  c->Nmax = cfg->max_tokens;
  c->kmax = topk_for(c->Nmax, cfg->topk, cfg->topk_ratio);
  c->U = (int64_t)c->L * c->B * c->Hkv;
  c->stream = static_cast<cudaStream_t>(cfg->stream);
  c->ntok.assign((size_t)c->L * c->B, 0);

  int dev = 0;
  CLO_CUDA(cudaGetDevice(&dev));
  int can_map = 0;
  CLO_CUDA(cudaDeviceGetAttribute(&can_map, cudaDevAttrCanMapHostMemory, dev));
  if (!can_map) return fail(CLO_ERR_CUDA, "device cannot map host memory");

  // pinned, device-mapped host pool: [U][Nmax][K|V record]
  // a quantised record holds the codes only; the groups' (scale, min) pairs live in HBM
  const size_t rec = c->kv_bits == 16 ? (size_t)4 * c->d : (size_t)2 * c->d * c->kv_bits / 8;
  const size_t pool_bytes = (size_t)c->U * (size_t)c->Nmax * rec;
  void* hp = nullptr;
  c->pool_bytes = pool_bytes;
  if (memory_node_count() > 1) {  // several memory nodes: the pool's pages near the GPU
    const int node = device_numa_node(dev);
    if (node >= 0 && (hp = alloc_pool_on_node(pool_bytes, node)) != nullptr) {
      c->pool_registered = true;
      c->pool_node = node;
    }
  }
  if (!hp) {
    cudaError_t e = cudaHostAlloc(&hp, pool_bytes, cudaHostAllocMapped | cudaHostAllocPortable);
    if (e != cudaSuccess)
      return fail(CLO_ERR_OOM, "cudaHostAlloc(" + std::to_string(pool_bytes) + " B pinned pool): " +
                                   cudaGetErrorString(e));
  }
  c->pool_host = static_cast<uint16_t*>(hp);
  void* pd = nullptr;
  CLO_CUDA(cudaHostGetDevicePointer(&pd, hp, 0));
  CLO_CUDA(cudaHostAlloc((void**)&c->ntok_pinned, sizeof(int64_t) * 2 * c->B, cudaHostAllocDefault));

  DevState& s = c->ds;
  s.L = c->L;
  s.B = c->B;
  s.Hq = c->Hq;
  s.Hkv = c->Hkv;
  s.d = c->d;
  s.G = c->G;
  s.P = c->P;
  s.Nmax = c->Nmax;
  s.kmax = c->kmax;
  s.pool = static_cast<const uint16_t*>(pd);
  s.kv_bits = c->kv_bits;
  s.rec_bytes = (int)rec;
  s.wait_timeout_ns = cfg->wait_timeout_ns > 0 ? cfg->wait_timeout_ns : 2000000000LL;
  s.drop_flag_layer = cfg->debug_drop_flag_layer;
  // attention partials for the smallest split (256 rows, see enqueue_layers)
  s.split_rows = 256;
  s.nsplit = (int)((c->kmax + s.split_rows - 1) / s.split_rows);
  s.nchunk = (int)((c->kmax + kChunkRows - 1) / kChunkRows);
  s.fetch_rows = kChunkRows;
  const int64_t U = c->U;
  const int LH = c->L * c->Hkv;
  int64_t* ntok_d = nullptr;
  int32_t* kcount_d = nullptr;
  uint16_t* R_d = nullptr;
  CLO_TRY(c->dalloc(&ntok_d, c->B));
  CLO_TRY(c->dalloc(&kcount_d, c->B));
  s.ntok = ntok_d;
  s.kcount = kcount_d;
  CLO_TRY(c->dalloc(&R_d, (size_t)LH * c->d * 128));
  CLO_CUDA(cudaMemcpy(R_d, cfg->hash_R, sizeof(uint16_t) * (size_t)LH * c->d * 128, cudaMemcpyHostToDevice));
  s.R = R_d;
  CLO_TRY(c->dalloc(&s.codes, (size_t)U * c->Nmax));
  CLO_TRY(c->dalloc(&s.qcodes, (size_t)c->L * c->B * c->Hq));
  CLO_TRY(c->dalloc(&s.qcache, (size_t)U * c->G * c->d));
  CLO_TRY(c->dalloc(&s.qvalid, (size_t)U));
  CLO_TRY(c->dalloc(&s.tau, (size_t)LH));
  CLO_TRY(c->dalloc(&s.persist, (size_t)LH));
  CLO_TRY(c->dalloc(&s.persist_slot, (size_t)LH));
  CLO_TRY(c->dalloc(&s.shat_sum, (size_t)LH));
  CLO_TRY(c->dalloc(&s.shat, (size_t)LH));
  CLO_TRY(c->dalloc(&s.decision, (size_t)U));
  CLO_TRY(c->dalloc(&s.cosv, (size_t)U));
  CLO_TRY(c->dalloc(&s.idx, (size_t)U * c->kmax));
  CLO_TRY(c->dalloc(&s.slots, (size_t)U * c->kmax * 2 * c->d));
  if (c->kv_bits != 16) {
    CLO_TRY(c->dalloc(&s.qparams, (size_t)U * c->Nmax * (2 * c->d / 64)));
  } else {
    s.qparams = nullptr;
  }
  if (c->P > 0) {
    CLO_TRY(c->dalloc(&s.resident, (size_t)c->L * c->B * c->P * c->Nmax * 2 * c->d));
  } else {
    s.resident = nullptr;
  }
  // per-step zeroed region: step counters, per-layer list lengths, work queues, ready
  // flags of the fetch chunks, selection progress counters
  // selection in chunks of 8192 (contexts up to 32K) or 16384 tokens (refined per launch)
  s.sel_chunk = c->Nmax <= 32768 ? 8192 : kSelChunkMax;
  s.nch = (int)((c->Nmax + s.sel_chunk - 1) / s.sel_chunk);
  s.sel_chunk_miss = c->Nmax <= 32768 ? 8192 : kSelChunkMax;
  s.nch_miss = (int)((c->Nmax + s.sel_chunk_miss - 1) / s.sel_chunk_miss);
  {  // launches with few units use smaller chunks and fetch items (see enqueue_layers)
    int sms = 0;
    CLO_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    c->sms = sms;
    c->whole_unit_min_units = 4 * sms;
  }
  const int nch_max = (int)((c->Nmax + kSelChunkMin - 1) / kSelChunkMin);
  s.nbp = (128 * c->G + 1 + 31) / 32 * 32;
  {
    size_t off = 2 * (size_t)C_NUM * kCtrLanes;
    const size_t o_lcnt = off;
    off += 3 * (size_t)c->L;
    const size_t o_queue = off;
    off += 4;
    const size_t o_ready = off;
    off += (size_t)U * s.nchunk;
    const size_t o_sel = off;
    off += 4 * (size_t)U;
    off = (off + 1) / 2 * 2;  // 8-byte alignment for the timeline
    const size_t o_tl = off;
    off += 2 * (size_t)kTimelineSlots;
    uint32_t* z = nullptr;
    CLO_TRY(c->dalloc(&z, off));
    c->step_zero = z;
    c->step_zero_bytes = off * sizeof(uint32_t);
    s.step_ctr = reinterpret_cast<unsigned long long*>(z);
    s.lcnt = reinterpret_cast<int*>(z + o_lcnt);
    s.queue = z + o_queue;
    s.ready = z + o_ready;
    s.score_done = z + o_sel;
    s.cnt_done = z + o_sel + 2 * U;
    s.sel_cnt = z + o_sel + 3 * U;
    c->timeline_dev = reinterpret_cast<unsigned long long*>(z + o_tl);
    s.timeline = cfg->timing ? c->timeline_dev : nullptr;
  }
  if (cfg->timing) {
    CLO_TRY(c->dalloc(&s.step_bytes, (size_t)kStepHist * 2));
  } else {
    s.step_bytes = nullptr;
  }
  CLO_TRY(c->dalloc(&s.hit_list, (size_t)c->L * c->B * c->Hkv));
  CLO_TRY(c->dalloc(&s.pers_list, (size_t)c->L * c->B * c->Hkv));
  CLO_TRY(c->dalloc(&s.miss_list, (size_t)c->L * c->B * c->Hkv));
  CLO_TRY(c->dalloc(&s.unit_hist, (size_t)U * s.nbp));
  s.tau_ema = cfg->tau_ema;
  s.tau_offset = cfg->tau_offset;
  if (cfg->adaptive_tau) {
    CLO_TRY(c->dalloc(&s.qprev, (size_t)U * c->G * c->d));
    CLO_TRY(c->dalloc(&s.qprev_valid, (size_t)U));
    CLO_TRY(c->dalloc(&s.cos_sum, (size_t)LH));
    CLO_TRY(c->dalloc(&s.cos_cnt, (size_t)LH));
  } else {
    s.qprev = nullptr;
    s.qprev_valid = nullptr;
    s.cos_sum = nullptr;
    s.cos_cnt = nullptr;
  }
  CLO_TRY(c->dalloc(&s.sel_meta, (size_t)U * nch_max));
  CLO_TRY(c->dalloc(&s.total_ctr, (size_t)C_NUM * kCtrLanes));
  CLO_TRY(c->dalloc(&s.err, 1));
  CLO_TRY(c->dalloc(&s.unit_done, (size_t)U));
  CLO_TRY(c->dalloc(&s.part, (size_t)U * s.nsplit * c->G * (c->d + 2)));

  std::vector<int32_t> pslot((size_t)LH, -1);
  std::vector<uint8_t> pm((size_t)LH, 0);
  if (!c->warmup_mode) {
    CLO_CUDA(cudaMemcpy(s.tau, cfg->tau, sizeof(float) * LH, cudaMemcpyHostToDevice));
    if (cfg->adaptive_tau) {  // the running average starts from the given thresholds
      std::vector<double> sh((size_t)LH);
      for (int i = 0; i < LH; ++i) sh[(size_t)i] = (double)cfg->tau[i] + (double)cfg->tau_offset;
      CLO_CUDA(cudaMemcpy(s.shat, sh.data(), sizeof(double) * LH, cudaMemcpyHostToDevice));
    }
    if (cfg->persist_mask) {
      for (int l = 0; l < c->L; ++l) {
        int p = 0;
        for (int h = 0; h < c->Hkv; ++h)
          if (cfg->persist_mask[l * c->Hkv + h]) {
            pm[(size_t)l * c->Hkv + h] = 1;
            pslot[(size_t)l * c->Hkv + h] = p++;
          }
      }
    }
    c->persist_host = pm;
    c->persist_host_valid = true;
  }
  CLO_CUDA(cudaMemcpy(s.persist, pm.data(), LH, cudaMemcpyHostToDevice));
  CLO_CUDA(cudaMemcpy(s.persist_slot, pslot.data(), sizeof(int32_t) * LH, cudaMemcpyHostToDevice));

  CLO_TRY(c->dalloc(&c->kstage, (size_t)kStageTokens * c->Hkv * c->d));
  CLO_TRY(c->dalloc(&c->vstage, (size_t)kStageTokens * c->Hkv * c->d));
  return CLO_OK;
}

CLO_API clo_status clo_init(const clo_config* cfg, clo_ctx** out) {
  if (!cfg || !out) return fail(CLO_ERR_INVALID, "null argument");
  *out = nullptr;
  clo_ctx* c = new (std::nothrow) clo_ctx();
  if (!c) return fail(CLO_ERR_OOM, "context allocation");
  clo_status st = init_impl(cfg, c);
  if (st != CLO_OK) {
    const std::string msg = g_last_error;
    c->release();
    delete c;
    g_last_error = msg;
    return st;
  }
  *out = c;
  return CLO_OK;
}

CLO_API clo_status clo_destroy(clo_ctx* ctx) {
  if (!ctx) return CLO_OK;
  ctx->release();
  delete ctx;
  return CLO_OK;
}

static clo_status read_device_error(clo_ctx* c) {
  uint32_t err = 0;
  CLO_CUDA(cudaMemcpy(&err, c->ds.err, sizeof(err), cudaMemcpyDeviceToHost));
  if (err == 0) return CLO_OK;
  CLO_CUDA(cudaMemset(c->ds.err, 0, sizeof(uint32_t)));
  if (err & kErrFlagTimeout) return fail(CLO_ERR_TIMEOUT, "a ready-flag wait gave up (fetch never signalled)");
  if (err & kErrMbarTimeout) return fail(CLO_ERR_TIMEOUT, "a bulk-copy barrier wait gave up");
  return fail(CLO_ERR_DEVICE, "device-side bounds check failed (error word " + std::to_string(err) + ")");
}

CLO_API clo_status clo_sync(clo_ctx* c) {
  if (!c) return fail(CLO_ERR_INVALID, "null context");
  CLO_CUDA(cudaStreamSynchronize(c->stream));
  return read_device_error(c);
}

CLO_API clo_status clo_append_kv(clo_ctx* c, int32_t layer, int32_t seq, const void* k, const void* v,
                                 int64_t n_tokens, int32_t src_is_device) {
  if (!c) return fail(CLO_ERR_INVALID, "null context");
  if (layer < 0 || layer >= c->L || seq < 0 || seq >= c->B) return fail(CLO_ERR_INVALID, "layer/seq out of range");
  if (n_tokens < 0 || (n_tokens > 0 && (!k || !v))) return fail(CLO_ERR_INVALID, "bad k/v/n_tokens");
  if (c->next_layer != 0) return fail(CLO_ERR_STATE, "a layer-by-layer step is in progress");
  int64_t& cur = c->ntok[(size_t)layer * c->B + seq];
  if (cur + n_tokens > c->Nmax)
    return fail(CLO_ERR_CAPACITY, "append of " + std::to_string(n_tokens) + " tokens exceeds max_tokens " +
                                      std::to_string(c->Nmax) + " (current " + std::to_string(cur) + ")");
  if (n_tokens == 0) return CLO_OK;
  const size_t row = (size_t)c->Hkv * c->d;  // elements per token
  for (int64_t t = 0; t < n_tokens; t += kStageTokens) {
    const int64_t n = std::min<int64_t>(kStageTokens, n_tokens - t);
    const uint16_t* ks = static_cast<const uint16_t*>(k) + (size_t)t * row;
    const uint16_t* vs = static_cast<const uint16_t*>(v) + (size_t)t * row;
    const uint16_t *kd = ks, *vd = vs;
    if (!src_is_device) {
      CLO_CUDA(cudaMemcpyAsync(c->kstage, ks, sizeof(uint16_t) * n * row, cudaMemcpyHostToDevice, c->stream));
      CLO_CUDA(cudaMemcpyAsync(c->vstage, vs, sizeof(uint16_t) * n * row, cudaMemcpyHostToDevice, c->stream));
      kd = c->kstage;
      vd = c->vstage;
    }
    CLO_CUDA(launch_pool_write(c->ds, layer, seq, cur + t, n, kd, vd, c->stream));
    CLO_CUDA(launch_hash_keys(c->ds, layer, seq, cur + t, n, kd, c->stream));
    if (!src_is_device) CLO_CUDA(cudaStreamSynchronize(c->stream));  // staging is reused
  }
  CLO_CUDA(cudaStreamSynchronize(c->stream));
  cur += n_tokens;
  c->ntok_dirty = true;
  return read_device_error(c);
}

static clo_status refresh_lengths(clo_ctx* c);

CLO_API clo_status clo_append_step(clo_ctx* c, const void* k, const void* v, int32_t src_is_device) {
  if (!c) return fail(CLO_ERR_INVALID, "null context");
  if (!k || !v) return fail(CLO_ERR_INVALID, "null k/v");
  if (c->next_layer != 0) return fail(CLO_ERR_STATE, "a layer-by-layer step is in progress");
  for (int b = 0; b < c->B; ++b) {
    const int64_t n0 = c->ntok[b];
    for (int l = 1; l < c->L; ++l)
      if (c->ntok[(size_t)l * c->B + b] != n0)
        return fail(CLO_ERR_STATE, "sequence " + std::to_string(b) + " has layers of different lengths");
    if (n0 < 1) return fail(CLO_ERR_STATE, "sequence " + std::to_string(b) + " has no K/V appended");
    if (n0 + 1 > c->Nmax)
      return fail(CLO_ERR_CAPACITY, "sequence " + std::to_string(b) + " is at max_tokens " + std::to_string(c->Nmax));
  }
  if (c->ntok_dirty) CLO_TRY(refresh_lengths(c));  // the device lengths are the current ones
  const size_t n = (size_t)c->L * c->B * c->Hkv * c->d;
  const uint16_t* kd = static_cast<const uint16_t*>(k);
  const uint16_t* vd = static_cast<const uint16_t*>(v);
  if (!src_is_device) {
    if (!c->kstep) {
      CLO_TRY(c->dalloc(&c->kstep, n));
      CLO_TRY(c->dalloc(&c->vstep, n));
    }
    CLO_CUDA(cudaMemcpyAsync(c->kstep, k, sizeof(uint16_t) * n, cudaMemcpyHostToDevice, c->stream));
    CLO_CUDA(cudaMemcpyAsync(c->vstep, v, sizeof(uint16_t) * n, cudaMemcpyHostToDevice, c->stream));
    kd = c->kstep;
    vd = c->vstep;
  }
  CLO_CUDA(launch_append_step(c->ds, kd, vd, c->cfg.topk, c->cfg.topk_ratio, c->stream));
  for (auto& x : c->ntok) x += 1;  // the device lengths advance in the same stream
  return CLO_OK;
}

static clo_status refresh_lengths(clo_ctx* c) {
  for (int b = 0; b < c->B; ++b) {
    const int64_t n0 = c->ntok[b];
    for (int l = 1; l < c->L; ++l)
      if (c->ntok[(size_t)l * c->B + b] != n0)
        return fail(CLO_ERR_STATE, "sequence " + std::to_string(b) + " has layers of different lengths");
    if (n0 < 1) return fail(CLO_ERR_STATE, "sequence " + std::to_string(b) + " has no K/V appended");
    c->ntok_pinned[b] = n0;
  }
  int32_t* kc = reinterpret_cast<int32_t*>(c->ntok_pinned + c->B);
  for (int b = 0; b < c->B; ++b) kc[b] = (int32_t)topk_for(c->ntok[b], c->cfg.topk, c->cfg.topk_ratio);
  CLO_CUDA(cudaMemcpyAsync(const_cast<int64_t*>(c->ds.ntok), c->ntok_pinned, sizeof(int64_t) * c->B,
                           cudaMemcpyHostToDevice, c->stream));
  CLO_CUDA(cudaMemcpyAsync(const_cast<int32_t*>(c->ds.kcount), kc, sizeof(int32_t) * c->B, cudaMemcpyHostToDevice,
                           c->stream));
  CLO_CUDA(cudaStreamSynchronize(c->stream));  // the pinned staging is reused
  c->ntok_dirty = false;
  return CLO_OK;
}

// Enqueues layers [l0, l1) of the current step: q / out hold those layers' blocks.
static clo_status enqueue_layers(clo_ctx* c, int l0, int l1, const uint16_t* qd, float* od) {
  DevState& s = c->ds;
  s.l0 = l0;
  s.l1 = l1;
  s.q_l0 = l0;
  const int64_t units = (int64_t)(l1 - l0) * c->B * c->Hkv;
  // chunks of 8192 (contexts up to 32K) or 16384 tokens, halved (down to 1024) while the
  // launch's units would give fewer than 8 chunks per SM: a launch with few units (one
  // layer, a small batch) spreads each selection over more compute groups.  All chunks
  // of a unit run at once (their waits need it), so a unit has at most one chunk per SM.
  int chunk = c->Nmax <= 32768 ? 8192 : kSelChunkMax;
  auto nchunks = [&](int ch) { return (c->Nmax + ch - 1) / ch; };
  while (chunk > kSelChunkMin && units * nchunks(chunk) < 8LL * c->sms && nchunks(chunk / 2) <= c->sms) chunk /= 2;
  s.sel_chunk_miss = chunk;
  // persistent units of contexts up to 32K are selected whole by one group (no waits on
  // other groups) when the launch holds units enough to occupy the groups
  s.sel_chunk = (c->Nmax <= 32768 && units >= c->whole_unit_min_units) ? (int)c->Nmax : chunk;
  s.nch = (int)nchunks(s.sel_chunk);
  s.nch_miss = (int)nchunks(s.sel_chunk_miss);
  // fetch items: 256 rows, or smaller while the launch's selected rows would give fewer
  // than 2 items per SM's fetch warps (3 per SM)
  int frows = kChunkRows;
  while (frows > 32 && units * c->kmax / frows < 6LL * c->sms) frows /= 2;
  s.fetch_rows = frows;
  // attention splits: long selections take 2048 rows (fewer partials to merge, measured
  // ~5 % faster on 512K contexts), others 1024; a small launch takes 256 (one fetch chunk),
  // so the attention that waits for the last fetched rows is short
  const bool small = units < c->whole_unit_min_units;
  s.split_rows = small ? 256 : (c->kmax > 8192 ? 2048 : 1024);
  s.nsplit = (int)((c->kmax + s.split_rows - 1) / s.split_rows);
  // query rows hashed per decide CTA: fewer in a small launch, for more CTAs
  s.decide_rows = small ? 16 : 32;
  const bool warm = c->warmup_mode && c->step < c->W;
  s.adapt_active = (c->cfg.adaptive_tau && !warm) ? 1 : 0;
  s.step_index = c->step;
  const bool timed = c->cfg.timing != 0;
  cudaEvent_t* ev = nullptr;
  if (timed) {
    if (c->ev_used == c->ev_pool.size()) {
      std::array<cudaEvent_t, 3> set{};
      for (auto& e : set) CLO_CUDA(cudaEventCreate(&e));
      c->ev_pool.push_back(set);
    }
    ev = c->ev_pool[c->ev_used++].data();
  }
  if (l0 == 0) ++c->epoch;
  if (timed) CLO_CUDA(cudaEventRecord(ev[0], c->stream));
  // the step's counters are zeroed once per step; queues, lists and flags per launch
  const size_t ctr_bytes = l0 == 0 ? 0 : sizeof(unsigned long long) * C_NUM * kCtrLanes;
  CLO_CUDA(cudaMemsetAsync(reinterpret_cast<unsigned char*>(c->step_zero) + ctr_bytes, 0,
                           c->step_zero_bytes - ctr_bytes, c->stream));
  CLO_CUDA(launch_decide(s, qd, c->step, warm ? 1 : 0, c->stream));
  if (timed) CLO_CUDA(cudaEventRecord(ev[1], c->stream));
  CLO_CUDA(launch_step_fused(s, qd, od, c->stream));
  if (timed) CLO_CUDA(cudaEventRecord(ev[2], c->stream));
  if (l1 == c->L) {  // the step is complete
    if (warm && c->step == c->W - 1) {
      CLO_CUDA(launch_finish_warmup(s, c->W, c->cfg.tau_offset, c->cfg.n_persist, c->stream));
      CLO_CUDA(launch_resident_fill(s, 0, c->Nmax, c->stream));
      c->warmup_done = true;
      c->persist_host_valid = false;
    }
    ++c->step;
  }
  c->next_layer = l1 == c->L ? 0 : l1;
  return CLO_OK;
}

// Host-buffer mode: stage nq elements of q into the device copy; returns the device
// pointers to use.
static clo_status stage_io(clo_ctx* c, const void* q, float* out, size_t nq, int32_t io_on_device,
                           const uint16_t** qd, float** od) {
  *qd = static_cast<const uint16_t*>(q);
  *od = out;
  if (io_on_device) return CLO_OK;
  if (!c->q_io) {
    const size_t full = (size_t)c->L * c->B * c->Hq * c->d;
    CLO_TRY(c->dalloc(&c->q_io, full));
    CLO_TRY(c->dalloc(&c->out_io, full));
  }
  CLO_CUDA(cudaMemcpyAsync(c->q_io, q, sizeof(uint16_t) * nq, cudaMemcpyHostToDevice, c->stream));
  *qd = c->q_io;
  *od = c->out_io;
  return CLO_OK;
}

CLO_API clo_status clo_decode_step(clo_ctx* c, const void* q, float* out, int32_t io_on_device) {
  if (!c) return fail(CLO_ERR_INVALID, "null context");
  if (!q || !out) return fail(CLO_ERR_INVALID, "null q/out");
  if (c->next_layer != 0)
    return fail(CLO_ERR_STATE, "a layer-by-layer step is in progress (next layer " +
                                   std::to_string(c->next_layer) + ")");
  if (c->ntok_dirty) CLO_TRY(refresh_lengths(c));
  const size_t nq = (size_t)c->L * c->B * c->Hq * c->d;
  const uint16_t* qd = nullptr;
  float* od = nullptr;
  CLO_TRY(stage_io(c, q, out, nq, io_on_device, &qd, &od));
  CLO_TRY(enqueue_layers(c, 0, c->L, qd, od));
  if (!io_on_device) {
    CLO_CUDA(cudaMemcpyAsync(out, c->out_io, sizeof(float) * nq, cudaMemcpyDeviceToHost, c->stream));
    return clo_sync(c);
  }
  return CLO_OK;
}

CLO_API clo_status clo_decode_layer(clo_ctx* c, int32_t layer, const void* q, float* out, int32_t io_on_device) {
  if (!c) return fail(CLO_ERR_INVALID, "null context");
  if (!q || !out) return fail(CLO_ERR_INVALID, "null q/out");
  if (layer < 0 || layer >= c->L) return fail(CLO_ERR_INVALID, "layer out of range");
  if (layer != c->next_layer)
    return fail(CLO_ERR_STATE, "layers must be decoded in order: expected layer " + std::to_string(c->next_layer) +
                                   ", got " + std::to_string(layer));
  if (layer == 0 && c->ntok_dirty) CLO_TRY(refresh_lengths(c));
  const size_t nq = (size_t)c->B * c->Hq * c->d;
  const uint16_t* qd = nullptr;
  float* od = nullptr;
  CLO_TRY(stage_io(c, q, out, nq, io_on_device, &qd, &od));
  CLO_TRY(enqueue_layers(c, layer, layer + 1, qd, od));
  if (!io_on_device) {
    CLO_CUDA(cudaMemcpyAsync(out, c->out_io, sizeof(float) * nq, cudaMemcpyDeviceToHost, c->stream));
    return clo_sync(c);
  }
  return CLO_OK;
}

CLO_API clo_status clo_stats(clo_ctx* c, clo_stats_t* out) {
  if (!c || !out) return fail(CLO_ERR_INVALID, "null argument");
  CLO_CUDA(cudaStreamSynchronize(c->stream));
  unsigned long long last_l[C_NUM * kCtrLanes], tot_l[C_NUM * kCtrLanes], last[C_NUM] = {}, tot[C_NUM] = {};
  CLO_CUDA(cudaMemcpy(last_l, c->ds.step_ctr, sizeof(last_l), cudaMemcpyDeviceToHost));
  CLO_CUDA(cudaMemcpy(tot_l, c->ds.total_ctr, sizeof(tot_l), cudaMemcpyDeviceToHost));
  for (int i = 0; i < C_NUM * kCtrLanes; ++i) {
    last[i / kCtrLanes] += last_l[i];
    tot[i / kCtrLanes] += tot_l[i];
  }
  std::memset(out, 0, sizeof(*out));
  out->steps = c->step;
  out->units_hit = (int64_t)tot[C_HIT];
  out->units_miss = (int64_t)tot[C_MISS];
  out->units_persist = (int64_t)tot[C_PERSIST];
  out->host_bytes = (int64_t)tot[C_HOST_BYTES];
  out->hbm_bytes_alg = (int64_t)tot[C_HBM_BYTES];
  out->timeouts = (int64_t)tot[C_TIMEOUTS];
  out->last_hit = (int64_t)last[C_HIT];
  out->last_miss = (int64_t)last[C_MISS];
  out->last_persist = (int64_t)last[C_PERSIST];
  out->last_host_bytes = (int64_t)last[C_HOST_BYTES];
  out->last_hbm_bytes_alg = (int64_t)last[C_HBM_BYTES];
  out->warmup_done = c->warmup_done ? 1 : 0;
  out->timed_steps = (int32_t)c->ev_used;
  for (size_t i = 0; i < c->ev_used; ++i) {
    const cudaEvent_t* e = c->ev_pool[i].data();
    float t[3];
    CLO_CUDA(cudaEventElapsedTime(&t[0], e[0], e[1]));
    CLO_CUDA(cudaEventElapsedTime(&t[1], e[1], e[2]));
    CLO_CUDA(cudaEventElapsedTime(&t[2], e[0], e[2]));
    out->sum_ms_decide += t[0];
    out->sum_ms_fused += t[1];
    out->sum_ms_total += t[2];
    if (i + 1 == c->ev_used) {
      out->last_ms_decide = t[0];
      out->last_ms_fused = t[1];
      out->last_ms_total = t[2];
    }
  }
  c->ev_used = 0;
  return read_device_error(c);
}

CLO_API clo_status clo_debug_get(clo_ctx* c, int32_t what, int32_t layer, int32_t seq, int32_t kvh, void* dst,
                                 int64_t dst_bytes) {
  if (!c || !dst) return fail(CLO_ERR_INVALID, "null argument");
  const bool per_unit = what == CLO_DBG_KEY_CODES || what == CLO_DBG_QUERY_CODES || what == CLO_DBG_IDX ||
                        what == CLO_DBG_SLOT_ROWS;
  if (per_unit && (layer < 0 || layer >= c->L || seq < 0 || seq >= c->B || kvh < 0 || kvh >= c->Hkv))
    return fail(CLO_ERR_INVALID, "unit out of range");
  CLO_CUDA(cudaStreamSynchronize(c->stream));
  const DevState& s = c->ds;
  const int64_t u = ((int64_t)layer * c->B + seq) * c->Hkv + kvh;
  const int64_t N = per_unit ? c->ntok[(size_t)layer * c->B + seq] : 0;
  const int64_t k = per_unit ? topk_for(N, c->cfg.topk, c->cfg.topk_ratio) : 0;
  const void* src = nullptr;
  int64_t bytes = 0;
  switch (what) {
    case CLO_DBG_KEY_CODES:
      src = s.codes + u * c->Nmax;
      bytes = N * 16;
      break;
    case CLO_DBG_QUERY_CODES:
      src = s.qcodes + ((int64_t)layer * c->B + seq) * c->Hq + (int64_t)kvh * c->G;
      bytes = (int64_t)c->G * 16;
      break;
    case CLO_DBG_IDX:
      src = s.idx + u * c->kmax;
      bytes = k * 4;
      break;
    case CLO_DBG_DECISION:
      src = s.decision;
      bytes = c->U;
      break;
    case CLO_DBG_SLOT_ROWS:
      src = s.slots + u * c->kmax * 2 * c->d;
      bytes = k * 4 * c->d;
      break;
    case CLO_DBG_TAU:
      src = s.tau;
      bytes = (int64_t)c->L * c->Hkv * 4;
      break;
    case CLO_DBG_PERSIST:
      src = s.persist;
      bytes = (int64_t)c->L * c->Hkv;
      break;
    case CLO_DBG_SHAT:
      src = s.shat;
      bytes = (int64_t)c->L * c->Hkv * 8;
      break;
    case CLO_DBG_COS:
      src = s.cosv;
      bytes = c->U * 4;
      break;
    case CLO_DBG_TIMELINE:
      src = c->timeline_dev;
      bytes = (int64_t)kTimelineSlots * 8;
      break;
    case CLO_DBG_STEP_BYTES:
      if (!s.step_bytes) return fail(CLO_ERR_STATE, "the per-step byte history needs timing mode");
      src = s.step_bytes;
      bytes = (int64_t)kStepHist * 16;
      break;
    case CLO_DBG_POOL_NODE: {  // host-side value
      if (dst_bytes < 4) return fail(CLO_ERR_INVALID, "dst too small: need 4 bytes");
      *static_cast<int32_t*>(dst) = c->pool_node;
      return read_device_error(c);
    }
    case CLO_DBG_TOPK: {  // host-side values: the same rule as the device's counts
      if (dst_bytes < (int64_t)c->L * c->B * 4)
        return fail(CLO_ERR_INVALID, "dst too small: need " + std::to_string((int64_t)c->L * c->B * 4) + " bytes");
      int32_t* kd = static_cast<int32_t*>(dst);
      for (size_t i = 0; i < c->ntok.size(); ++i) kd[i] = (int32_t)topk_for(c->ntok[i], c->cfg.topk, c->cfg.topk_ratio);
      return read_device_error(c);
    }
    default:
      return fail(CLO_ERR_INVALID, "unknown debug item " + std::to_string(what));
  }
  if (dst_bytes < bytes)
    return fail(CLO_ERR_INVALID, "dst too small: need " + std::to_string(bytes) + " bytes");
  CLO_CUDA(cudaMemcpy(dst, src, (size_t)bytes, cudaMemcpyDeviceToHost));
  return read_device_error(c);
}

CLO_API clo_status clo_set(clo_ctx* c, int32_t key, int64_t value) {
  if (!c) return fail(CLO_ERR_INVALID, "null context");
  switch (key) {
    case CLO_SET_DROP_FLAG_LAYER:
      c->ds.drop_flag_layer = (int)value;
      c->cfg.debug_drop_flag_layer = (int32_t)value;
      return CLO_OK;
    case CLO_SET_WAIT_TIMEOUT_NS:
      if (value <= 0) return fail(CLO_ERR_INVALID, "timeout must be > 0");
      c->ds.wait_timeout_ns = value;
      c->cfg.wait_timeout_ns = value;
      return CLO_OK;
    default:
      return fail(CLO_ERR_INVALID, "unknown setting " + std::to_string(key));
  }
}

}  // extern "C"

namespace clo {
void set_last_error_text(const char* msg) { g_last_error = msg ? msg : ""; }
}  // namespace clo
