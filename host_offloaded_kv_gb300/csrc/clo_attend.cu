// Zero-copy fetch of missed heads' rows fused with split-K sparse decode attention.
//
// One persistent, warp-specialised kernel per decode step:
//   * fetch warps pull the selected K|V rows of every missed unit straight from
//     pinned, device-mapped host memory (16-byte loads, no CPU thread on the data
//     path) into the unit's on-GPU cache slot, chunk by chunk in layer order, and
//     release a ready flag per chunk (CLO abstract, feature (3): zero-copy transfer
//     engine and GPU-centric synchronisation; "CLO (2511.14510) - L3 Per-Paper
//     Synthesis", section 2.1 item 3: UVA polling instead of CPU-side sync);
//   * attention warp groups compute out_g = sum_{r in S} softmax_r(q_g.k_r/sqrt(d)) v_r
//     split over rows: first the units that need no transfer (reused and
//     persistent heads), then the missed units in layer order, each split waiting
//     (bounded) on the ready flag of the chunk it reads -- the fetch runs ahead of
//     the attention that consumes it, as CLO's prefetch runs a layer ahead
//     (section 5.6).  The last split of a unit merges the splits by log-sum-exp.
// Fetch warps never wait, so every flag an attention group waits on is released
// by a warp that is running: no co-residency assumption is needed.
#include "clo_internal.cuh"

namespace clo {

namespace {

constexpr int kFetchWarps = 4;
constexpr int kAttWarps = 4;
constexpr int kAttThreads = 32 * kAttWarps;
constexpr int kFAThreads = 32 * (kFetchWarps + kAttWarps);
constexpr int kFetchUnroll = 8;
constexpr int kAttTile = 32;

__device__ __forceinline__ void att_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kAttThreads) : "memory"); }

// position p of a per-layer list -> layer (pre: exclusive prefix over layers, pre[L] > p)
__device__ __forceinline__ int layer_of(const int* pre, int L, int p) {
  int lo = 0, hi = L;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pre[mid] <= p)
      lo = mid;
    else
      hi = mid;
  }
  return lo;
}

__device__ void wait_ready(const uint32_t* flag, const DevState& s) {
  if (ld_acquire_u32(flag) >= 1u) return;
  const uint64_t t0 = global_timer_ns();
  unsigned ns = 32;
  while (ld_acquire_u32(flag) < 1u) {
    if (global_timer_ns() - t0 > (uint64_t)s.wait_timeout_ns) {
      atomicOr(s.err, kErrFlagTimeout);
      atomicAdd(&s.step_ctr[C_TIMEOUTS], 1ull);
      atomicAdd(&s.total_ctr[C_TIMEOUTS], 1ull);
      return;
    }
    __nanosleep(ns);
    if (ns < 2048) ns <<= 1;
  }
}

template <int D>
__device__ void fetch_role(const DevState& s, const int* pre_m, int n_miss, int lane) {
  constexpr int VPR = D / 4;  // 16-byte vectors per K|V record
  const int NS = s.nsplit, RS = s.split_rows, L = s.L, BH = s.B * s.Hkv;
  const int64_t n_items = (int64_t)n_miss * NS;
  while (true) {
    unsigned item = 0;
    if (lane == 0) item = atomicAdd(&s.queue[0], 1u);
    item = __shfl_sync(0xffffffffu, item, 0);
    if ((int64_t)item >= n_items) break;
    const int p = (int)(item / NS), c = (int)(item % NS);
    const int l = layer_of(pre_m, L, p);
    const int64_t u = s.miss_list[(int64_t)l * BH + (p - pre_m[l])];
    const int b = (int)((u / s.Hkv) % s.B);
    const int64_t k = s.kcount[b];
    const int64_t N = s.ntok[b];
    const int64_t r0 = (int64_t)c * RS;
    const int64_t r1 = (r0 + RS < k) ? r0 + RS : k;
    if (r0 < r1) {
      const uint4* pool = reinterpret_cast<const uint4*>(s.pool) + u * s.Nmax * VPR;
      uint4* slot = reinterpret_cast<uint4*>(s.slots) + u * s.kmax * VPR;
      const int32_t* ix = s.idx + u * s.kmax;
      const int64_t total = (r1 - r0) * VPR;
      for (int64_t e0 = lane; e0 < total; e0 += 32 * kFetchUnroll) {
        uint4 v[kFetchUnroll];
#pragma unroll
        for (int j = 0; j < kFetchUnroll; ++j) {
          const int64_t e = e0 + 32 * j;
          if (e < total) {
            const int64_t t = ix[r0 + e / VPR];
            if (t >= 0 && t < N) {
              v[j] = ld_nc_v4(pool + t * VPR + (e % VPR));
            } else {
              atomicOr(s.err, kErrBounds);
              v[j] = make_uint4(0, 0, 0, 0);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < kFetchUnroll; ++j) {
          const int64_t e = e0 + 32 * j;
          if (e < total) slot[r0 * VPR + e] = v[j];
        }
      }
    }
    __threadfence();
    __syncwarp();
    if (lane == 0 && l != s.drop_flag_layer) red_release_add_u32(&s.ready[u * NS + c], 1u);
  }
}

template <int D>
struct AttSmem {
  static constexpr int ROWW = 2 * D + 8;  // bf16 per smem row, padded by 16 bytes
  static constexpr int NG = kAttThreads / D;
  float qs[kMaxG][D];
  uint16_t rows[kAttTile][ROWW];
  float sc[kMaxG][kAttTile];
  float m_run[kMaxG], l_run[kMaxG], alpha[kMaxG];
  float red[NG > 1 ? NG : 1][kMaxG][D];
  int item;
  int last;
};

// One split (rows [r0, r1) of unit u) by the 128-thread attention group.
template <int D>
__device__ void attend_split(const DevState& s, AttSmem<D>& sm, const uint16_t* __restrict__ q,
                             float* __restrict__ out, int64_t u, int split, int64_t r0, int64_t r1, int gtid) {
  constexpr int VPR = D / 4;
  constexpr int NG = AttSmem<D>::NG;
  const int h = (int)(u % s.Hkv);
  const int b = (int)((u / s.Hkv) % s.B);
  const int l = (int)(u / ((int64_t)s.Hkv * s.B));
  const int G = s.G;
  const int warp = gtid >> 5, lane = gtid & 31;
  const int64_t N = s.ntok[b];
  const bool persistent = s.decision[u] == CLO_DEC_PERSIST;
  const int32_t* ix = s.idx + u * s.kmax;
  const uint4* src;
  if (persistent) {
    const int p = s.persist_slot[l * s.Hkv + h];
    src = reinterpret_cast<const uint4*>(s.resident) + ((((int64_t)l * s.B + b) * s.P + p) * s.Nmax) * VPR;
  } else {
    src = reinterpret_cast<const uint4*>(s.slots) + (u * s.kmax) * VPR;
  }
  const float qscale = 1.4426950408889634f * rsqrtf((float)D);  // scores in log2 units
  const uint16_t* qg = q + (((int64_t)l * s.B + b) * s.Hq + (int64_t)h * G) * D;
  for (int e = gtid; e < G * D; e += kAttThreads) sm.qs[e / D][e % D] = bf16_bits_to_f32(qg[e]) * qscale;
  if (gtid < kMaxG) {
    sm.m_run[gtid] = -INFINITY;
    sm.l_run[gtid] = 0.f;
  }
  float acc[kMaxG];
#pragma unroll
  for (int g = 0; g < kMaxG; ++g) acc[g] = 0.f;
  const int dj = gtid % D;
  const int rg = gtid / D;
  att_bar();

  for (int64_t rb = r0; rb < r1; rb += kAttTile) {
    const int nrows = (int)((r1 - rb) < kAttTile ? (r1 - rb) : kAttTile);
    for (int e = gtid; e < nrows * VPR; e += kAttThreads) {
      const int r = e / VPR, c = e % VPR;
      int64_t srow = rb + r;
      if (persistent) {
        srow = ix[rb + r];
        if (srow < 0 || srow >= N) {
          atomicOr(s.err, kErrBounds);
          srow = 0;
        }
      }
      cp_async16(&sm.rows[r][c * 8], src + srow * VPR + c);
    }
    cp_async_commit();
    cp_async_wait<0>();
    att_bar();
    for (int p = gtid; p < G * kAttTile; p += kAttThreads) {
      const int g = p / kAttTile, r = p % kAttTile;
      float dot = -INFINITY;
      if (r < nrows) {
        dot = 0.f;
        const uint4* kr = reinterpret_cast<const uint4*>(&sm.rows[r][0]);
#pragma unroll 4
        for (int i = 0; i < D / 8; ++i) {
          const uint4 w = kr[i];
          const float4 qa = *reinterpret_cast<const float4*>(&sm.qs[g][8 * i]);
          const float4 qb = *reinterpret_cast<const float4*>(&sm.qs[g][8 * i + 4]);
          dot = fmaf(qa.x, __uint_as_float(w.x << 16), dot);
          dot = fmaf(qa.y, __uint_as_float(w.x & 0xffff0000u), dot);
          dot = fmaf(qa.z, __uint_as_float(w.y << 16), dot);
          dot = fmaf(qa.w, __uint_as_float(w.y & 0xffff0000u), dot);
          dot = fmaf(qb.x, __uint_as_float(w.z << 16), dot);
          dot = fmaf(qb.y, __uint_as_float(w.z & 0xffff0000u), dot);
          dot = fmaf(qb.z, __uint_as_float(w.w << 16), dot);
          dot = fmaf(qb.w, __uint_as_float(w.w & 0xffff0000u), dot);
        }
      }
      sm.sc[g][r] = dot;
    }
    att_bar();
    for (int g = warp; g < G; g += kAttWarps) {
      const float v = sm.sc[g][lane];
      const float mx = warp_max(v);
      const float mo = sm.m_run[g];
      const float mn = fmaxf(mo, mx);
      const float pv = exp2f(v - mn);
      const float ps = warp_sum(pv);
      sm.sc[g][lane] = pv;
      if (lane == 0) {
        const float a = exp2f(mo - mn);
        sm.alpha[g] = a;
        sm.l_run[g] = sm.l_run[g] * a + ps;
        sm.m_run[g] = mn;
      }
    }
    att_bar();
#pragma unroll
    for (int g = 0; g < kMaxG; ++g)
      if (g < G) acc[g] *= sm.alpha[g];
    for (int r = rg; r < nrows; r += NG) {
      const float v = bf16_bits_to_f32(sm.rows[r][D + dj]);
#pragma unroll
      for (int g = 0; g < kMaxG; ++g)
        if (g < G) acc[g] = fmaf(sm.sc[g][r], v, acc[g]);
    }
    att_bar();
  }

  if (NG > 1) {
#pragma unroll
    for (int g = 0; g < kMaxG; ++g)
      if (g < G) sm.red[rg][g][dj] = acc[g];
    att_bar();
  }
  float* part = s.part + ((u * s.nsplit + split) * G) * (D + 2);
  if (gtid < D) {
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) {
      if (g < G) {
        float a = acc[g];
        if (NG > 1) {
          a = 0.f;
          for (int r = 0; r < NG; ++r) a += sm.red[r][g][gtid];
        }
        part[g * (D + 2) + 2 + gtid] = a;
      }
    }
  }
  if (gtid < G) {
    part[gtid * (D + 2) + 0] = sm.m_run[gtid];
    part[gtid * (D + 2) + 1] = sm.l_run[gtid];
  }
  __threadfence();
  att_bar();
  if (gtid == 0) {
    const uint32_t prev = atomicAdd(&s.unit_done[u], 1u);
    sm.last = (prev == (uint32_t)s.nsplit - 1u);
  }
  att_bar();
  if (!sm.last) return;
  __threadfence();
  const float* pu = s.part + (u * s.nsplit) * G * (D + 2);
  float* og = out + (((int64_t)l * s.B + b) * s.Hq + (int64_t)h * G) * D;
  for (int e = gtid; e < G * D; e += kAttThreads) {
    const int g = e / D, j = e % D;
    float M = -INFINITY;
    for (int sp = 0; sp < s.nsplit; ++sp) M = fmaxf(M, __ldcg(pu + (sp * G + g) * (D + 2)));
    float Lsum = 0.f, O = 0.f;
    for (int sp = 0; sp < s.nsplit; ++sp) {
      const float* ps = pu + (sp * G + g) * (D + 2);
      const float ls = __ldcg(ps + 1);
      if (ls > 0.f) {
        const float w = exp2f(__ldcg(ps) - M);
        Lsum = fmaf(ls, w, Lsum);
        O = fmaf(__ldcg(ps + 2 + j), w, O);
      }
    }
    og[g * D + j] = O / Lsum;
  }
  if (gtid == 0) s.unit_done[u] = 0u;
}

template <int D>
__global__ void __launch_bounds__(kFAThreads, 4) k_fetch_attend(DevState s, const uint16_t* __restrict__ q,
                                                             float* __restrict__ out) {
  __shared__ int pre_o[kMaxLayers + 1], pre_m[kMaxLayers + 1];
  __shared__ __align__(16) AttSmem<D> sm;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = s.L;
  if (tid == 0) {
    int a = 0, c = 0;
    pre_o[0] = 0;
    pre_m[0] = 0;
    for (int l = 0; l < L; ++l) {
      a += s.lcnt[l];
      c += s.lcnt[L + l];
      pre_o[l + 1] = a;
      pre_m[l + 1] = c;
    }
  }
  __syncthreads();
  const int n_other = pre_o[L], n_miss = pre_m[L];
  if (warp < kFetchWarps) {
    fetch_role<D>(s, pre_m, n_miss, lane);
    return;  // no block-wide barrier after this point
  }
  const int gtid = tid - 32 * kFetchWarps;
  const int NS = s.nsplit, RS = s.split_rows, BH = s.B * s.Hkv;
  const int64_t n_items_o = (int64_t)n_other * NS;
  const int64_t n_items = (int64_t)(n_other + n_miss) * NS;
  while (true) {
    if (gtid == 0) sm.item = (int)atomicAdd(&s.queue[1], 1u);
    att_bar();
    const int64_t item = sm.item;
    if (item >= n_items) break;
    const bool missed = item >= n_items_o;
    const int64_t j = missed ? item - n_items_o : item;
    const int p = (int)(j / NS), sp = (int)(j % NS);
    const int* pre = missed ? pre_m : pre_o;
    const int l = layer_of(pre, L, p);
    const int64_t u = (missed ? s.miss_list : s.other_list)[(int64_t)l * BH + (p - pre[l])];
    const int b = (int)((u / s.Hkv) % s.B);
    const int64_t k = s.kcount[b];
    const int64_t r0 = (int64_t)sp * RS;
    const int64_t r1 = (r0 + RS < k) ? r0 + RS : k;
    if (missed && r0 < r1) {
      if (gtid == 0) wait_ready(&s.ready[u * NS + sp], s);
      att_bar();
    }
    attend_split<D>(s, sm, q, out, u, sp, r0, r1, gtid);
    att_bar();
  }
}

// Full K/V of persistent heads, host pool -> resident HBM copy, tokens [t0, t1).
__global__ void k_resident_fill(DevState s, int64_t t0, int64_t t1) {
  const int vpr = s.d / 4;
  const int64_t nunits = (int64_t)s.L * s.B * s.Hkv;
  for (int64_t u = blockIdx.y; u < nunits; u += gridDim.y) {
    const int h = (int)(u % s.Hkv);
    const int b = (int)((u / s.Hkv) % s.B);
    const int l = (int)(u / ((int64_t)s.Hkv * s.B));
    const int p = s.persist_slot[l * s.Hkv + h];
    if (p < 0) continue;
    const int64_t tend = (t1 < s.ntok[b]) ? t1 : s.ntok[b];
    if (tend <= t0) continue;
    const int64_t n = (tend - t0) * vpr;
    const uint4* src = reinterpret_cast<const uint4*>(s.pool) + (u * s.Nmax + t0) * vpr;
    uint4* dst = reinterpret_cast<uint4*>(s.resident) + ((((int64_t)l * s.B + b) * s.P + p) * s.Nmax + t0) * vpr;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x)
      dst[e] = ld_nc_v4(src + e);
  }
}

template <int D>
int fa_grid() {
  static int grid = 0;
  if (grid == 0) {
    int dev = 0, sms = 0, per_sm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_fetch_attend<D>, kFAThreads, 0);
    grid = sms * (per_sm > 0 ? per_sm : 1);
  }
  return grid;
}

}  // namespace

cudaError_t launch_fetch_attend(const DevState& s, const uint16_t* q, float* out, cudaStream_t st) {
  if (s.L > kMaxLayers) return cudaErrorInvalidValue;
  if (s.d == 128) {
    k_fetch_attend<128><<<fa_grid<128>(), kFAThreads, 0, st>>>(s, q, out);
  } else if (s.d == 64) {
    k_fetch_attend<64><<<fa_grid<64>(), kFAThreads, 0, st>>>(s, q, out);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_resident_fill(const DevState& s, int64_t t0, int64_t t1, cudaStream_t st) {
  if (s.P <= 0 || s.resident == nullptr || t1 <= t0) return cudaSuccess;
  const int64_t U = (int64_t)s.L * s.B * s.Hkv;
  dim3 grid(64, (unsigned)(U < 65535 ? U : 65535));
  k_resident_fill<<<grid, 256, 0, st>>>(s, t0, t1);
  return cudaGetLastError();
}

}  // namespace clo
