// Zero-copy fetch of missed heads' rows and split-K sparse decode attention.
//
// Fetch: for a unit that missed, the selected K/V rows are loaded by the GPU
// straight from pinned, device-mapped host memory (16-byte loads, no CPU thread on
// the data path) into the unit's on-GPU cache slot (CLO abstract, feature (3):
// zero-copy transfer engine; "CLO (2511.14510) - L3 Per-Paper Synthesis",
// section 2.1 item 3: GDRCopy + UVA).
//
// Attention: out_g = sum_{r in S} softmax_r(q_g . k_r / sqrt(d)) v_r over the
// selected rows S of the unit (top-k sparse attention, CLO abstract), split over
// rows; the splits are merged with their log-sum-exp by the last CTA of the unit.
// Rows come from the slot (missed / reused heads) or, for persistent heads, from
// the resident copy through the selection indices.
#include "clo_internal.cuh"

namespace clo {

namespace {

constexpr int kGatherThreads = 256;
constexpr int kGatherRows = 128;
constexpr int kGatherUnroll = 8;

__global__ void __launch_bounds__(kGatherThreads) k_gather(DevState s) {
  const int64_t u = blockIdx.y;
  if (s.decision[u] != CLO_DEC_MISS) return;
  const int b = (int)((u / s.Hkv) % s.B);
  const int64_t k = s.kcount[b];
  const int64_t N = s.ntok[b];
  const int64_t r0 = (int64_t)blockIdx.x * kGatherRows;
  if (r0 >= k) return;
  const int64_t r1 = (r0 + kGatherRows < k) ? r0 + kGatherRows : k;
  const int vpr = s.d / 4;  // 16-byte vectors per K|V record
  const int64_t total = (r1 - r0) * vpr;
  const uint4* pool = reinterpret_cast<const uint4*>(s.pool) + u * s.Nmax * vpr;
  uint4* slot = reinterpret_cast<uint4*>(s.slots) + u * s.kmax * vpr;
  const int32_t* ix = s.idx + u * s.kmax;
  for (int64_t e0 = threadIdx.x; e0 < total; e0 += (int64_t)kGatherThreads * kGatherUnroll) {
    uint4 v[kGatherUnroll];
#pragma unroll
    for (int j = 0; j < kGatherUnroll; ++j) {
      const int64_t e = e0 + (int64_t)j * kGatherThreads;
      if (e < total) {
        const int64_t r = r0 + e / vpr;
        const int c = (int)(e % vpr);
        const int64_t t = ix[r];
        if (t >= 0 && t < N) {
          v[j] = ld_nc_v4(pool + t * vpr + c);
        } else {
          atomicOr(s.err, kErrBounds);
          v[j] = make_uint4(0, 0, 0, 0);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kGatherUnroll; ++j) {
      const int64_t e = e0 + (int64_t)j * kGatherThreads;
      if (e < total) slot[(r0 + e / vpr) * vpr + (e % vpr)] = v[j];
    }
  }
}

constexpr int kAttThreads = 128;
constexpr int kAttTile = 32;

template <int D>
__global__ void __launch_bounds__(kAttThreads) k_attend(DevState s, const uint16_t* __restrict__ q,
                                                        float* __restrict__ out) {
  constexpr int VPR = D / 4;            // 16-byte vectors per record
  constexpr int ROWW = 2 * D + 8;       // bf16 elements per smem row (padded by 16 bytes)
  constexpr int NG = kAttThreads / D;   // row groups in the PV phase
  __shared__ __align__(16) float qs[kMaxG][D];
  __shared__ __align__(16) uint16_t rows[kAttTile][ROWW];
  __shared__ float sc[kMaxG][kAttTile];
  __shared__ float m_run[kMaxG], l_run[kMaxG], alpha[kMaxG];
  __shared__ float red[NG > 1 ? NG : 1][kMaxG][D];
  __shared__ int s_last;

  const int64_t u = blockIdx.y;
  const int split = blockIdx.x;
  const int h = (int)(u % s.Hkv);
  const int b = (int)((u / s.Hkv) % s.B);
  const int l = (int)(u / ((int64_t)s.Hkv * s.B));
  const int G = s.G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t k = s.kcount[b];
  const int64_t N = s.ntok[b];
  const int64_t r0 = (int64_t)split * s.split_rows;
  const int64_t r1 = (r0 + s.split_rows < k) ? r0 + s.split_rows : k;
  const bool persistent = s.decision[u] == CLO_DEC_PERSIST;
  const int32_t* ix = s.idx + u * s.kmax;
  const uint4* src;
  if (persistent) {
    const int p = s.persist_slot[l * s.Hkv + h];
    src = reinterpret_cast<const uint4*>(s.resident) + ((((int64_t)l * s.B + b) * s.P + p) * s.Nmax) * VPR;
  } else {
    src = reinterpret_cast<const uint4*>(s.slots) + (u * s.kmax) * VPR;
  }

  // q scaled so that scores are in log2 units: q . k / sqrt(d) * log2(e)
  const float qscale = 1.4426950408889634f * rsqrtf((float)D);
  const uint16_t* qg = q + (((int64_t)l * s.B + b) * s.Hq + (int64_t)h * G) * D;
  for (int e = tid; e < G * D; e += kAttThreads) qs[e / D][e % D] = bf16_bits_to_f32(qg[e]) * qscale;
  if (tid < kMaxG) {
    m_run[tid] = -INFINITY;
    l_run[tid] = 0.f;
  }
  float acc[kMaxG];
#pragma unroll
  for (int g = 0; g < kMaxG; ++g) acc[g] = 0.f;
  const int dj = tid % D;
  const int rg = tid / D;
  __syncthreads();

  for (int64_t rb = r0; rb < r1; rb += kAttTile) {
    const int nrows = (int)((r1 - rb) < kAttTile ? (r1 - rb) : kAttTile);
    for (int e = tid; e < nrows * VPR; e += kAttThreads) {
      const int r = e / VPR, c = e % VPR;
      int64_t srow = rb + r;
      if (persistent) {
        srow = ix[rb + r];
        if (srow < 0 || srow >= N) {
          atomicOr(s.err, kErrBounds);
          srow = 0;
        }
      }
      cp_async16(&rows[r][c * 8], src + srow * VPR + c);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    // scores of (head, row) pairs
    for (int p = tid; p < G * kAttTile; p += kAttThreads) {
      const int g = p / kAttTile, r = p % kAttTile;
      float dot = -INFINITY;
      if (r < nrows) {
        dot = 0.f;
        const uint4* kr = reinterpret_cast<const uint4*>(&rows[r][0]);
#pragma unroll 4
        for (int i = 0; i < D / 8; ++i) {
          const uint4 w = kr[i];
          const float4 qa = *reinterpret_cast<const float4*>(&qs[g][8 * i]);
          const float4 qb = *reinterpret_cast<const float4*>(&qs[g][8 * i + 4]);
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
      sc[g][r] = dot;
    }
    __syncthreads();
    // online softmax statistics, one warp per head
    for (int g = warp; g < G; g += kAttThreads / 32) {
      const float v = sc[g][lane];
      const float mx = warp_max(v);
      const float mo = m_run[g];
      const float mn = fmaxf(mo, mx);
      const float pv = exp2f(v - mn);
      const float ps = warp_sum(pv);
      sc[g][lane] = pv;
      if (lane == 0) {
        const float a = exp2f(mo - mn);
        alpha[g] = a;
        l_run[g] = l_run[g] * a + ps;
        m_run[g] = mn;
      }
    }
    __syncthreads();
#pragma unroll
    for (int g = 0; g < kMaxG; ++g)
      if (g < G) acc[g] *= alpha[g];
    for (int r = rg; r < nrows; r += NG) {
      const float v = bf16_bits_to_f32(rows[r][D + dj]);
#pragma unroll
      for (int g = 0; g < kMaxG; ++g)
        if (g < G) acc[g] = fmaf(sc[g][r], v, acc[g]);
    }
    __syncthreads();
  }

  // reduce row groups, write this split's partial: {m, l, acc[D]} per head
  if (NG > 1) {
#pragma unroll
    for (int g = 0; g < kMaxG; ++g)
      if (g < G) red[rg][g][dj] = acc[g];
    __syncthreads();
  }
  float* part = s.part + ((u * s.nsplit + split) * G) * (D + 2);
  if (tid < D) {
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) {
      if (g < G) {
        float a = acc[g];
        if (NG > 1) {
          a = 0.f;
          for (int r = 0; r < NG; ++r) a += red[r][g][tid];
        }
        part[g * (D + 2) + 2 + tid] = a;
      }
    }
  }
  if (tid < G) {
    part[tid * (D + 2) + 0] = m_run[tid];
    part[tid * (D + 2) + 1] = l_run[tid];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const uint32_t prev = atomicAdd(&s.unit_done[u], 1u);
    s_last = (prev == (uint32_t)s.nsplit - 1u);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const float* pu = s.part + (u * s.nsplit) * G * (D + 2);
  float* og = out + (((int64_t)l * s.B + b) * s.Hq + (int64_t)h * G) * D;
  for (int e = tid; e < G * D; e += kAttThreads) {
    const int g = e / D, j = e % D;
    float M = -INFINITY;
    for (int sp = 0; sp < s.nsplit; ++sp) M = fmaxf(M, __ldcg(pu + (sp * G + g) * (D + 2)));
    float L = 0.f, O = 0.f;
    for (int sp = 0; sp < s.nsplit; ++sp) {
      const float* ps = pu + (sp * G + g) * (D + 2);
      const float ls = __ldcg(ps + 1);
      if (ls > 0.f) {
        const float w = exp2f(__ldcg(ps) - M);
        L = fmaf(ls, w, L);
        O = fmaf(__ldcg(ps + 2 + j), w, O);
      }
    }
    og[g * D + j] = O / L;
  }
  if (tid == 0) s.unit_done[u] = 0u;
}

// Full K/V of persistent heads, host pool -> resident HBM copy, tokens [t0, t1).
__global__ void k_resident_fill(DevState s, int64_t t0, int64_t t1) {
  const int vpr = s.d / 4;
  const int64_t per_unit = (t1 - t0) * vpr;
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
    (void)per_unit;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x)
      dst[e] = ld_nc_v4(src + e);
  }
}

}  // namespace

cudaError_t launch_gather(const DevState& s, uint32_t epoch, cudaStream_t st) {
  (void)epoch;
  const int64_t U = (int64_t)s.L * s.B * s.Hkv;
  dim3 grid((unsigned)((s.kmax + kGatherRows - 1) / kGatherRows), (unsigned)U);
  k_gather<<<grid, kGatherThreads, 0, st>>>(s);
  return cudaGetLastError();
}

cudaError_t launch_attend(const DevState& s, const uint16_t* q, float* out, uint32_t epoch, cudaStream_t st) {
  (void)epoch;
  const int64_t U = (int64_t)s.L * s.B * s.Hkv;
  dim3 grid((unsigned)s.nsplit, (unsigned)U);
  if (s.d == 128) {
    k_attend<128><<<grid, kAttThreads, 0, st>>>(s, q, out);
  } else if (s.d == 64) {
    k_attend<64><<<grid, kAttThreads, 0, st>>>(s, q, out);
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
