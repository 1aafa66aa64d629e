// Head-wise reuse decision and query hashing (one CTA per kv head and group of sequences).
//
// Reuse test: adjacent-step query cosine similarity is high (> 0.8) on most
// heads, which CLO turns into a cache-reuse condition ("CLO (2511.14510) - L3
// Per-Paper Synthesis", section 2.1 item 2; CLO abstract, feature (1):
// coarse-grained head-wise approximate on-GPU caching).  A unit reuses its
// previous selection iff cos(q_group, q_cached) >= tau[l][h], q_cached being the
// query of the unit's last refresh.  Persistent heads always reselect (CLO
// abstract, feature (2)).  Thresholds and persistent heads come from profiling
// (section 3.3 attack 6: s_hat_i, D_i, N_persist): warm-up steps reselect every
// unit and accumulate cos(q_t, q_{t-1}).
#include "clo_hash.cuh"
#include "clo_internal.cuh"

namespace clo {

namespace {

constexpr int kDecideThreads = 512;
constexpr int kHashSlots = kDecideThreads / 128;  // threads per code bit
constexpr int kMaxRows = 32;                        // hashed query rows per CTA

struct StridedF32 {
  const float* p;
  int stride;
  __device__ float operator()(int i) const { return p[i * stride]; }
};
struct StridedBF16 {
  const uint16_t* p;
  int stride;
  __device__ float operator()(int i) const { return bf16_bits_to_f32(p[i * stride]); }
};

// Units of one kv head handled by one CTA: as many sequences as fit `rows` (<= 32) query rows,
// at most one per warp.
__host__ __device__ inline int units_per_cta(int G, int B, int rows) {
  int n = (rows < kMaxRows ? rows : kMaxRows) / G;
  n = n < 1 ? 1 : (n > kDecideThreads / 32 ? kDecideThreads / 32 : n);
  return n < B ? n : B;
}

// One CTA per (layer, kv head, group of up to 32 / G sequences).  The head's
// projection R (d x 128 bf16) is staged once in shared memory by asynchronous
// 16-byte copies that overlap the reuse tests.  Warp w decides unit w from the query
// it holds in registers and writes the unit's G query rows (rows w*G .. w*G+G-1) to
// a transposed fp32 copy [d][slot][M] (row r at column (r % slots) * M + r / slots);
// then thread (slot, bit j) computes bit j of M rows at once from broadcast float4
// loads.
//   dynamic shared memory: Rs bf16 [d][128] | xs fp32 [d][kHashSlots * M]
template <int M>
__global__ void __launch_bounds__(kDecideThreads) k_decide(DevState s, const uint16_t* __restrict__ q, int64_t step,
                                                            int warmup_active) {
  extern __shared__ __align__(16) unsigned char dsm[];
  constexpr int XW = kHashSlots * M;  // floats per dimension in xs
  __shared__ int s_dec[kMaxRows];
  __shared__ uint32_t words[kMaxRows][4];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = s.G, d = s.d, GD = s.G * s.d;
  const int UPC = units_per_cta(G, s.B, s.decide_rows);
  const int ngrp = (s.B + UPC - 1) / UPC;
  const int lh = s.l0 * s.Hkv + (int)(blockIdx.x / ngrp);
  const int b0 = (blockIdx.x % ngrp) * UPC;
  const int nu = (s.B - b0) < UPC ? (s.B - b0) : UPC;
  const int l = lh / s.Hkv, h = lh % s.Hkv;
  uint16_t* Rs = reinterpret_cast<uint16_t*>(dsm);
  float* xs = reinterpret_cast<float*>(dsm + (size_t)d * 128 * 2);
  if (tid == 0 && s.timeline) atomicCAS(&s.timeline[TL_DEC_START], 0ull, global_timer_ns());
  {
    const uint4* src = reinterpret_cast<const uint4*>(s.R + (int64_t)lh * d * 128);
    for (int e = tid; e < d * 128 / 8; e += kDecideThreads) cp_async16(&Rs[e * 8], src + e);
    cp_async_commit();
  }

  // 1. reuse test of unit w by warp w; its query rows go to xs from registers
  if (warp < nu) {
    const int b = b0 + warp;
    const int64_t u = ((int64_t)l * s.B + b) * s.Hkv + h;
    // the unit's scalars, loaded up front (independent loads)
    const bool valid = s.qvalid[u] != 0;
    const bool pers = s.persist[lh] != 0;
    const float tau = s.tau[lh];
    const int64_t N = s.ntok[b], k = s.kcount[b];
    const uint16_t* qg = q + (((int64_t)(l - s.q_l0) * s.B + b) * s.Hq + (int64_t)h * G) * d;
    uint16_t* qc = s.qcache + u * GD;
    constexpr int kMaxPer = kMaxG * kMaxD / 256;  // uint4 of the group's query per lane
    uint4 xv[kMaxPer];
    float dot = 0.f, nq = 0.f, nc = 0.f;
#pragma unroll
    for (int p = 0; p < kMaxPer; ++p) {
      const int e = 8 * lane + 256 * p;
      if (e < GD) {
        xv[p] = *reinterpret_cast<const uint4*>(qg + e);
        const uint4 cv = *reinterpret_cast<const uint4*>(qc + e);
        const uint32_t xw[4] = {xv[p].x, xv[p].y, xv[p].z, xv[p].w}, cw[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float x0 = bf16_bits_to_f32(xw[i] & 0xffffu), x1 = bf16_bits_to_f32(xw[i] >> 16);
          const float c0 = bf16_bits_to_f32(cw[i] & 0xffffu), c1 = bf16_bits_to_f32(cw[i] >> 16);
          dot = fmaf(x1, c1, fmaf(x0, c0, dot));
          nq = fmaf(x1, x1, fmaf(x0, x0, nq));
          nc = fmaf(c1, c1, fmaf(c0, c0, nc));
        }
      }
    }
    dot = warp_sum(dot);
    nq = warp_sum(nq);
    nc = warp_sum(nc);
    const float cosv = (nq > 0.f && nc > 0.f) ? dot / (sqrtf(nq) * sqrtf(nc)) : 0.f;
    if (s.qprev) {  // adaptive thresholds: cos(q_t, q_{t-1}); q_t becomes the previous query
      uint16_t* qp = s.qprev + u * GD;
      const bool pvalid = s.qprev_valid[u] != 0;
      float pd = 0.f, pn = 0.f;
#pragma unroll
      for (int p = 0; p < kMaxPer; ++p) {
        const int e = 8 * lane + 256 * p;
        if (e < GD) {
          const uint4 pv = *reinterpret_cast<const uint4*>(qp + e);
          const uint32_t xw[4] = {xv[p].x, xv[p].y, xv[p].z, xv[p].w}, pw[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float x0 = bf16_bits_to_f32(xw[i] & 0xffffu), x1 = bf16_bits_to_f32(xw[i] >> 16);
            const float p0 = bf16_bits_to_f32(pw[i] & 0xffffu), p1 = bf16_bits_to_f32(pw[i] >> 16);
            pd = fmaf(x1, p1, fmaf(x0, p0, pd));
            pn = fmaf(p1, p1, fmaf(p0, p0, pn));
          }
          *reinterpret_cast<uint4*>(qp + e) = xv[p];
        }
      }
      pd = warp_sum(pd);
      pn = warp_sum(pn);
      if (lane == 0) {
        if (pvalid && s.adapt_active) {
          const float cp = (nq > 0.f && pn > 0.f) ? pd / (sqrtf(nq) * sqrtf(pn)) : 0.f;
          atomicAdd(&s.cos_sum[lh], (double)cp);
          atomicAdd(&s.cos_cnt[lh], 1u);
        }
        s.qprev_valid[u] = 1;
      }
    }
    int dec;
    if (warmup_active)
      dec = CLO_DEC_MISS;
    else if (pers)
      dec = CLO_DEC_PERSIST;
    else if (!valid)
      dec = CLO_DEC_MISS;
    else
      dec = (cosv >= tau) ? CLO_DEC_HIT : CLO_DEC_MISS;
    if (dec != CLO_DEC_HIT) {
#pragma unroll
      for (int p = 0; p < kMaxPer; ++p) {
        const int e = 8 * lane + 256 * p;
        if (e < GD) {
          const uint32_t xw[4] = {xv[p].x, xv[p].y, xv[p].z, xv[p].w};
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int ee = e + i, r = warp * G + ee / d, dim = ee % d;
            const uint32_t bits = (i & 1) ? (xw[i >> 1] >> 16) : (xw[i >> 1] & 0xffffu);
            xs[dim * XW + (r % kHashSlots) * M + r / kHashSlots] = bf16_bits_to_f32(bits);
          }
          if (dec == CLO_DEC_MISS) *reinterpret_cast<uint4*>(qc + e) = xv[p];
        }
      }
    }
    if (lane == 0) {
      if (warmup_active && step >= 1 && valid) atomicAdd(&s.shat_sum[lh], (double)cosv);
      if (dec == CLO_DEC_MISS) s.qvalid[u] = 1;
      s.decision[u] = (uint8_t)dec;
      s.cosv[u] = valid ? cosv : __int_as_float(0x7fc00000);
      s_dec[warp] = dec;
      // work lists and counters
      const int BH = s.B * s.Hkv;
      const int li = dec == CLO_DEC_HIT ? 0 : (dec == CLO_DEC_PERSIST ? 1 : 2);
      int32_t* lst = li == 0 ? s.hit_list : (li == 1 ? s.pers_list : s.miss_list);
      lst[(int64_t)l * BH + atomicAdd(&s.lcnt[li * s.L + l], 1)] = (int32_t)u;
      const int64_t rec = 4LL * d;  // bf16 K|V row in HBM
      const unsigned long long host = (dec == CLO_DEC_MISS) ? (unsigned long long)(k * s.rec_bytes) : 0ull;
      int64_t hbm = (int64_t)GD * 2 + (int64_t)GD * 4 + (valid ? (int64_t)GD * 2 : 0) + k * rec;
      if (dec != CLO_DEC_HIT) hbm += N * 16 + k * 4;
      if (dec == CLO_DEC_MISS) hbm += (int64_t)GD * 2 + k * rec;
      if (dec == CLO_DEC_MISS && s.kv_bits != 16) hbm += k * (2 * d / 64) * 8;  // groups' (scale, min)
      if (dec == CLO_DEC_PERSIST) hbm += k * 4;
      const int slot = dec == CLO_DEC_HIT ? C_HIT : (dec == CLO_DEC_MISS ? C_MISS : C_PERSIST);
      atomicAdd(&s.step_ctr[ctr_at(slot, u)], 1ull);
      atomicAdd(&s.total_ctr[ctr_at(slot, u)], 1ull);
      if (host) {
        atomicAdd(&s.step_ctr[ctr_at(C_HOST_BYTES, u)], host);
        atomicAdd(&s.total_ctr[ctr_at(C_HOST_BYTES, u)], host);
      }
      atomicAdd(&s.step_ctr[ctr_at(C_HBM_BYTES, u)], (unsigned long long)hbm);
      atomicAdd(&s.total_ctr[ctr_at(C_HBM_BYTES, u)], (unsigned long long)hbm);
    }
  }
  cp_async_wait<0>();  // R staged (also before any exit: no copy may outlive the CTA)
  __syncthreads();
  int any = 0;
  for (int w = 0; w < nu; ++w) any |= s_dec[w] != CLO_DEC_HIT;
  if (!any) {  // uniform over the CTA
    if (tid == 0 && s.timeline) atomicMax(&s.timeline[TL_DEC_END], global_timer_ns());
    return;
  }

  // 2. query codes: thread (slot, j) computes bit j of rows slot, slot + 4, ... (rows of
  //    reused units are computed but neither certified nor stored)
  const int nrows = nu * G;
  const int j = tid & 127, slot = tid >> 7;
  float acc[M], aab[M];
#pragma unroll
  for (int m = 0; m < M; ++m) acc[m] = aab[m] = 0.f;
  const float* xrow = xs + slot * M;
  for (int i = 0; i < d; ++i) {
    const float r = bf16_bits_to_f32(Rs[i * 128 + j]);
    const float ar = fabsf(r);
#pragma unroll
    for (int m = 0; m < M; m += 4) {
      const float4 x = *reinterpret_cast<const float4*>(xrow + i * XW + m);
      acc[m] = fmaf(x.x, r, acc[m]);
      aab[m] = fmaf(fabsf(x.x), ar, aab[m]);
      acc[m + 1] = fmaf(x.y, r, acc[m + 1]);
      aab[m + 1] = fmaf(fabsf(x.y), ar, aab[m + 1]);
      acc[m + 2] = fmaf(x.z, r, acc[m + 2]);
      aab[m + 2] = fmaf(fabsf(x.z), ar, aab[m + 2]);
      acc[m + 3] = fmaf(x.w, r, acc[m + 3]);
      aab[m + 3] = fmaf(fabsf(x.w), ar, aab[m + 3]);
    }
  }
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const int row = m * kHashSlots + slot;
    if (row >= nrows) break;                         // uniform over the warp
    if (s_dec[row / G] == CLO_DEC_HIT) continue;     // uniform over the warp
    bool bit;
    if (sign_certified_f32(acc[m], aab[m], d))
      bit = acc[m] > 0.f;
    else
      bit = hash_bit_slow(StridedF32{xrow + m, XW}, StridedBF16{Rs + j, 128}, d);
    const uint32_t wbits = __ballot_sync(0xffffffffu, bit);
    if (lane == 0) words[row][j >> 5] = wbits;
  }
  __syncthreads();
  for (int r = tid; r < nrows; r += kDecideThreads) {
    const int w = r / G, g = r % G;
    if (s_dec[w] == CLO_DEC_HIT) continue;
    s.qcodes[((int64_t)l * s.B + b0 + w) * s.Hq + (int64_t)h * G + g] =
        make_uint4(words[r][0], words[r][1], words[r][2], words[r][3]);
  }
  if (tid == 0 && s.timeline) atomicMax(&s.timeline[TL_DEC_END], global_timer_ns());
}

// End of warm-up: s_hat = mean adjacent-step cosine, tau = s_hat - offset, and the
// n_persist lowest-s_hat heads of each layer (ties: lower head index) persistent.
__global__ void k_finish_warmup(DevState s, int W, float tau_offset, int n_persist) {
  const int l = blockIdx.x * blockDim.x + threadIdx.x;
  if (l >= s.L) return;
  const double npairs = (double)s.B * (double)(W - 1);
  for (int h = 0; h < s.Hkv; ++h) {
    const int lh = l * s.Hkv + h;
    const double sh = s.shat_sum[lh] / npairs;
    s.shat[lh] = sh;
    s.tau[lh] = (float)(sh - (double)tau_offset);
    s.persist[lh] = 0;
    s.persist_slot[lh] = -1;
  }
  for (int p = 0; p < n_persist; ++p) {
    int best = -1;
    for (int h = 0; h < s.Hkv; ++h) {
      const int lh = l * s.Hkv + h;
      if (s.persist[lh]) continue;
      if (best < 0 || s.shat[lh] < s.shat[l * s.Hkv + best]) best = h;
    }
    if (best >= 0) s.persist[l * s.Hkv + best] = 1;
  }
  int p = 0;
  for (int h = 0; h < s.Hkv; ++h)
    if (s.persist[l * s.Hkv + h]) s.persist_slot[l * s.Hkv + h] = p++;
}

}  // namespace

template <int M>
cudaError_t launch_decide_m(const DevState& s, const uint16_t* q, int64_t step, int warmup_active, cudaStream_t st) {
  const int upc = units_per_cta(s.G, s.B, s.decide_rows);
  const unsigned grid = (unsigned)((s.l1 - s.l0) * s.Hkv * ((s.B + upc - 1) / upc));
  const size_t smem = (size_t)s.d * 128 * 2 + (size_t)s.d * kHashSlots * M * 4;
  cudaError_t e = cudaFuncSetAttribute(k_decide<M>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k_decide<M><<<grid, kDecideThreads, smem, st>>>(s, q, step, warmup_active);
  return cudaGetLastError();
}

cudaError_t launch_decide(const DevState& s, const uint16_t* q, int64_t step, int warmup_active,
                          cudaStream_t st) {
  // query rows per thread slot: enough for all rows of one CTA (at most 32 rows)
  const int rows = units_per_cta(s.G, s.B, s.decide_rows) * s.G;
  const int per_slot = (rows + kHashSlots - 1) / kHashSlots;
  if (per_slot <= 4) return launch_decide_m<4>(s, q, step, warmup_active, st);
  return launch_decide_m<8>(s, q, step, warmup_active, st);
}

cudaError_t launch_finish_warmup(const DevState& s, int W, float tau_offset, int n_persist, cudaStream_t st) {
  k_finish_warmup<<<(s.L + 63) / 64, 64, 0, st>>>(s, W, tau_offset, n_persist);
  return cudaGetLastError();
}

}  // namespace clo
