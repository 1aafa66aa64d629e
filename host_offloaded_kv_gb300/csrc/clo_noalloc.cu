// Allocation-free split-K sparse decode attention (clo_sparse_attention_noalloc).
//
// The paper has no counterpart to this entry point.  It exists for callers that
// may not allocate device memory at all: an inference server or plugin host that
// hands every kernel a pre-planned memory budget and forbids allocations behind
// its back, a real-time decode loop that cannot afford the device-wide
// synchronisation cudaMalloc/cudaFree can cause, or code running where the
// allocator is unavailable.  Such callers pass only inputs and outputs; the
// split-K partials and the per-group combine counters live in one file-scope
// device array of fixed size that every GPU loading this library keeps until the
// process exits.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "clo.h"
#include "clo_internal.cuh"

namespace clo {
namespace {

constexpr int kNaThreads = 128;
constexpr int kNaTile = 32;
constexpr int kNaSplitRows = 256;
constexpr int kNaMaxGroups = 4096;                        // combine counters
constexpr int64_t kNaPartWords = 2 * 1024 * 1024;         // 8 MiB of fp32 split partials
constexpr int64_t kNaWords = kNaMaxGroups + kNaPartWords;  // counters first, then partials
constexpr int kNaMaxDevices = 64;

// The scratch: [kNaMaxGroups] uint32 combine counters, then fp32 partials
// [group][split][G][d + 2] = {running max, running sum, acc[d]}.
static __device__ __align__(256) uint32_t g_noalloc_scratch[kNaWords];

template <int D>
__global__ void __launch_bounds__(kNaThreads) k_attend_noalloc(const uint16_t* __restrict__ q,
                                                                const uint16_t* __restrict__ rows_g, float* __restrict__ out,
                                                                int G, int64_t k, int nsplit, uint32_t* scratch) {
  constexpr int VPR = D / 4;
  constexpr int ROWW = 2 * D + 8;
  constexpr int NG = kNaThreads / D;
  __shared__ __align__(16) float qs[kMaxG][D];
  __shared__ __align__(16) uint16_t rows[kNaTile][ROWW];
  __shared__ float sc[kMaxG][kNaTile];
  __shared__ float m_run[kMaxG], l_run[kMaxG], alpha[kMaxG];
  __shared__ float red[NG > 1 ? NG : 1][kMaxG][D];
  __shared__ int s_last;

  uint32_t* done = scratch;
  float* part_all = reinterpret_cast<float*>(scratch + kNaMaxGroups);
  const int64_t grp = blockIdx.y;
  const int split = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t r0 = (int64_t)split * kNaSplitRows;
  const int64_t r1 = (r0 + kNaSplitRows < k) ? r0 + kNaSplitRows : k;
  const uint4* src = reinterpret_cast<const uint4*>(rows_g) + grp * k * VPR;

  const float qscale = 1.4426950408889634f * rsqrtf((float)D);
  const uint16_t* qg = q + grp * G * D;
  for (int e = tid; e < G * D; e += kNaThreads) qs[e / D][e % D] = bf16_bits_to_f32(qg[e]) * qscale;
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

  for (int64_t rb = r0; rb < r1; rb += kNaTile) {
    const int nrows = (int)((r1 - rb) < kNaTile ? (r1 - rb) : kNaTile);
    for (int e = tid; e < nrows * VPR; e += kNaThreads) {
      const int r = e / VPR, c = e % VPR;
      cp_async16(&rows[r][c * 8], src + (rb + r) * VPR + c);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    for (int p = tid; p < G * kNaTile; p += kNaThreads) {
      const int g = p / kNaTile, r = p % kNaTile;
      float dot = -INFINITY;
      if (r < nrows) {
        dot = 0.f;
        const uint4* kr = reinterpret_cast<const uint4*>(&rows[r][0]);
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
    for (int g = warp; g < G; g += kNaThreads / 32) {
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

  if (NG > 1) {
#pragma unroll
    for (int g = 0; g < kMaxG; ++g)
      if (g < G) red[rg][g][dj] = acc[g];
    __syncthreads();
  }
  float* part = part_all + ((grp * nsplit + split) * G) * (D + 2);
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
    const uint32_t prev = atomicAdd(&done[grp], 1u);
    s_last = (prev == (uint32_t)nsplit - 1u);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const float* pu = part_all + (grp * nsplit) * G * (D + 2);
  float* og = out + grp * G * D;
  for (int e = tid; e < G * D; e += kNaThreads) {
    const int g = e / D, j = e % D;
    float M = -INFINITY;
    for (int sp = 0; sp < nsplit; ++sp) M = fmaxf(M, __ldcg(pu + (sp * G + g) * (D + 2)));
    float L = 0.f, O = 0.f;
    for (int sp = 0; sp < nsplit; ++sp) {
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
  if (tid == 0) done[grp] = 0u;
}

std::mutex g_setup_mu;
uint32_t* g_scratch_dev[kNaMaxDevices] = {};

}  // namespace
}  // namespace clo

using namespace clo;

extern "C" CLO_API clo_status clo_sparse_attention_noalloc(const void* q, const void* rows, float* out,
                                                           int32_t n_groups, int32_t group_size, int32_t head_dim,
                                                           int64_t k, void* stream) {
  // Errors are reported through the same thread-local text as the other calls.
  auto fail = [](clo_status st, const std::string& m) {
    set_last_error_text(m.c_str());
    return st;
  };
  if (!q || !rows || !out) return fail(CLO_ERR_INVALID, "clo_sparse_attention_noalloc: null pointer");
  if (n_groups < 1 || group_size < 1 || group_size > kMaxG || (head_dim != 64 && head_dim != 128) || k < 1)
    return fail(CLO_ERR_INVALID, "clo_sparse_attention_noalloc: need n_groups >= 1, 1 <= group_size <= 8, "
                                 "head_dim 64 or 128, k >= 1");
  // rows are read with 16-byte asynchronous copies, q as bf16 and out as fp32 words
  if ((reinterpret_cast<uintptr_t>(rows) & 15u) != 0 || (reinterpret_cast<uintptr_t>(q) & 1u) != 0 ||
      (reinterpret_cast<uintptr_t>(out) & 3u) != 0)
    return fail(CLO_ERR_INVALID, "clo_sparse_attention_noalloc: rows must be 16-byte aligned, q 2-byte and out "
                                 "4-byte aligned");
  const int64_t nsplit = (k + kNaSplitRows - 1) / kNaSplitRows;
  const int64_t need = (int64_t)n_groups * nsplit * group_size * (head_dim + 2);
  if (n_groups > kNaMaxGroups || need > kNaPartWords)
    return fail(CLO_ERR_INVALID,
                "clo_sparse_attention_noalloc: size beyond the fixed scratch: n_groups <= " +
                    std::to_string(kNaMaxGroups) + " and n_groups * ceil(k/256) * group_size * (head_dim+2) <= " +
                    std::to_string(kNaPartWords) + " (asked " + std::to_string(need) + ")");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(CLO_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= kNaMaxDevices) return fail(CLO_ERR_INVALID, "device ordinal beyond 63");
  uint32_t* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_dev[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess)
        return fail(CLO_ERR_CUDA, std::string("cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(e));
      g_scratch_dev[dev] = static_cast<uint32_t*>(p);
    }
    scratch = g_scratch_dev[dev];
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the combine counters must start at zero on every call
  e = cudaMemsetAsync(scratch, 0, sizeof(uint32_t) * (size_t)n_groups, st);
  if (e != cudaSuccess) return fail(CLO_ERR_CUDA, std::string("cudaMemsetAsync: ") + cudaGetErrorString(e));
  dim3 grid((unsigned)nsplit, (unsigned)n_groups);
  if (head_dim == 128)
    k_attend_noalloc<128><<<grid, kNaThreads, 0, st>>>(static_cast<const uint16_t*>(q),
                                                       static_cast<const uint16_t*>(rows), out, group_size, k,
                                                       (int)nsplit, scratch);
  else
    k_attend_noalloc<64><<<grid, kNaThreads, 0, st>>>(static_cast<const uint16_t*>(q),
                                                      static_cast<const uint16_t*>(rows), out, group_size, k,
                                                      (int)nsplit, scratch);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(CLO_ERR_CUDA, std::string("launch: ") + cudaGetErrorString(e));
  return CLO_OK;
}
