// Prefill offload (KV produced once at prefill and offloaded: "CLO (2511.14510) -
// L3 Per-Paper Synthesis", section 5.7): K/V rows go to the pinned host pool, and
// each key's 128-bit hash code is computed once and kept in HBM.
#include "clo_hash.cuh"
#include "clo_internal.cuh"

namespace clo {

namespace {

struct StridedF32 {
  const float* p;
  int stride;
  __device__ float operator()(int i) const { return p[i * stride]; }
};

constexpr int kHashTokTile = 64;   // tokens per CTA
constexpr int kHashThreads = 256;  // 8 warps x 8 tokens

// codes[u(l,b,h)][t0 + t] = hash(K[t][h]) for t in [0, n); K: bf16 [n][Hkv][d] in HBM.
__global__ void __launch_bounds__(kHashThreads) k_hash_keys(DevState s, int l, int b, int64_t t0, int64_t n,
                                                             const uint16_t* __restrict__ K) {
  extern __shared__ __align__(16) float sm[];
  const int d = s.d;
  const int h = blockIdx.y;
  float* Rs = sm;                 // [d][128]
  float* Ks = sm + d * 128;       // [64][d]
  const uint16_t* Rg = s.R + ((int64_t)l * s.Hkv + h) * d * 128;
  for (int e = threadIdx.x; e < d * 128; e += blockDim.x) Rs[e] = bf16_bits_to_f32(Rg[e]);
  const int64_t tile0 = (int64_t)blockIdx.x * kHashTokTile;
  for (int e = threadIdx.x; e < kHashTokTile * d; e += blockDim.x) {
    const int tt = e / d, i = e - tt * d;
    const int64_t t = tile0 + tt;
    Ks[e] = (t < n) ? bf16_bits_to_f32(K[(t * s.Hkv + h) * d + i]) : 0.0f;
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* xw = Ks + warp * 8 * d;
  float acc[8][4], aab[8][4];
#pragma unroll
  for (int tt = 0; tt < 8; ++tt)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[tt][c] = aab[tt][c] = 0.0f;
  for (int i = 0; i < d; ++i) {
    float r[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) r[c] = Rs[i * 128 + lane + 32 * c];
#pragma unroll
    for (int tt = 0; tt < 8; ++tt) {
      const float x = xw[tt * d + i];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        acc[tt][c] = fmaf(x, r[c], acc[tt][c]);
        aab[tt][c] = fmaf(fabsf(x), fabsf(r[c]), aab[tt][c]);
      }
    }
  }
  const int64_t u = unit_of(s, l, b, h);
#pragma unroll
  for (int tt = 0; tt < 8; ++tt) {
    uint32_t w[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      bool bit;
      if (sign_certified_f32(acc[tt][c], aab[tt][c], d))
        bit = acc[tt][c] > 0.0f;
      else
        bit = hash_bit_slow(StridedF32{xw + tt * d, 1}, StridedF32{Rs + lane + 32 * c, 128}, d);
      w[c] = __ballot_sync(0xffffffffu, bit);
    }
    const int64_t t = tile0 + warp * 8 + tt;
    if (lane == 0 && t < n) s.codes[u * s.Nmax + t0 + t] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// pool[u][t0 + t] = K[t][h] | V[t][h]; also the resident copy when the head is
// persistent.  One thread per 16-byte vector of a record.
__global__ void k_pool_write(DevState s, int l, int b, int64_t t0, int64_t n, const uint16_t* __restrict__ K,
                             const uint16_t* __restrict__ V) {
  const int d = s.d;
  const int vpr = d / 8;  // uint4 per K (or V) row
  const int64_t total = n * s.Hkv * 2 * vpr;
  uint4* pool = reinterpret_cast<uint4*>(const_cast<uint16_t*>(s.pool));
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
    const int v = (int)(e % vpr);
    const int kv = (int)((e / vpr) % 2);
    const int h = (int)((e / (2 * vpr)) % s.Hkv);
    const int64_t t = e / (2 * (int64_t)vpr * s.Hkv);
    const uint16_t* src = (kv == 0 ? K : V) + (t * s.Hkv + h) * d;
    const uint4 val = reinterpret_cast<const uint4*>(src)[v];
    const int64_t u = unit_of(s, l, b, h);
    const int64_t rec = (u * s.Nmax + t0 + t) * (2 * vpr) + kv * vpr + v;
    pool[rec] = val;
    const int p = s.persist_slot[l * s.Hkv + h];
    if (p >= 0 && s.resident != nullptr) {
      const int64_t ru = ((int64_t)l * s.B + b) * s.P + p;
      reinterpret_cast<uint4*>(s.resident)[(ru * s.Nmax + t0 + t) * (2 * vpr) + kv * vpr + v] = val;
    }
  }
}

// Quantised pool write: one thread per (token, kv head, K or V, 64-channel group).
//   mn, mx of the group; scale = (mx - mn) / (2^BITS - 1);
//   q = clamp(rint((x - mn) / scale), 0, 2^BITS - 1), 0 when scale is 0
// (every operation fp32, rounded to nearest).  The codes and (scale, mn) go to the
// token's record; a persistent head's resident copy gets the dequantised values.
template <int D, int BITS>
__global__ void k_pool_write_q(DevState s, int l, int b, int64_t t0, int64_t n, const uint16_t* __restrict__ K,
                               const uint16_t* __restrict__ V) {
  using Q = QRec<D, BITS>;
  constexpr int NG = D / 64;  // groups per row
  constexpr float kLevels = (float)((1 << BITS) - 1);
  const int64_t total = n * s.Hkv * 2 * NG;
  unsigned char* pool = reinterpret_cast<unsigned char*>(const_cast<uint16_t*>(s.pool));
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
    const int g = (int)(e % NG);
    const int kv = (int)((e / NG) % 2);
    const int h = (int)((e / (2 * NG)) % s.Hkv);
    const int64_t t = e / (2 * (int64_t)NG * s.Hkv);
    const uint4* src = reinterpret_cast<const uint4*>((kv == 0 ? K : V) + (t * s.Hkv + h) * D + 64 * g);
    float x[64];
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      const uint4 w = src[v];
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[8 * v + 2 * i] = bf16_bits_to_f32(ww[i] & 0xffffu);
        x[8 * v + 2 * i + 1] = bf16_bits_to_f32(ww[i] >> 16);
      }
    }
    float mn = x[0], mx = x[0];
#pragma unroll
    for (int i = 1; i < 64; ++i) {
      mn = fminf(mn, x[i]);
      mx = fmaxf(mx, x[i]);
    }
    mn = __fadd_rn(mn, 0.f);  // a zero minimum is +0 whichever zero fminf returned
    const float scale = __fdiv_rn(__fsub_rn(mx, mn), kLevels);
    uint32_t words[2 * BITS];  // 64 codes
#pragma unroll
    for (int w = 0; w < 2 * BITS; ++w) words[w] = 0u;
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      float q = 0.f;
      if (scale > 0.f) q = fminf(fmaxf(rintf(__fdiv_rn(__fsub_rn(x[i], mn), scale)), 0.f), kLevels);
      words[i / (32 / BITS)] |= (uint32_t)q << (BITS * (i % (32 / BITS)));
    }
    const int64_t u = unit_of(s, l, b, h);
    unsigned char* rec = pool + (u * s.Nmax + t0 + t) * Q::kBytes;
    uint4* codes = reinterpret_cast<uint4*>(rec + (size_t)(kv * NG + g) * 64 * BITS / 8);
#pragma unroll
    for (int v = 0; v < BITS / 2; ++v)
      codes[v] = make_uint4(words[4 * v], words[4 * v + 1], words[4 * v + 2], words[4 * v + 3]);
    *reinterpret_cast<float2*>(rec + Q::kParamOff + 8 * (kv * NG + g)) = make_float2(scale, mn);
    const int p = s.persist_slot[l * s.Hkv + h];
    if (p >= 0 && s.resident != nullptr) {
      const int64_t ru = ((int64_t)l * s.B + b) * s.P + p;
      uint4* dst = reinterpret_cast<uint4*>(s.resident + (ru * s.Nmax + t0 + t) * 2 * D + kv * D + 64 * g);
#pragma unroll
      for (int v = 0; v < BITS / 2; ++v)
        dequant_vec<BITS>(make_uint4(words[4 * v], words[4 * v + 1], words[4 * v + 2], words[4 * v + 3]), scale, mn,
                          dst + v * (16 / BITS));
    }
  }
}

template <int D, int BITS>
cudaError_t launch_pool_write_q(const DevState& s, int l, int b, int64_t t0, int64_t n, const uint16_t* kdev,
                                const uint16_t* vdev, cudaStream_t st) {
  const int64_t total = n * s.Hkv * 2 * (D / 64);
  const int64_t blocks = (total + 127) / 128;
  k_pool_write_q<D, BITS><<<(unsigned)(blocks < 152 * 32 ? blocks : 152 * 32), 128, 0, st>>>(s, l, b, t0, n, kdev,
                                                                                            vdev);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_hash_keys(const DevState& s, int l, int b, int64_t t0, int64_t n, const uint16_t* kdev,
                             cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const size_t smem = (size_t)(s.d * 128 + kHashTokTile * s.d) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(k_hash_keys, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((n + kHashTokTile - 1) / kHashTokTile), (unsigned)s.Hkv);
  k_hash_keys<<<grid, kHashThreads, smem, st>>>(s, l, b, t0, n, kdev);
  return cudaGetLastError();
}

cudaError_t launch_pool_write(const DevState& s, int l, int b, int64_t t0, int64_t n, const uint16_t* kdev,
                              const uint16_t* vdev, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  if (s.kv_bits != 16) {
    if (s.d == 128) return s.kv_bits == 4 ? launch_pool_write_q<128, 4>(s, l, b, t0, n, kdev, vdev, st)
                                           : launch_pool_write_q<128, 2>(s, l, b, t0, n, kdev, vdev, st);
    return s.kv_bits == 4 ? launch_pool_write_q<64, 4>(s, l, b, t0, n, kdev, vdev, st)
                          : launch_pool_write_q<64, 2>(s, l, b, t0, n, kdev, vdev, st);
  }
  const int64_t total = n * s.Hkv * 2 * (s.d / 8);
  const int64_t blocks = (total + 255) / 256;
  k_pool_write<<<(unsigned)(blocks < 152 * 32 ? blocks : 152 * 32), 256, 0, st>>>(s, l, b, t0, n, kdev, vdev);
  return cudaGetLastError();
}

}  // namespace clo
