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

// Token sources of the key hash: the prefill rows of one (layer, sequence), or one new
// token of every sequence of one layer (its position: the sequence's current length).
struct PrefillKeys {
  const uint16_t* K;  // bf16 [n][Hkv][d]
  int l, b;
  int64_t t0, n;
  __device__ int layer() const { return l; }
  __device__ bool valid(int64_t t) const { return t < n; }
  __device__ const uint16_t* row(const DevState& s, int64_t t, int h) const { return K + (t * s.Hkv + h) * s.d; }
  __device__ int64_t code_at(const DevState& s, int64_t t, int h) const {
    return unit_of(s, l, b, h) * s.Nmax + t0 + t;
  }
};
struct StepKeys {
  const uint16_t* K;  // bf16 [L][B][Hkv][d]: token t of a tile is sequence t of layer blockIdx.z
  __device__ int layer() const { return (int)blockIdx.z; }
  __device__ bool valid(int64_t t) const { return true; }
  __device__ const uint16_t* row(const DevState& s, int64_t t, int h) const {
    return K + (((int64_t)blockIdx.z * s.B + t) * s.Hkv + h) * s.d;
  }
  __device__ int64_t code_at(const DevState& s, int64_t t, int h) const {
    return unit_of(s, (int)blockIdx.z, (int)t, h) * s.Nmax + s.ntok[t];
  }
};

// codes[...] = hash(key) for the tokens of a source, tiles of 64 tokens per CTA, kv head
// blockIdx.y; n_tok tokens in all.
template <class Src>
__global__ void __launch_bounds__(kHashThreads) k_hash_keys(DevState s, Src src, int64_t n_tok) {
  extern __shared__ __align__(16) float sm[];
  const int d = s.d;
  const int h = blockIdx.y;
  const int l = src.layer();
  float* Rs = sm;                 // [d][128]
  float* Ks = sm + d * 128;       // [64][d]
  const uint16_t* Rg = s.R + ((int64_t)l * s.Hkv + h) * d * 128;
  for (int e = threadIdx.x; e < d * 128; e += blockDim.x) Rs[e] = bf16_bits_to_f32(Rg[e]);
  const int64_t tile0 = (int64_t)blockIdx.x * kHashTokTile;
  for (int e = threadIdx.x; e < kHashTokTile * d; e += blockDim.x) {
    const int tt = e / d, i = e - tt * d;
    const int64_t t = tile0 + tt;
    Ks[e] = (t < n_tok && src.valid(t)) ? bf16_bits_to_f32(src.row(s, t, h)[i]) : 0.0f;
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
#pragma unroll
  for (int tt = 0; tt < 8; ++tt) {
    const int64_t t = tile0 + warp * 8 + tt;
    if (!(t < n_tok && src.valid(t))) continue;  // padding of the tile (uniform over the warp)
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
    if (lane == 0) s.codes[src.code_at(s, t, h)] = make_uint4(w[0], w[1], w[2], w[3]);
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
// Quantises one 64-channel group (values at src, 16-byte aligned) into record rec:
//   mn, mx of the group (a zero minimum as +0); scale = (mx - mn) / (2^BITS - 1);
//   q = clamp(rint((x - mn) / scale), 0, 2^BITS - 1), 0 when scale is 0
// (every operation fp32, rounded to nearest).  The codes go to the record, (scale, mn)
// to the token's parameters in HBM; resident (or null) gets the dequantised values.
template <int D, int BITS>
__device__ __forceinline__ void quantise_group(const uint16_t* src, unsigned char* rec, float2* params, int kv, int g,
                                               uint16_t* resident) {
  constexpr int NG = D / 64;  // groups per row
  constexpr float kLevels = (float)((1 << BITS) - 1);
  float x[64];
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    const uint4 w = reinterpret_cast<const uint4*>(src)[v];
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
  uint4* codes = reinterpret_cast<uint4*>(rec + (size_t)(kv * NG + g) * 64 * BITS / 8);
#pragma unroll
  for (int v = 0; v < BITS / 2; ++v)
    codes[v] = make_uint4(words[4 * v], words[4 * v + 1], words[4 * v + 2], words[4 * v + 3]);
  params[kv * NG + g] = make_float2(scale, mn);
  if (resident) {
    uint4* dst = reinterpret_cast<uint4*>(resident);
#pragma unroll
    for (int v = 0; v < BITS / 2; ++v)
      dequant_vec<BITS>(make_uint4(words[4 * v], words[4 * v + 1], words[4 * v + 2], words[4 * v + 3]), scale, mn,
                        dst + v * (16 / BITS));
  }
}

// Quantised pool write of prefill rows: one thread per (token, kv head, K or V, group).
template <int D, int BITS>
__global__ void k_pool_write_q(DevState s, int l, int b, int64_t t0, int64_t n, const uint16_t* __restrict__ K,
                               const uint16_t* __restrict__ V) {
  using Q = QRec<D, BITS>;
  constexpr int NG = D / 64;
  const int64_t total = n * s.Hkv * 2 * NG;
  unsigned char* pool = reinterpret_cast<unsigned char*>(const_cast<uint16_t*>(s.pool));
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
    const int g = (int)(e % NG);
    const int kv = (int)((e / NG) % 2);
    const int h = (int)((e / (2 * NG)) % s.Hkv);
    const int64_t t = e / (2 * (int64_t)NG * s.Hkv);
    const uint16_t* src = (kv == 0 ? K : V) + (t * s.Hkv + h) * D + 64 * g;
    const int64_t u = unit_of(s, l, b, h);
    const int p = s.persist_slot[l * s.Hkv + h];
    uint16_t* res = nullptr;
    if (p >= 0 && s.resident != nullptr)
      res = s.resident + ((((int64_t)l * s.B + b) * s.P + p) * s.Nmax + t0 + t) * 2 * D + kv * D + 64 * g;
    quantise_group<D, BITS>(src, pool + (u * s.Nmax + t0 + t) * Q::kBytes, s.qparams + (u * s.Nmax + t0 + t) * Q::kGroups,
                            kv, g, res);
  }
}

// One new token per (layer, sequence) at the sequence's current length: K, V bf16
// [L][B][Hkv][d].  bf16 pools: one thread per 16-byte vector; quantised pools: one
// thread per 64-channel group.  Persistent heads also get their resident row.
__global__ void k_step_pool_write(DevState s, const uint16_t* __restrict__ K, const uint16_t* __restrict__ V) {
  const int d = s.d;
  const int vpr = d / 8;
  const int64_t total = (int64_t)s.L * s.B * s.Hkv * 2 * vpr;
  uint4* pool = reinterpret_cast<uint4*>(const_cast<uint16_t*>(s.pool));
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
    const int v = (int)(e % vpr);
    const int kv = (int)((e / vpr) % 2);
    const int64_t lbh = e / (2 * vpr);  // (l * B + b) * Hkv + h = the unit
    const int h = (int)(lbh % s.Hkv);
    const int b = (int)((lbh / s.Hkv) % s.B);
    const int l = (int)(lbh / ((int64_t)s.Hkv * s.B));
    const int64_t t = s.ntok[b];
    const uint4 val = reinterpret_cast<const uint4*>((kv == 0 ? K : V) + lbh * d)[v];
    pool[(lbh * s.Nmax + t) * (2 * vpr) + kv * vpr + v] = val;
    const int p = s.persist_slot[l * s.Hkv + h];
    if (p >= 0 && s.resident != nullptr) {
      const int64_t ru = ((int64_t)l * s.B + b) * s.P + p;
      reinterpret_cast<uint4*>(s.resident)[(ru * s.Nmax + t) * (2 * vpr) + kv * vpr + v] = val;
    }
  }
}

template <int D, int BITS>
__global__ void k_step_pool_write_q(DevState s, const uint16_t* __restrict__ K, const uint16_t* __restrict__ V) {
  using Q = QRec<D, BITS>;
  constexpr int NG = D / 64;
  const int64_t total = (int64_t)s.L * s.B * s.Hkv * 2 * NG;
  unsigned char* pool = reinterpret_cast<unsigned char*>(const_cast<uint16_t*>(s.pool));
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
    const int g = (int)(e % NG);
    const int kv = (int)((e / NG) % 2);
    const int64_t lbh = e / (2 * NG);
    const int h = (int)(lbh % s.Hkv);
    const int b = (int)((lbh / s.Hkv) % s.B);
    const int l = (int)(lbh / ((int64_t)s.Hkv * s.B));
    const int64_t t = s.ntok[b];
    const int p = s.persist_slot[l * s.Hkv + h];
    uint16_t* res = nullptr;
    if (p >= 0 && s.resident != nullptr)
      res = s.resident + ((((int64_t)l * s.B + b) * s.P + p) * s.Nmax + t) * 2 * D + kv * D + 64 * g;
    quantise_group<D, BITS>((kv == 0 ? K : V) + lbh * D + 64 * g, pool + (lbh * s.Nmax + t) * Q::kBytes,
                            s.qparams + (lbh * s.Nmax + t) * Q::kGroups, kv, g, res);
  }
}

// After a step's append: N_b += 1 and k_b = top-k count of the new length (the same
// rule as at offload: min(topk, N), or ceil(ratio * N) as one double product, in [1, N]).
__global__ void k_step_lengths(DevState s, int64_t topk, double ratio) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= s.B) return;
  int64_t* ntok = const_cast<int64_t*>(s.ntok);
  const int64_t N = ntok[b] + 1;
  ntok[b] = N;
  int64_t k;
  if (topk > 0) {
    k = topk < N ? topk : N;
  } else {
    k = (int64_t)ceil(ratio * (double)N);
    k = k < 1 ? 1 : (k > N ? N : k);
  }
  const_cast<int32_t*>(s.kcount)[b] = (int32_t)k;
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
  cudaError_t e = cudaFuncSetAttribute(k_hash_keys<PrefillKeys>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((n + kHashTokTile - 1) / kHashTokTile), (unsigned)s.Hkv);
  k_hash_keys<PrefillKeys><<<grid, kHashThreads, smem, st>>>(s, PrefillKeys{kdev, l, b, t0, n}, n);
  return cudaGetLastError();
}

cudaError_t launch_append_step(const DevState& s, const uint16_t* kdev, const uint16_t* vdev, int64_t topk,
                               double ratio, cudaStream_t st) {
  // the new keys' hash codes (one CTA per tile of sequences, kv head and layer)
  const size_t smem = (size_t)(s.d * 128 + kHashTokTile * s.d) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(k_hash_keys<StepKeys>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((s.B + kHashTokTile - 1) / kHashTokTile), (unsigned)s.Hkv, (unsigned)s.L);
  k_hash_keys<StepKeys><<<grid, kHashThreads, smem, st>>>(s, StepKeys{kdev}, (int64_t)s.B);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // the new records
  const int64_t per = s.kv_bits == 16 ? (int64_t)s.d / 8 : (int64_t)s.d / 64;
  const int64_t total = (int64_t)s.L * s.B * s.Hkv * 2 * per;
  const unsigned blocks = (unsigned)((total + 127) / 128 < 152 * 16 ? (total + 127) / 128 : 152 * 16);
  if (s.kv_bits == 16)
    k_step_pool_write<<<blocks, 128, 0, st>>>(s, kdev, vdev);
  else if (s.d == 128)
    s.kv_bits == 4 ? k_step_pool_write_q<128, 4><<<blocks, 128, 0, st>>>(s, kdev, vdev)
                   : k_step_pool_write_q<128, 2><<<blocks, 128, 0, st>>>(s, kdev, vdev);
  else
    s.kv_bits == 4 ? k_step_pool_write_q<64, 4><<<blocks, 128, 0, st>>>(s, kdev, vdev)
                   : k_step_pool_write_q<64, 2><<<blocks, 128, 0, st>>>(s, kdev, vdev);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // then the lengths (both kernels above read the old ones)
  k_step_lengths<<<(s.B + 127) / 128, 128, 0, st>>>(s, topk, ratio);
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
