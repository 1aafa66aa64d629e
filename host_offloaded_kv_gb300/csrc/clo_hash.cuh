// 128-bit sign hash of bf16 vectors with an exactly decided sign.
//
// Bit j of the code of x is 1 iff the exact real value of sum_i x_i * R_ij is
// greater than zero (R: the per-(layer, kv head) d x 128 bf16 projection).  The
// hash-code scorer is the HATA top-k scorer CLO integrates ("CLO (2511.14510) -
// L3 Per-Paper Synthesis", section 3.2); the sign code is the reading used here.
//
// Three tiers, each exact about the sign it returns:
//   1. fp32 FMA chain s and the chain a = sum |x_i||R_ij|.  Products of two bf16
//      are exact in fp32 and the FMA chain's error (underflow included) is below
//      T32 = n * 2^-22 * a + n * 2^-147, so |s| > T32 fixes the sign.
//   2. fp64: every product is exact and no partial sum can underflow (all are
//      multiples of 2^-266); error below T64 = n * 2^-51 * a64.
//   3. fixed point: each product is an integer (< 2^16) times 2^(e - 266) with
//      0 <= e <= 506, accumulated into 17 int64 limbs of 32 bits; exact.
// Inputs must be finite; a non-finite element contributes nothing in tier 3.
#pragma once

#include "clo_internal.cuh"

namespace clo {

__device__ __forceinline__ bool sign_certified_f32(float s, float a, int n) {
  const float bound = (float)n * (a * 2.384185791015625e-7f) + (float)n * 5.605193857299268e-45f;
  return fabsf(s) > bound;
}

// Tier 3: exact sign of sum_i x_i * r_i for bf16 bit patterns.
static __device__ __noinline__ int exact_dot_sign_bits(const uint32_t* xb, const uint32_t* rb, int n) {
  long long acc[17];
#pragma unroll
  for (int i = 0; i < 17; ++i) acc[i] = 0;
  for (int i = 0; i < n; ++i) {
    const uint32_t a = xb[i] & 0xffffu, b = rb[i] & 0xffffu;
    const uint32_t ea = (a >> 7) & 0xffu, eb = (b >> 7) & 0xffu;
    if (ea == 0xffu || eb == 0xffu) continue;
    const uint32_t ma = (a & 0x7fu) | (ea ? 0x80u : 0u);
    const uint32_t mb = (b & 0x7fu) | (eb ? 0x80u : 0u);
    if (ma == 0u || mb == 0u) continue;
    // value = m * 2^(max(E,1) - 134); product exponent + 266 in [0, 506]
    const int shift = (int)(ea ? ea : 1u) + (int)(eb ? eb : 1u) - 268 + 266;
    long long v = (long long)(ma * mb) << (shift & 31);
    if ((a ^ b) & 0x8000u) v = -v;
    acc[shift >> 5] += v;
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const long long c = acc[i] >> 32;  // floor division by 2^32
    acc[i] -= c * 4294967296LL;
    acc[i + 1] += c;
  }
  if (acc[16] != 0) return acc[16] > 0 ? 1 : -1;
  for (int i = 0; i < 16; ++i)
    if (acc[i] != 0) return 1;
  return 0;
}

// Tiers 2 and 3 for one (vector, column): x and r given as float values that are
// exactly bf16 (strided accessors), n <= 256.
template <class XAt, class RAt>
__device__ __noinline__ bool hash_bit_slow(XAt x, RAt r, int n) {
  double s = 0.0, a = 0.0;
  for (int i = 0; i < n; ++i) {
    const double p = (double)x(i) * (double)r(i);
    s += p;
    a += fabs(p);
  }
  if (fabs(s) > (double)n * 4.440892098500626e-16 * a) return s > 0.0;
  uint32_t xb[256], rb[256];
  for (int i = 0; i < n; ++i) {
    xb[i] = __float_as_uint(x(i)) >> 16;
    rb[i] = __float_as_uint(r(i)) >> 16;
  }
  return exact_dot_sign_bits(xb, rb, n) > 0;
}

}  // namespace clo
