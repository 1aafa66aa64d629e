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
//   2. compensated fp32 sum of the products: a TwoSum chain whose rounding errors
//      are summed separately (the "Sum2" scheme of Ogita, Rump and Oishi, "Accurate
//      sum and dot product", 2005).  Its result r is within eps |s| + g^2 a of the
//      exact sum (eps = 2^-24, g = (n-1) eps / (1 - (n-1) eps)), plus n * 2^-150
//      for products that fall below the fp32 normal range, so |r| > 2 g^2 a +
//      n * 2^-148 fixes the sign.  No fp64: its rate on this GPU is so low that one
//      fp64 fallback held a whole CTA for ~20 us.
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
  float sh = 0.f, sl = 0.f, a = 0.f;
  for (int i = 0; i < n; ++i) {
    const float p = __fmul_rn(x(i), r(i));  // exact unless below the normal range
    const float t = __fadd_rn(sh, p);       // TwoSum(sh, p) = (t, e), t + e = sh + p exactly
    const float bp = __fsub_rn(t, sh);
    const float e = __fadd_rn(__fsub_rn(sh, __fsub_rn(t, bp)), __fsub_rn(p, bp));
    sh = t;
    sl = __fadd_rn(sl, e);
    a = __fadd_rn(a, fabsf(p));
  }
  const float res = __fadd_rn(sh, sl);
  const float nm1 = (float)(n - 1) * 5.9604644775390625e-8f;  // (n - 1) 2^-24
  const float g = nm1 / (1.f - nm1);
  // a carries its own rounding (relative error below g): scaled up by 1 + 2g
  const float bound = 2.f * g * g * (a * (1.f + 2.f * g)) + (float)n * 2.802596928649634e-45f;
  if (fabsf(res) > bound) return res > 0.f;
  uint32_t xb[256], rb[256];
  for (int i = 0; i < n; ++i) {
    xb[i] = __float_as_uint(x(i)) >> 16;
    rb[i] = __float_as_uint(r(i)) >> 16;
  }
  return exact_dot_sign_bits(xb, rb, n) > 0;
}

}  // namespace clo
