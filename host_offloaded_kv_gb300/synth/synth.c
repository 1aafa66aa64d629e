/*
 * Seeded synthetic workload generator for the CLO decode-step workloads.
 *
 * This module holds no arithmetic of the method itself: it only produces the
 * inputs (keys, values, queries, hash projection) that both the CUDA library
 * and the CPU oracle consume.  Every value is a pure function of
 * (seed, stream, counter), so any unit of a workload can be regenerated on its
 * own without generating the rest.
 *
 * Distributions (from the workload statements of the CLO decode workloads):
 *   - keys and values ~ N(0,1), rounded once to bf16 (round to nearest even);
 *   - heavy-hitter keys: k = 4*u_{l,h} + N(0,I), u_{l,h} a seeded unit vector per
 *     (layer, kv head); a token is a heavy hitter with probability hh_ratio,
 *     drawn independently per token from its own counter;
 *   - hash projection R_{l,h} in R^{d x 128}, entries N(0,1), stored bf16;
 *   - queries AR(1): q_0 ~ N(0,I), q_t = rho q_{t-1} + sqrt(1-rho^2) eps_t, with
 *     rho ~ U[rho_lo, rho_hi] per (layer, seq, query head); the recursion state
 *     is kept in double and rounded to bf16 on output.
 *
 * Normals come from Box-Muller on two 32-bit uniforms of one splitmix64 draw.
 * Build with -ffp-contract=off so results do not depend on FMA contraction.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define SYN_KIND_K 1u
#define SYN_KIND_V 2u
#define SYN_KIND_HH 3u
#define SYN_KIND_DIR 4u
#define SYN_KIND_R 5u
#define SYN_KIND_Q0 6u
#define SYN_KIND_QEPS 7u
#define SYN_KIND_RHO 8u

static inline uint64_t syn_mix(uint64_t z) {
  /* splitmix64 finaliser (Steele, Lea, Flood 2014). */
  z += 0x9e3779b97f4a7c15ull;
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

/* One 64-bit draw for (seed, stream, counter). */
uint64_t synth_u64(uint64_t seed, uint64_t stream, uint64_t counter) {
  uint64_t s = syn_mix(seed ^ 0x6a09e667f3bcc909ull);
  s = syn_mix(s ^ stream);
  return syn_mix(s ^ (counter * 0xd1b54a32d192ed03ull));
}

static inline uint64_t syn_stream(uint32_t kind, uint64_t a, uint64_t b, uint64_t c, uint64_t e) {
  uint64_t s = syn_mix(((uint64_t)kind << 56) ^ 0x243f6a8885a308d3ull);
  s = syn_mix(s ^ a);
  s = syn_mix(s ^ (b + 0x13198a2e03707344ull));
  s = syn_mix(s ^ (c + 0xa4093822299f31d0ull));
  return syn_mix(s ^ (e + 0x082efa98ec4e6c89ull));
}

/* Standard normal number i of a stream (Box-Muller, pairs share one draw). */
double synth_normal(uint64_t seed, uint64_t stream, uint64_t i) {
  uint64_t h = synth_u64(seed, stream, i >> 1);
  double u1 = ((double)(h >> 32) + 0.5) * (1.0 / 4294967296.0); /* (0,1) */
  double u2 = (double)(h & 0xffffffffull) * (1.0 / 4294967296.0);
  double r = sqrt(-2.0 * log(u1));
  double th = 6.283185307179586476925286766559 * u2;
  return (i & 1) ? r * sin(th) : r * cos(th);
}

/* Uniform in [0,1) with 53 bits. */
static inline double syn_uniform(uint64_t seed, uint64_t stream, uint64_t i) {
  return (double)(synth_u64(seed, stream, i) >> 11) * (1.0 / 9007199254740992.0);
}

/* double -> bf16, round to nearest even, with a single rounding.
 * Goes through float with round-to-odd so the second rounding is exact. */
uint16_t synth_bf16_from_double(double x) {
  if (x != x) return 0x7fc0;
  float f = (float)x;
  if (isinf(f)) {
    uint32_t b;
    memcpy(&b, &f, 4);
    return (uint16_t)(b >> 16);
  }
  if (fabs((double)f) > fabs(x)) f = nextafterf(f, 0.0f);
  uint32_t bits;
  memcpy(&bits, &f, 4);
  if ((double)f != x) bits |= 1u; /* sticky: round to odd */
  uint32_t lsb = (bits >> 16) & 1u;
  bits += 0x7fffu + lsb;
  return (uint16_t)(bits >> 16);
}

double synth_bf16_to_double(uint16_t b) {
  uint32_t bits = (uint32_t)b << 16;
  float f;
  memcpy(&f, &bits, 4);
  return (double)f;
}

/* Unit direction u_{l,h} (length d, double) used by heavy-hitter keys. */
void synth_head_direction(uint64_t seed, int l, int h, int d, double* u) {
  uint64_t st = syn_stream(SYN_KIND_DIR, (uint64_t)l, (uint64_t)h, 0, 0);
  double n2 = 0.0;
  for (int i = 0; i < d; ++i) {
    u[i] = synth_normal(seed, st, (uint64_t)i);
    n2 += u[i] * u[i];
  }
  double inv = 1.0 / sqrt(n2);
  for (int i = 0; i < d; ++i) u[i] *= inv;
}

int synth_is_heavy(uint64_t seed, int l, int b, int h, int64_t t, double hh_ratio) {
  uint64_t st = syn_stream(SYN_KIND_HH, (uint64_t)l, (uint64_t)b, (uint64_t)h, 0);
  return syn_uniform(seed, st, (uint64_t)t) < hh_ratio;
}

/*
 * Keys and values of tokens [t0, t0+n) of one unit (layer l, seq b, kv head h),
 * written as bf16 rows K[n][d], V[n][d] (row stride ld elements, so callers can
 * write straight into a [n][Hkv][d] buffer with ld = Hkv*d).
 */
void synth_unit_kv(uint64_t seed, int l, int b, int h, int64_t t0, int64_t n, int d,
                   double hh_ratio, uint16_t* K, uint16_t* V, int64_t ld) {
  double u[1024];
  if (d > 1024) return;
  synth_head_direction(seed, l, h, d, u);
  uint64_t sk = syn_stream(SYN_KIND_K, (uint64_t)l, (uint64_t)b, (uint64_t)h, 0);
  uint64_t sv = syn_stream(SYN_KIND_V, (uint64_t)l, (uint64_t)b, (uint64_t)h, 0);
#pragma omp parallel for schedule(static) if (n >= 256)
  for (int64_t r = 0; r < n; ++r) {
    int64_t t = t0 + r;
    int heavy = synth_is_heavy(seed, l, b, h, t, hh_ratio);
    uint16_t* kr = K + r * ld;
    uint16_t* vr = V + r * ld;
    for (int i = 0; i < d; ++i) {
      uint64_t c = (uint64_t)t * (uint64_t)d + (uint64_t)i;
      double z = synth_normal(seed, sk, c);
      if (heavy) z += 4.0 * u[i];
      kr[i] = synth_bf16_from_double(z);
      vr[i] = synth_bf16_from_double(synth_normal(seed, sv, c));
    }
  }
}

/* Keys and values of tokens [t0, t0+n) of all kv heads of (layer l, seq b),
 * layout [n][Hkv][d] bf16 (the layout the library's append call takes). */
void synth_layer_seq_kv(uint64_t seed, int l, int b, int Hkv, int64_t t0, int64_t n, int d,
                        double hh_ratio, uint16_t* K, uint16_t* V) {
  for (int h = 0; h < Hkv; ++h)
    synth_unit_kv(seed, l, b, h, t0, n, d, hh_ratio, K + (int64_t)h * d, V + (int64_t)h * d,
                  (int64_t)Hkv * d);
}

/* Hash projection R_{l,h}: d x 128, row-major (R[i*128 + j]), bf16. */
void synth_hash_matrix(uint64_t seed, int l, int h, int d, uint16_t* R) {
  uint64_t st = syn_stream(SYN_KIND_R, (uint64_t)l, (uint64_t)h, 0, 0);
  for (int64_t c = 0; c < (int64_t)d * 128; ++c)
    R[c] = synth_bf16_from_double(synth_normal(seed, st, (uint64_t)c));
}

/* AR(1) coefficients rho ~ U[lo, hi] per (layer, seq, query head), flat [L*B*Hq]. */
void synth_query_rho(uint64_t seed, int L, int B, int Hq, double lo, double hi, double* rho) {
  for (int l = 0; l < L; ++l)
    for (int b = 0; b < B; ++b)
      for (int q = 0; q < Hq; ++q) {
        uint64_t st = syn_stream(SYN_KIND_RHO, (uint64_t)l, (uint64_t)b, (uint64_t)q, 0);
        rho[((int64_t)l * B + b) * Hq + q] = lo + (hi - lo) * syn_uniform(seed, st, 0);
      }
}

/*
 * Advance the AR(1) query state to decode step t and emit bf16 queries.
 * state: double [L*B*Hq*d]; step 0 initialises it with N(0,I).
 * q_out: bf16 [L][B][Hq][d].
 */
void synth_query_step(uint64_t seed, int L, int B, int Hq, int d, int64_t t, const double* rho,
                      double* state, uint16_t* q_out) {
  int64_t nvec = (int64_t)L * B * Hq;
#pragma omp parallel for schedule(static) if (nvec >= 64)
  for (int64_t v = 0; v < nvec; ++v) {
    int q = (int)(v % Hq);
    int b = (int)((v / Hq) % B);
    int l = (int)(v / ((int64_t)Hq * B));
    double* s = state + v * d;
    uint16_t* o = q_out + v * d;
    if (t == 0) {
      uint64_t st = syn_stream(SYN_KIND_Q0, (uint64_t)l, (uint64_t)b, (uint64_t)q, 0);
      for (int i = 0; i < d; ++i) s[i] = synth_normal(seed, st, (uint64_t)i);
    } else {
      uint64_t st = syn_stream(SYN_KIND_QEPS, (uint64_t)l, (uint64_t)b, (uint64_t)q, (uint64_t)t);
      double r = rho[v];
      double c = sqrt(1.0 - r * r);
      for (int i = 0; i < d; ++i) s[i] = r * s[i] + c * synth_normal(seed, st, (uint64_t)i);
    }
    for (int i = 0; i < d; ++i) o[i] = synth_bf16_from_double(s[i]);
  }
}

/* Plain N(0,1) bf16 fill of an arbitrary stream (for test fixtures). */
void synth_normal_bf16(uint64_t seed, uint64_t stream, int64_t n, uint16_t* out) {
#pragma omp parallel for schedule(static) if (n >= 4096)
  for (int64_t i = 0; i < n; ++i) out[i] = synth_bf16_from_double(synth_normal(seed, stream, (uint64_t)i));
}
