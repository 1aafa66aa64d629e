/*
 * CPU oracle for the CLO decode step -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the package smoke check and the benchmark's CPU-baseline leg
 * load this library.  It shares no code, header, table or helper with the CUDA
 * library; it is written as plainly as possible from the method's statement:
 * fp64 arithmetic, a scalar bit-counting loop, a full sort for top-k.
 *
 * Sources (page title, section):
 *   [SYN] "CLO (2511.14510) - L3 Per-Paper Synthesis"
 *   [KVO] "KV Cache Offloading 完全拆解" (KV-cache offloading survey blog)
 *   [ABS] CLO abstract (arXiv 2511.14510v1, paper-check page)
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (no FMA contraction:
 * the error-free sum below needs exactly rounded + and -).
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bf16 bit pattern -> exact double. */
double orc_bf16(uint16_t b) {
  uint32_t bits = (uint32_t)b << 16;
  float f;
  memcpy(&f, &bits, 4);
  return (double)f;
}

/*
 * KV bytes per token for a whole stack: 2 (K and V) * n_kv * d_head * bytes * L.
 * [KVO] section "KV Cache 到底有多大" (per-layer formula and its 70B worked value).
 */
int64_t orc_kv_bytes_per_token(int64_t n_kv, int64_t d_head, int64_t elem_bytes, int64_t n_layers) {
  return 2 * n_kv * d_head * elem_bytes * n_layers;
}

/* ---------------------------------------------------------------------------
 * Exact sign of a sum of doubles (Shewchuk, "Adaptive Precision Floating-Point
 * Arithmetic and Fast Robust Geometric Predicates", 1997: TWO-SUM and
 * GROW-EXPANSION).  The running sum is kept as a nonoverlapping expansion whose
 * components are ordered by increasing magnitude; its sign is the sign of the
 * largest nonzero component.
 * ------------------------------------------------------------------------- */
static void two_sum(double a, double b, double* x, double* y) {
  double s = a + b;
  double bv = s - a;
  double av = s - bv;
  double br = b - bv;
  double ar = a - av;
  *x = s;
  *y = ar + br;
}

int orc_exact_sign(const double* p, int n) {
  double e[1100];
  int m = 0;
  if (n > 1000) return 0;
  for (int i = 0; i < n; ++i) {
    double q = p[i];
    int k = 0;
    for (int j = 0; j < m; ++j) {
      double hi, lo;
      two_sum(q, e[j], &hi, &lo);
      q = hi;
      if (lo != 0.0) e[k++] = lo; /* zero elimination */
    }
    if (q != 0.0) e[k++] = q;
    m = k;
  }
  if (m == 0) return 0;
  return e[m - 1] > 0.0 ? 1 : -1;
}

/*
 * Hash code of one vector x (length d, bf16) against the projection R (d x 128,
 * row-major, bf16): bit j is set iff the exact real value of sum_i x_i * R_ij is
 * greater than zero.  Bit j is stored in word j/64 at position j%64.
 * The hash-based top-k scorer CLO integrates is named in [SYN] section 3.2
 * (HATA); the 128-bit sign code is the reading of that scorer used here.
 * The fp64 sum is trusted when its magnitude exceeds the recursive-summation
 * error bound; otherwise the exact sign decides.
 */
static void hash_one(const uint16_t* x, const uint16_t* R, int d, uint64_t* code) {
  double prod[1024];
  code[0] = 0;
  code[1] = 0;
  for (int j = 0; j < 128; ++j) {
    double s = 0.0, a = 0.0;
    for (int i = 0; i < d; ++i) {
      double p = orc_bf16(x[i]) * orc_bf16(R[(int64_t)i * 128 + j]); /* exact in fp64 */
      prod[i] = p;
      s += p;
      a += fabs(p);
    }
    double bound = 2.0 * (double)d * ldexp(1.0, -53) * a;
    int sign;
    if (fabs(s) > bound)
      sign = s > 0.0 ? 1 : -1;
    else
      sign = orc_exact_sign(prod, d);
    if (sign > 0) code[j >> 6] |= (uint64_t)1 << (j & 63);
  }
}

void orc_hash_codes(const uint16_t* X, int64_t n, int d, const uint16_t* R, uint64_t* codes) {
  if (d > 1000) return;
#pragma omp parallel for schedule(dynamic, 64)
  for (int64_t t = 0; t < n; ++t) hash_one(X + t * d, R, d, codes + 2 * t);
}

/*
 * Cosine similarity of two bf16 vectors, fp64; 0 when either vector is zero.
 * The reuse test compares adjacent-step query similarity per head ([SYN] section
 * 2.1 item 2; [ABS] feature (1)).
 */
double orc_cosine(const uint16_t* a, const uint16_t* b, int64_t n) {
  double ab = 0.0, aa = 0.0, bb = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    double x = orc_bf16(a[i]), y = orc_bf16(b[i]);
    ab += x * y;
    aa += x * x;
    bb += y * y;
  }
  if (aa == 0.0 || bb == 0.0) return 0.0;
  return ab / (sqrt(aa) * sqrt(bb));
}

/* Number of set bits, one bit at a time. */
static int count_bits(uint64_t w) {
  int c = 0;
  for (int i = 0; i < 64; ++i) c += (int)((w >> i) & 1u);
  return c;
}

/*
 * Scores of N cached tokens against the G query codes of a GQA group:
 * score[t] = sum_g (128 - hamming(qcode_g, kcode_t)), i.e. matching bits summed
 * over the group's query heads.
 */
void orc_scores(const uint64_t* qcodes, int G, const uint64_t* kcodes, int64_t N, int32_t* scores) {
#pragma omp parallel for schedule(static) if (N >= 8192)
  for (int64_t t = 0; t < N; ++t) {
    int s = 0;
    for (int g = 0; g < G; ++g) {
      int ham = count_bits(qcodes[2 * g] ^ kcodes[2 * t]) + count_bits(qcodes[2 * g + 1] ^ kcodes[2 * t + 1]);
      s += 128 - ham;
    }
    scores[t] = s;
  }
}

typedef struct {
  int32_t score;
  int32_t index;
} orc_pair;

static int by_score_desc_index_asc(const void* pa, const void* pb) {
  const orc_pair* a = (const orc_pair*)pa;
  const orc_pair* b = (const orc_pair*)pb;
  if (a->score != b->score) return a->score > b->score ? -1 : 1;
  return a->index < b->index ? -1 : (a->index > b->index ? 1 : 0);
}

static int by_int_asc(const void* pa, const void* pb) {
  int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
  return a < b ? -1 : (a > b ? 1 : 0);
}

/*
 * Top-k selection: sort all N tokens by (score descending, index ascending),
 * keep the first k, and return them in ascending index order.  k is the top-k
 * budget of the sparse attention (10 % of the context, [SYN] section 2.2).
 */
int orc_topk(const int32_t* scores, int64_t N, int64_t k, int32_t* idx) {
  if (k < 0 || k > N) return -1;
  orc_pair* all = (orc_pair*)malloc(sizeof(orc_pair) * (size_t)(N > 0 ? N : 1));
  if (!all) return -2;
  for (int64_t t = 0; t < N; ++t) {
    all[t].score = scores[t];
    all[t].index = (int32_t)t;
  }
  qsort(all, (size_t)N, sizeof(orc_pair), by_score_desc_index_asc);
  for (int64_t r = 0; r < k; ++r) idx[r] = all[r].index;
  qsort(idx, (size_t)k, sizeof(int32_t), by_int_asc);
  free(all);
  return 0;
}

/*
 * Sparse softmax attention of the G query heads of a group over k selected rows
 * (K, V bf16 [k][d]), fp64: out_g = sum_r softmax_r(q_g . k_r / sqrt(d)) v_r.
 * Top-k sparse attention over the selected rows is CLO's attention ([SYN] section
 * 2.6; [ABS]).  k == 0 gives a zero output.
 */
void orc_attention(const uint16_t* q, int G, int d, const uint16_t* K, const uint16_t* V, int64_t k,
                   double* out) {
  double* s = (double*)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
  double scale = 1.0 / sqrt((double)d);
  for (int g = 0; g < G; ++g) {
    double* o = out + (int64_t)g * d;
    for (int i = 0; i < d; ++i) o[i] = 0.0;
    if (k == 0) continue;
    double m = -INFINITY;
    for (int64_t r = 0; r < k; ++r) {
      double dot = 0.0;
      for (int i = 0; i < d; ++i) dot += orc_bf16(q[(int64_t)g * d + i]) * orc_bf16(K[r * d + i]);
      s[r] = dot * scale;
      if (s[r] > m) m = s[r];
    }
    double z = 0.0;
    for (int64_t r = 0; r < k; ++r) {
      double w = exp(s[r] - m);
      z += w;
      for (int i = 0; i < d; ++i) o[i] += w * orc_bf16(V[r * d + i]);
    }
    for (int i = 0; i < d; ++i) o[i] /= z;
  }
  free(s);
}

/* Number of OpenMP threads the oracle's parallel loops use. */
int orc_num_threads(void) {
  int n = 1;
#pragma omp parallel
  {
#pragma omp single
    n = omp_get_num_threads();
  }
  return n;
}

/* Quantised host KV ([KVO] section on quantised offloading: the offloaded K/V are
 * stored at a few bits per value with an asymmetric scale and offset and
 * dequantised on the GPU after the transfer).  Reading used here, per token and
 * per K or V row, in groups of 64 consecutive channels, every operation in fp32
 * rounded to nearest even:
 *   mn = min of the group (+0 for a zero), mx = max, scale = (mx - mn) / (2^bits - 1),
 *   q_i = 0 if scale == 0, else clamp(rint((x_i - mn) / scale), 0, 2^bits - 1),
 *   value_i = bf16(fma(q_i, scale, mn)).
 * orc_kv_roundtrip maps n_values bf16 values (a whole number of groups) to the
 * values the GPU sees after dequantisation. */
static float bf16_to_float(uint16_t b) {
  uint32_t bits = (uint32_t)b << 16;
  float f;
  memcpy(&f, &bits, 4);
  return f;
}

static uint16_t float_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u); /* NaN stays NaN */
  const uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

void orc_kv_roundtrip(const uint16_t* x, int64_t n_values, int bits, uint16_t* y) {
  const float levels = (float)((1 << bits) - 1);
  for (int64_t g0 = 0; g0 < n_values; g0 += 64) {
    float mn = bf16_to_float(x[g0]), mx = mn;
    for (int i = 1; i < 64; ++i) {
      const float v = bf16_to_float(x[g0 + i]);
      if (v < mn) mn = v;
      if (v > mx) mx = v;
    }
    mn = mn + 0.0f; /* a zero minimum is +0 whichever zero the comparison kept */
    const float scale = (mx - mn) / levels;
    for (int i = 0; i < 64; ++i) {
      float q = 0.0f;
      if (scale > 0.0f) {
        q = rintf((bf16_to_float(x[g0 + i]) - mn) / scale);
        if (q < 0.0f) q = 0.0f;
        if (q > levels) q = levels;
      }
      y[g0 + i] = float_to_bf16_rne(fmaf(q, scale, mn));
    }
  }
}

/* Host-pool bytes of one token's K|V record of one kv head, the bytes a fetch moves
 * over the host link: 4 d (bf16), or the codes of both rows for bits < 16 (the
 * groups' fp32 scale and min stay in GPU memory). */
int64_t orc_kv_record_bytes(int64_t d, int bits) {
  if (bits >= 16) return 4 * d;
  return 2 * d * bits / 8;
}
