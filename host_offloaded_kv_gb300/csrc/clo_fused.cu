// One persistent, warp-specialised kernel per decode step (or per layer): top-k
// selection of the missed and persistent units, zero-copy fetch of the missed units'
// rows from pinned host memory, and split-K sparse attention, ordered by device-side
// flags only.  The reuse decisions, query codes and per-layer work lists come from the
// decide kernel launched just before.
//
// Each CTA holds one fetch warp and one 4-warp compute group (3 CTAs per SM).
//   * The compute group takes items from one queue, in this order (each list in layer
//     order, the chunks of a unit next to each other):
//       1. selection chunks of the missed units (their fetch waits for them);
//       2. selection of the persistent units (whole units of up to 32K tokens in a large
//          launch, else chunks);
//       3. attention splits of the reused units, then of the persistent units, then of
//          the missed units.
//     A selection scores every cached token, score[t] = sum_g (128 - popc(qcode_g ^
//     kcode_t)) (HATA hash scorer, "CLO (2511.14510) - L3 Per-Paper Synthesis", section
//     3.2), and keeps the k = 10 % best (section 2.2), ties to the lowest index, in
//     ascending order: a one-digit radix select over the <= 128 G + 1 score values.
//     An attention split feeds 16-row chunks of K|V rows to each warp through a
//     shared-memory ring filled by bulk copies on the TMA engine (one 4 d-byte row per
//     copy, from the unit's cache slot or, for persistent units, gathered from its
//     resident copy), computes out_g = sum_r softmax_r(q_g . k_r / sqrt(d)) v_r with
//     tensor-core tiles, and merges partials by log-sum-exp.
//   * Fetch warps copy the selected K|V rows of missed units from pinned host memory
//     into the units' on-GPU cache slots with 16-byte loads, 256-row chunk by chunk in
//     layer order, and release one ready flag per chunk (CLO abstract, feature (3):
//     zero-copy transfer engine and GPU-centric synchronisation; the fetch runs ahead of
//     the attention that consumes it, as CLO prefetches a layer ahead, section 5.6).
// Every wait targets work that sits earlier in the compute queue (or a fetch, which
// itself waits only on earlier compute items), so the waits form no cycle; each wait is
// bounded by the context's timeout and reports CLO_ERR_TIMEOUT.
#include <cuda_bf16.h>
#include <stdlib.h>

#include "clo_internal.cuh"

namespace clo {

namespace {

constexpr int kCompWarps = 4;
constexpr int kCompThreads = 32 * kCompWarps;
constexpr int kFetchUnroll = 4;
constexpr int kAttStages = 2;  // ring stages of 16 rows per compute warp

__device__ __forceinline__ void comp_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kCompThreads) : "memory"); }

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

// Bounded wait until *flag >= target (acquire); on timeout: error word + counter.  The
// poll interval doubles from 32 ns up to max_sleep_ns.
__device__ void wait_flag(const uint32_t* flag, uint32_t target, const DevState& s, unsigned max_sleep_ns = 2048) {
  if (ld_acquire_u32(flag) >= target) return;
  const uint64_t t0 = global_timer_ns();
  unsigned ns = 32;
  while (ld_acquire_u32(flag) < target) {
    if (global_timer_ns() - t0 > (uint64_t)s.wait_timeout_ns) {
      atomicOr(s.err, kErrFlagTimeout);
      atomicAdd(&s.step_ctr[ctr_at(C_TIMEOUTS, 0)], 1ull);
      atomicAdd(&s.total_ctr[ctr_at(C_TIMEOUTS, 0)], 1ull);
      return;
    }
    __nanosleep(ns);
    if (ns < max_sleep_ns) ns <<= 1;
  }
}

template <int D>
struct AttSmem {
  static constexpr int ROWW = 2 * D + 8;             // bf16 per smem row (K | V), padded by 16 bytes
  uint16_t rows[kCompWarps][kAttStages][16][ROWW];   // each warp's ring of 16-row stages
  float red[kCompWarps];
  int last;
};

struct SelSmem {
  uint16_t scores[kSelChunkMax];     // scores of the chunk's tokens
  uint32_t hist[kCompWarps][kNBPad]; // each warp's histogram of its segment
  uint32_t tot[kNBPad];              // the unit's histogram
  int wc[kCompWarps][2];             // {above T, at T} of each warp's segment
  int2 thr;                          // {T, count above T}
  int misc[8];
};

// A whole unit of up to 32K tokens selected by one compute group.
struct SelUnitSmem {
  uint16_t scores[32768];
  uint32_t hist[kNBPad];
  int wc[kCompWarps][2];  // {above T, at T} of each warp's segment
  int2 thr;               // {T, count above T}
  int misc[8];
};

template <int D>
union CompSmem {
  AttSmem<D> att;
  SelSmem sel;
  SelUnitSmem unit;
};

// ---- hash-code scores -------------------------------------------------------------------
// score(k) = sum_g (128 - popc(k ^ q_g)) over the G query codes of the group.  Per bit j let
// c_j = number of query codes with bit j set; then the summed Hamming distance is
//   X(k) = sum_j (k_j ? G - c_j : c_j),
// a sum of small numbers v_j.  With the binary digits of c_j and of G - c_j held as bit
// planes A_p and B_p (p < NP), digit p of v_j is one bit-select, (k & B_p) | (~k & A_p),
// and X = sum_p 2^p popc(V_p).  A carry-save adder tree folds the NP x 4 plane words into
// one word per weight, so a token costs 5 or 6 popcounts instead of 4 G.
template <int G>
struct QPlanes {
  static constexpr int NP = G < 2 ? 1 : (G < 4 ? 2 : (G < 8 ? 3 : 4));  // digits of 0..G
  uint32_t A[NP][4], B[NP][4];
};

template <int G>
__device__ __forceinline__ void load_qplanes(const DevState& s, int64_t u, QPlanes<G>& qp) {
  constexpr int NP = QPlanes<G>::NP;
  const int h = (int)(u % s.Hkv);
  const int b = (int)((u / s.Hkv) % s.B);
  const int l = (int)(u / ((int64_t)s.Hkv * s.B));
  const uint4* qc = s.qcodes + ((int64_t)l * s.B + b) * s.Hq + (int64_t)h * G;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t cnt[NP];
#pragma unroll
    for (int p = 0; p < NP; ++p) cnt[p] = 0u;
#pragma unroll
    for (int g = 0; g < G; ++g) {  // bit-sliced counter += query word
      const uint4 v = qc[g];
      uint32_t carry = w == 0 ? v.x : (w == 1 ? v.y : (w == 2 ? v.z : v.w));
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        const uint32_t t = cnt[p] & carry;
        cnt[p] ^= carry;
        carry = t;
      }
    }
    // G - c = (~c) + (G + 1) mod 2^NP, bit-sliced with the constant's digits
    uint32_t carry = 0u;
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      const uint32_t x = ~cnt[p];
      const uint32_t gb = ((G + 1) >> p) & 1 ? 0xffffffffu : 0u;
      qp.A[p][w] = cnt[p];
      qp.B[p][w] = x ^ gb ^ carry;
      carry = (x & gb) | (x & carry) | (gb & carry);
    }
  }
}

__device__ __forceinline__ void csa(uint32_t& sum, uint32_t& carry, uint32_t a, uint32_t b, uint32_t c) {
  sum = a ^ b ^ c;
  carry = (a & b) | (a & c) | (b & c);
}

template <int G>
__device__ __forceinline__ int score_of(const uint4 c, const QPlanes<G>& qp) {
  constexpr int NP = QPlanes<G>::NP;
  const uint32_t k[4] = {c.x, c.y, c.z, c.w};
  uint32_t v[4][4];  // digit planes of v_j (absent planes are zero and fold away)
#pragma unroll
  for (int p = 0; p < 4; ++p)
#pragma unroll
    for (int w = 0; w < 4; ++w) v[p][w] = p < NP ? ((k[w] & qp.B[p < NP ? p : 0][w]) | (~k[w] & qp.A[p < NP ? p : 0][w])) : 0u;
  // weight 1: 4 words -> o1 + 2 carries of weight 2
  uint32_t s, o1, k1, k2;
  csa(s, k1, v[0][0], v[0][1], v[0][2]);
  o1 = s ^ v[0][3];
  k2 = s & v[0][3];
  // weight 2: 4 words + 2 carries -> o2 + 3 carries of weight 4
  uint32_t s1, s2, o2, m1, m2, m3;
  csa(s1, m1, v[1][0], v[1][1], v[1][2]);
  csa(s2, m2, v[1][3], k1, k2);
  o2 = s1 ^ s2;
  m3 = s1 & s2;
  // weight 4: 4 words + 3 carries -> o4 + 3 carries of weight 8
  uint32_t t1, t2, o4, n1, n2, n3;
  csa(t1, n1, v[2][0], v[2][1], v[2][2]);
  csa(t2, n2, v[2][3], m1, m2);
  csa(o4, n3, t1, t2, m3);
  // weight 8: 4 words + 3 carries -> o8 + 3 carries of weight 16
  uint32_t r1, r2, o8, p1, p2, p3;
  csa(r1, p1, v[3][0], v[3][1], v[3][2]);
  csa(r2, p2, v[3][3], n1, n2);
  csa(o8, p3, r1, r2, n3);
  // weight 16: 3 words -> o16 + a carry of weight 32
  uint32_t o16, o32;
  csa(o16, o32, p1, p2, p3);
  const int X = __popc(o1) + 2 * __popc(o2) + 4 * __popc(o4) + 8 * __popc(o8) + 16 * __popc(o16) + 32 * __popc(o32);
  return 128 * G - X;
}

__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// ---- selection item: one chunk of sel_chunk tokens of one unit -------------------------
// Scores are small integers (0 .. 128 G), so the top-k is one histogram digit:
//   1. each warp scores its contiguous quarter of the chunk (16-byte codes read once,
//      coalesced), keeps the scores in shared memory and counts them in its own histogram,
//      the two halves of its quarter in the low and high 16 bits of each bin; the chunk's
//      histogram is added into the unit's histogram in global memory;
//   2. once every chunk's histogram is merged, each chunk finds the unit's threshold T,
//      the largest score with count(score >= T) >= k, and n_gt = count(score > T);
//   3. each lane counts the scores above and at T in its own contiguous span of the
//      warp's segment; a warp scan gives each lane the counts before its span and the
//      chunk publishes its totals; from the totals of the chunks before it, a chunk knows
//      where its indices go and how many of its ties it takes (ties go to the lowest token
//      index: the quota k - n_gt is filled in chunk order);
//   4. ordered compaction: each lane walks its span 8 tokens at a time and writes the
//      indices of the selected ones from its own output position, with no exchange
//      between lanes.
// The chunks of a unit sit next to each other in the work queue and every group runs its
// item to the end, so the waits of steps 2 and 3 only target items already running
// (provided at least nch groups run; the host checks this).

// Largest score T with count(score >= T) >= k from a histogram tot[0..NB) in shared
// memory, by all 128 threads of the group; writes {T, count(score > T)} to *res (only
// the thread whose bins hold the crossing writes).
template <int NB>
__device__ __forceinline__ void find_threshold(const uint32_t* tot, int k, int2* res, int* red, int gtid) {
  constexpr int SEG = (NB + kCompThreads - 1) / kCompThreads;  // bins per thread, from the top
  const int warp = gtid >> 5, lane = gtid & 31;
  const int hi = NB - gtid * SEG;
  const int lo = hi - SEG > 0 ? hi - SEG : 0;
  int segsum = 0;
#pragma unroll
  for (int i = 0; i < SEG; ++i)
    if (hi - 1 - i >= lo) segsum += (int)tot[hi - 1 - i];
  int incl = segsum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) red[warp] = incl;
  comp_bar();
  int before = 0;
#pragma unroll
  for (int w = 0; w < kCompWarps; ++w) before += w < warp ? red[w] : 0;
  incl += before;
  const int excl = incl - segsum;  // count of scores above this thread's bins
  if (excl < k && incl >= k) {
    int run = excl;
    for (int bin = hi - 1; bin >= lo; --bin) {
      if (run + (int)tot[bin] >= k) {
        *res = make_int2(bin, run);
        break;
      }
      run += (int)tot[bin];
    }
  }
}

// ---- lane spans ------------------------------------------------------------------------
// For counting and compaction each lane owns a contiguous span of a warp's segment: 8
// tokens times an odd number of 16-byte chunks, so that the 32 lanes' 16-byte loads fall
// into distinct bank groups of shared memory.  Scores are compared two per 32-bit word:
// for a word holding scores lo | hi << 16 (both <= 1024), (w + c * 0x10001) has bit 15
// (31) set iff lo (hi) >= 0x8000 - c, with no carry between the halves.
__device__ __forceinline__ int span_tokens(int seg) {
  const int ch = (seg + 255) / 256;  // 16-byte chunks per lane, made odd
  return 8 * (ch | 1);
}

// bit 15 - i (31 - i) of the result: token 2 i (2 i + 1) of the chunk has score >= 0x8000 - c
__device__ __forceinline__ uint32_t ge_bits(const uint4 v, uint32_t c2) {
  const uint32_t m = 0x80008000u;
  return ((v.x + c2) & m) | (((v.y + c2) & m) >> 1) | (((v.z + c2) & m) >> 2) | (((v.w + c2) & m) >> 3);
}

// token-order 8-bit mask (bit j = token j) from ge_bits' layout
__device__ __forceinline__ uint32_t token_mask(uint32_t x) {
  uint32_t lo = __brev(x << 16) & 0xfu;  // bit i = token 2 i
  uint32_t hi = __brev(x) & 0xfu;        // bit i = token 2 i + 1
  lo = (lo | (lo << 2)) & 0x33u;
  lo = (lo | (lo << 1)) & 0x55u;
  hi = (hi | (hi << 2)) & 0x33u;
  hi = (hi | (hi << 1)) & 0x55u;
  return lo | (hi << 1);
}

// the 8 scores of tokens [t, t + 8) as 4 words (tokens at or past b read as 0)
__device__ __forceinline__ uint4 load_chunk(const uint16_t* scores, int t, int b) {
  if (t + 8 <= b) return *reinterpret_cast<const uint4*>(&scores[t]);
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t l = t + 2 * j < b ? scores[t + 2 * j] : 0u;
    const uint32_t h = t + 2 * j + 1 < b ? scores[t + 2 * j + 1] : 0u;
    w[j] = l | (h << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// tokens of [t, t + 8) below b, in ge_bits' layout
__device__ __forceinline__ uint32_t valid_bits(int t, int b) {
  const int n = b - t;
  if (n >= 8) return 0xffffffffu;
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (j < n) m |= (j & 1) ? (1u << (31 - j / 2)) : (1u << (15 - j / 2));
  return m;
}

// {count above T, count at T} of tokens [lo, hi) (lo a multiple of 8)
__device__ __forceinline__ int2 count_span(const uint16_t* scores, int lo, int hi, int T) {
  const uint32_t cg = (uint32_t)(0x8000 - T - 1) * 0x10001u, ce = (uint32_t)(0x8000 - T) * 0x10001u;
  int g = 0, ge = 0;
#pragma unroll 4
  for (int t = lo; t < hi; t += 8) {
    const uint4 v = load_chunk(scores, t, hi);
    const uint32_t val = valid_bits(t, hi);
    g += __popc(ge_bits(v, cg) & val);
    ge += __popc(ge_bits(v, ce) & val);
  }
  return make_int2(g, ge - g);
}

// Ordered compaction of tokens [lo, hi): tokens above T, and ties while fewer than q ties
// precede them (er = ties before lo, counted like q), go to out[pos], out[pos + 1], ...
// as t0 + token.
__device__ __forceinline__ void compact_span(const uint16_t* scores, int lo, int hi, int pos, int er, int q, int T,
                                             int64_t t0, int32_t* out, int k, uint32_t* err) {
  const uint32_t cg = (uint32_t)(0x8000 - T - 1) * 0x10001u, ce = (uint32_t)(0x8000 - T) * 0x10001u;
  for (int t = lo; t < hi; t += 8) {
    const uint4 v = load_chunk(scores, t, hi);
    const uint32_t val = valid_bits(t, hi);
    const uint32_t gb = ge_bits(v, cg) & val, eb = ge_bits(v, ce) & val & ~gb;
    uint32_t sel = token_mask(gb);
    if (eb) {
      uint32_t em = token_mask(eb);
      const int ne = __popc(em);
      const int room = q - er;  // ties this chunk may still take, lowest index first
      if (room <= 0)
        em = 0;
      else
        for (int drop = ne - room; drop > 0; --drop) em &= ~(0x80000000u >> __clz(em));  // drop the highest
      sel |= em;
      er += ne;
    }
    while (sel) {
      const int j = __ffs(sel) - 1;
      if (pos < k)
        out[pos] = (int32_t)(t0 + t + j);
      else
        atomicOr(err, kErrBounds);
      ++pos;
      sel &= sel - 1;
    }
  }
}

// Counts of each lane's span of the warp's segment [w0, w1) and the warp scan over them:
// returns the lane's span and {above, at} before it; lane 31 stores the warp's totals.
struct LaneSpan {
  int lo, hi, gx, ex;
};

__device__ __forceinline__ LaneSpan span_counts(const uint16_t* scores, int w0, int w1, int T, int* wc, int lane) {
  const int e = w1 > w0 ? w1 : w0;
  const int S = span_tokens(e - w0);
  LaneSpan sp;
  sp.lo = min(w0 + lane * S, e);
  sp.hi = min(sp.lo + S, e);
  const int2 c = count_span(scores, sp.lo, sp.hi, T);
  const int v = c.x | (c.y << 16);  // a warp's segment holds <= 8192 tokens: 16-bit halves
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  const int excl = incl - v;
  sp.gx = excl & 0xffff;
  sp.ex = excl >> 16;
  if (lane == 31) {
    wc[0] = incl & 0xffff;
    wc[1] = incl >> 16;
  }
  return sp;
}

template <int G>
__device__ void sel_chunk(const DevState& s, SelSmem& sm, int64_t u, int c, int CH, int NC, int gtid) {
  constexpr int NB = 128 * G + 1;
  constexpr int kU = 8;                          // code loads in flight per lane
  const int WSEG = CH / kCompWarps;              // tokens per warp (CH: 1024 .. 16384), a multiple of 32 * kU
  const int b = (int)((u / s.Hkv) % s.B);
  const int64_t N = s.ntok[b];
  const int k = s.kcount[b];
  const int64_t t0 = (int64_t)c * CH;
  const int len = (int)(N - t0 <= 0 ? 0 : (N - t0 < CH ? N - t0 : CH));
  const int warp = gtid >> 5, lane = gtid & 31;
  uint32_t* wh = sm.hist[warp];
  for (int i = lane; i < NB; i += 32) wh[i] = 0;
  QPlanes<G> qp;
  load_qplanes<G>(s, u, qp);
  __syncwarp();

  // 1. scores and histograms of this warp's segment [w0, w1)
  const int w0 = warp * WSEG;
  const int w1 = (w0 + WSEG < len) ? w0 + WSEG : len;
  const uint4* src = s.codes + u * s.Nmax + t0;
  constexpr int kPfRounds = 4;  // L2 prefetch of the codes this many rounds ahead
  if (lane == 0)
    for (int r = 1; r < kPfRounds; ++r) {
      const int pb = w0 + r * 32 * kU;
      if (pb < w1) prefetch_l2(src + pb, 16u * (uint32_t)((w1 - pb) < 32 * kU ? (w1 - pb) : 32 * kU));
    }
  for (int base = w0; base < w1; base += 32 * kU) {
    if (lane == 0) {
      const int pb = base + kPfRounds * 32 * kU;
      if (pb < w1) prefetch_l2(src + pb, 16u * (uint32_t)((w1 - pb) < 32 * kU ? (w1 - pb) : 32 * kU));
    }
    uint4 cv[kU];
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      const int t = base + 32 * j + lane;
      if (t < w1) cv[j] = ld_nc_v4(src + t);
    }
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      const int t = base + 32 * j + lane;
      if (t < w1) {
        const int sc = score_of<G>(cv[j], qp);
        sm.scores[t] = (uint16_t)sc;
        atomicAdd(&wh[sc], 1u);
      }
    }
  }
  comp_bar();
  uint32_t* UH = s.unit_hist + u * s.nbp;
  for (int i = gtid; i < NB; i += kCompThreads) {
    uint32_t v = 0;
#pragma unroll
    for (int w = 0; w < kCompWarps; ++w) v += sm.hist[w][i];
    if (v) atomicAdd(UH + i, v);
  }
  comp_bar();  // the group's additions happen before gtid 0's release below
  if (gtid == 0) {
    red_release_add_u32(&s.score_done[u], 1u);
    wait_flag(&s.score_done[u], (uint32_t)NC, s, 256);  // every chunk's histogram is merged
  }
  comp_bar();

  // 2. threshold: every chunk reads the unit's histogram and finds T itself (the chunk
  //    that finishes its compaction last zeroes the histogram for the next step)
  {
    constexpr int PER = (NB + kCompThreads - 1) / kCompThreads;
    uint32_t v[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int bin = gtid + i * kCompThreads;
      v[i] = bin < NB ? __ldcg(UH + bin) : 0u;
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int bin = gtid + i * kCompThreads;
      if (bin < NB) sm.tot[bin] = v[i];
    }
    if (gtid == 0) sm.thr = make_int2(-1, 0);
    comp_bar();
    find_threshold<NB>(sm.tot, k, &sm.thr, &sm.misc[4], gtid);
    comp_bar();
    if (gtid == 0) {
      const int2 th = sm.thr;
      sm.misc[1] = th.x < 0 ? 0 : (th.x >= NB ? NB - 1 : th.x);  // clamped: garbage only after a timeout
      sm.misc[2] = th.y;
    }
  }
  comp_bar();
  const int T = sm.misc[1], n_gt = sm.misc[2];
  const int quota = k - n_gt;  // ties to take, unit-wide, lowest index first

  // 3. each lane's counts above and at T, the warp's totals, then the chunk's
  const LaneSpan sp = span_counts(sm.scores, w0, w1, T, sm.wc[warp], lane);
  comp_bar();
  int eq_c = 0;
#pragma unroll
  for (int w = 0; w < kCompWarps; ++w) eq_c += sm.wc[w][1];
  if (warp == 0) {
    if (lane == 0) {
      int gt_c = 0;
#pragma unroll
      for (int w = 0; w < kCompWarps; ++w) gt_c += sm.wc[w][0];
      s.sel_meta[u * NC + c] = make_int2(gt_c, eq_c);
      __threadfence();
      red_release_add_u32(&s.cnt_done[u], 1u);
      wait_flag(&s.cnt_done[u], (uint32_t)NC, s, 256);
    }
    __syncwarp();
    int base_sel = 0, eq_before = 0;
    for (int c0 = 0; c0 < c; c0 += 32) {
      const int2 m = (c0 + lane < c) ? __ldcg(&s.sel_meta[u * NC + c0 + lane]) : make_int2(0, 0);
      int ie = m.y;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, ie, o);
        if (lane >= o) ie += v;
      }
      int take = quota - (eq_before + ie - m.y);
      take = take < 0 ? 0 : (take > m.y ? m.y : take);
      int sel = m.x + take;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sel += __shfl_xor_sync(0xffffffffu, sel, o);
      base_sel += sel;
      eq_before += __shfl_sync(0xffffffffu, ie, 31);
    }
    if (lane == 0) {
      sm.misc[3] = base_sel;
      sm.misc[4] = eq_before;
    }
  }
  comp_bar();
  int take_eq = quota - sm.misc[4];  // ties this chunk takes
  take_eq = take_eq < 0 ? 0 : (take_eq > eq_c ? eq_c : take_eq);

  // 4. ordered compaction of each lane's span
  int off = sm.misc[3], eqb = 0;
  for (int w = 0; w < warp; ++w) {
    off += sm.wc[w][0] + min(max(take_eq - eqb, 0), sm.wc[w][1]);
    eqb += sm.wc[w][1];
  }
  const int q = max(take_eq - eqb, 0);  // ties the warp's segment takes
  compact_span(sm.scores, sp.lo, sp.hi, off + sp.gx + min(sp.ex, q), sp.ex, q, T, t0, s.idx + u * s.kmax, k,
               s.err);
  comp_bar();  // the group's index writes happen before gtid 0's release
  if (gtid == 0) sm.misc[0] = atom_add_acq_rel(&s.sel_cnt[u], 1u) == (uint32_t)NC - 1u;
  comp_bar();
  if (sm.misc[0])  // every chunk has read the unit's histogram: zero it for the next step
    for (int i = gtid; i < NB; i += kCompThreads) UH[i] = 0u;
}

// ---- selection item: a whole unit (contexts up to 32K tokens) ----------------------------
// One compute group scores all of the unit's tokens into shared memory, finds the
// threshold T from its histogram, counts each lane's span and compacts it as in a chunk:
// no hand-off with other groups.
template <int G>
__device__ void sel_unit(const DevState& s, SelUnitSmem& sm, int64_t u, int gtid) {
  constexpr int NB = 128 * G + 1;
  constexpr int kU = 4;  // code loads in flight per lane (more would spill in this kernel)
  const int b = (int)((u / s.Hkv) % s.B);
  const int N = (int)s.ntok[b];
  const int k = s.kcount[b];
  const int warp = gtid >> 5, lane = gtid & 31;
  const int WSEG = (((N + kCompWarps - 1) / kCompWarps) + 255) / 256 * 256;  // tokens per warp
  for (int i = gtid; i < NB; i += kCompThreads) sm.hist[i] = 0;
  QPlanes<G> qp;
  load_qplanes<G>(s, u, qp);
  comp_bar();
  const int w0 = warp * WSEG;
  const int w1 = (w0 + WSEG < N) ? w0 + WSEG : N;
  const uint4* src = s.codes + u * s.Nmax;
  constexpr int kPfRounds = 8;  // L2 prefetch of the codes this many rounds ahead
  if (lane == 0)
    for (int r = 1; r < kPfRounds; ++r) {
      const int pb = w0 + r * 32 * kU;
      if (pb < w1) prefetch_l2(src + pb, 16u * (uint32_t)((w1 - pb) < 32 * kU ? (w1 - pb) : 32 * kU));
    }
  for (int base = w0; base < w1; base += 32 * kU) {
    if (lane == 0) {
      const int pb = base + kPfRounds * 32 * kU;
      if (pb < w1) prefetch_l2(src + pb, 16u * (uint32_t)((w1 - pb) < 32 * kU ? (w1 - pb) : 32 * kU));
    }
    uint4 cv[kU];
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      const int t = base + 32 * j + lane;
      if (t < w1) cv[j] = ld_nc_v4(src + t);
    }
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      const int t = base + 32 * j + lane;
      if (t < w1) {
        const int sc = score_of<G>(cv[j], qp);
        sm.scores[t] = (uint16_t)sc;
        atomicAdd(&sm.hist[sc], 1u);
      }
    }
  }
  comp_bar();
  find_threshold<NB>(sm.hist, k, &sm.thr, &sm.misc[4], gtid);
  comp_bar();
  const int T = sm.thr.x < 0 ? 0 : (sm.thr.x >= NB ? NB - 1 : sm.thr.x);
  const int take_eq = k - sm.thr.y;  // ties taken, lowest index first
  const LaneSpan sp = span_counts(sm.scores, w0, w1, T, sm.wc[warp], lane);
  comp_bar();
  int off = 0, eqb = 0;
  for (int w = 0; w < warp; ++w) {
    off += sm.wc[w][0] + min(max(take_eq - eqb, 0), sm.wc[w][1]);
    eqb += sm.wc[w][1];
  }
  const int q = max(take_eq - eqb, 0);  // ties the warp's segment takes
  compact_span(sm.scores, sp.lo, sp.hi, off + sp.gx + min(sp.ex, q), sp.ex, q, T, 0, s.idx + u * s.kmax, k, s.err);
  comp_bar();  // the group's index writes happen before gtid 0's release
  if (gtid == 0) red_release_add_u32(&s.sel_cnt[u], 1u);
}

// ---- attention split -----------------------------------------------------------------
// Tensor-core (mma.sync m16n8k16, bf16 in, fp32 accumulate) split attention.  A split
// is split_rows (1024, or 2048 for k > 8192) selected rows; each of the 4 warps takes a
// quarter of them in chunks of
// 16 rows fed through its own 2-stage ring in shared memory: every row of a chunk is one
// 512-byte (d = 128) bulk copy on the TMA engine, issued by one lane and counted on the
// stage's mbarrier, so the next chunk's rows land while this chunk's math runs.  Per
// chunk:
//   S[16 rows x 8 heads] = K[16 x d] . Q^T[d x 8]      (G <= 8 query heads of the group
//                                                         on N; q fragments in registers)
//   online softmax per head on the accumulator fragments (scores in log2 units)
//   O^T[d x 8] += V^T[d x 16] . P^T[16 x 8]            (V^T via ldmatrix.trans; P split
//                                                         into bf16 hi + lo halves, so the
//                                                         weights keep ~16 mantissa bits)
// At the end of the split the 4 warps' {m, l, acc[d]} are merged in shared memory into one
// partial per split; the last split of the unit merges those by log-sum-exp.
__device__ __forceinline__ void mma_bf16_16816(float* c, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ void ldsm_x4(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

// bf16 pair (lo element in the low half) of two floats, round to nearest even
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const uint32_t a = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
  const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
  return a | (b << 16);
}
__device__ __forceinline__ float bf16_round(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// Running softmax state of one warp: heads 2*tig and 2*tig+1 (m = max score in log2
// units, l = sum of weights) and O^T fragments acc[m-block][4].
template <int D>
struct AttAcc {
  float m0, m1, l0, l1;
  float acc[D / 16][4];
};

// One 16-row chunk (rows[r][0..D) = K row, rows[r][D..2D) = V row; rows >= nrows hold
// finite values and are masked).
template <int D, int ROWW>
__device__ __forceinline__ void chunk_math(const uint16_t (*rows)[ROWW], int nrows, const uint32_t (*qb)[2],
                                           float qscale, AttAcc<D>& A, int lane) {
  constexpr int KS = D / 16;  // k-steps of S = K Q^T, also m-blocks of O^T
  const int gid = lane >> 2, tig = lane & 3;
  float sf[4] = {0.f, 0.f, 0.f, 0.f};
  {
    const int ar = (lane & 7) + 8 * ((lane >> 3) & 1), ac = 8 * (lane >> 4);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t a[4];
      ldsm_x4(a, &rows[ar][ks * 16 + ac]);
      mma_bf16_16816(sf, a, qb[ks]);
    }
  }
  // rows gid (sf[0], sf[1]) and gid + 8 (sf[2], sf[3]); heads 2*tig, 2*tig+1
  const float s00 = gid < nrows ? sf[0] * qscale : -INFINITY;
  const float s01 = gid < nrows ? sf[1] * qscale : -INFINITY;
  const float s10 = gid + 8 < nrows ? sf[2] * qscale : -INFINITY;
  const float s11 = gid + 8 < nrows ? sf[3] * qscale : -INFINITY;
  float mx0 = fmaxf(s00, s10), mx1 = fmaxf(s01, s11);
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
  }
  const float mn0 = fmaxf(A.m0, mx0), mn1 = fmaxf(A.m1, mx1);
  const float al0 = exp2f(A.m0 - mn0), al1 = exp2f(A.m1 - mn1);
  const float p00 = exp2f(s00 - mn0), p10 = exp2f(s10 - mn0);
  const float p01 = exp2f(s01 - mn1), p11 = exp2f(s11 - mn1);
  float rs0 = p00 + p10, rs1 = p01 + p11;
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    rs0 += __shfl_xor_sync(0xffffffffu, rs0, o);
    rs1 += __shfl_xor_sync(0xffffffffu, rs1, o);
  }
  A.l0 = A.l0 * al0 + rs0;
  A.l1 = A.l1 * al1 + rs1;
  A.m0 = mn0;
  A.m1 = mn1;
#pragma unroll
  for (int mb = 0; mb < KS; ++mb) {
    A.acc[mb][0] *= al0;
    A.acc[mb][2] *= al0;
    A.acc[mb][1] *= al1;
    A.acc[mb][3] *= al1;
  }
  // P^T fragments (B operand): rows 2*tig, 2*tig+1, 2*tig+8, 2*tig+9 of head gid.
  // P[r][hd] sits in lane 4*(r%8) + hd/2: element hd%2 of (p00,p01) for r < 8, of
  // (p10,p11) for r >= 8.
  const int sa = 8 * tig + (gid >> 1), sb = sa + 4;
  const bool odd = gid & 1;
  const float xa0 = __shfl_sync(0xffffffffu, p00, sa), xa1 = __shfl_sync(0xffffffffu, p01, sa);
  const float xb0 = __shfl_sync(0xffffffffu, p00, sb), xb1 = __shfl_sync(0xffffffffu, p01, sb);
  const float ya0 = __shfl_sync(0xffffffffu, p10, sa), ya1 = __shfl_sync(0xffffffffu, p11, sa);
  const float yb0 = __shfl_sync(0xffffffffu, p10, sb), yb1 = __shfl_sync(0xffffffffu, p11, sb);
  const float pr0 = odd ? xa1 : xa0, pr1 = odd ? xb1 : xb0;  // rows 2*tig, 2*tig+1
  const float pr8 = odd ? ya1 : ya0, pr9 = odd ? yb1 : yb0;  // rows 2*tig+8, 2*tig+9
  uint32_t bh[2], bl[2];
  bh[0] = pack_bf16(pr0, pr1);
  bh[1] = pack_bf16(pr8, pr9);
  bl[0] = pack_bf16(pr0 - bf16_round(pr0), pr1 - bf16_round(pr1));
  bl[1] = pack_bf16(pr8 - bf16_round(pr8), pr9 - bf16_round(pr9));
  // O^T += V^T P^T
  {
    const int vr = (lane & 7) + 8 * (lane >> 4), vc = 8 * ((lane >> 3) & 1);
#pragma unroll
    for (int mb = 0; mb < KS; ++mb) {
      uint32_t a[4];
      ldsm_x4_trans(a, &rows[vr][D + mb * 16 + vc]);
      mma_bf16_16816(A.acc[mb], a, bh);
      mma_bf16_16816(A.acc[mb], a, bl);
    }
  }
}

// bars: this warp's kAttStages mbarriers (one per ring stage); phase: bit st = parity of
// the next completion of stage st, carried across items.
template <int D>
__device__ void attend_split(const DevState& s, AttSmem<D>& sm, uint64_t* bars, uint32_t& phase,
                             const uint16_t* __restrict__ q, float* __restrict__ out, int64_t u, int split,
                             int gtid) {
  constexpr int ROWW = AttSmem<D>::ROWW;
  const int WROWS = s.split_rows / kCompWarps;
  constexpr int ST = kAttStages;
  const int h = (int)(u % s.Hkv);
  const int b = (int)((u / s.Hkv) % s.B);
  const int l = (int)(u / ((int64_t)s.Hkv * s.B));
  const int G = s.G;
  const int warp = gtid >> 5, lane = gtid & 31, gid = lane >> 2, tig = lane & 3;
  const int64_t N = s.ntok[b];
  const int64_t k = s.kcount[b];
  const int64_t r0 = (int64_t)split * s.split_rows + (int64_t)warp * WROWS;
  const int64_t r1 = (r0 + WROWS < k) ? r0 + WROWS : k;
  const int nch = r1 > r0 ? (int)((r1 - r0 + 15) / 16) : 0;
  const bool persistent = s.decision[u] == CLO_DEC_PERSIST;
  const int32_t* ix = s.idx + u * s.kmax;
  const uint16_t* src;
  if (persistent) {
    const int p = s.persist_slot[l * s.Hkv + h];
    src = s.resident + ((((int64_t)l * s.B + b) * s.P + p) * s.Nmax) * (2 * D);
  } else {
    src = s.slots + (u * s.kmax) * (2 * D);
  }
  // source row of lane's row (lane < 16) in chunk c: persistent units read their rows
  // through the selection's indices, loaded one chunk ahead of the copy that needs them
  auto row_of = [&](int c) -> int64_t {
    const int64_t t = r0 + 16 * c + lane;
    if (lane >= 16 || c >= nch || t >= r1) return -1;
    if (!persistent) return t;
    const int64_t v = __ldcg(ix + t);
    if (v < 0 || v >= N) {
      atomicOr(s.err, kErrBounds);
      return 0;
    }
    return v;
  };
  auto issue = [&](int c, int64_t row) {
    const int st = c % ST;
    const int nr = (int)((r1 - (r0 + 16 * c)) < 16 ? (r1 - (r0 + 16 * c)) : 16);
    fence_proxy_async_smem();  // this warp's earlier generic accesses of the stage first
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(&bars[st], (uint32_t)nr * 4 * D);
    __syncwarp();
    if (lane < nr) {
      bulk_copy_g2s(&sm.rows[warp][st][lane][0], src + row * (2 * D), 4 * D, &bars[st]);
    } else if (lane < 16) {  // rows past the end: zeros, so the masked rows stay finite
      uint4* z = reinterpret_cast<uint4*>(&sm.rows[warp][st][lane][0]);
#pragma unroll 4
      for (int e = 0; e < ROWW / 8; ++e) z[e] = make_uint4(0, 0, 0, 0);
    }
  };
  int64_t nxt = row_of(0);
  for (int c = 0; c < ST - 1 && c < nch; ++c) {
    issue(c, nxt);
    nxt = row_of(c + 1);
  }
  // Q^T fragments (B operand): head gid, dims 2*tig (+1, +8, +9) of each k-step
  uint32_t qb[D / 16][2];
  {
    const uint16_t* qg = q + (((int64_t)(l - s.q_l0) * s.B + b) * s.Hq + (int64_t)h * G) * D;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      if (gid < G) {
        qb[ks][0] = *reinterpret_cast<const uint32_t*>(qg + gid * D + ks * 16 + 2 * tig);
        qb[ks][1] = *reinterpret_cast<const uint32_t*>(qg + gid * D + ks * 16 + 2 * tig + 8);
      } else {
        qb[ks][0] = qb[ks][1] = 0u;
      }
    }
  }
  const float qscale = 1.4426950408889634f * rsqrtf((float)D);  // scores in log2 units
  AttAcc<D> A;
  A.m0 = A.m1 = -INFINITY;
  A.l0 = A.l1 = 0.f;
#pragma unroll
  for (int mb = 0; mb < D / 16; ++mb) A.acc[mb][0] = A.acc[mb][1] = A.acc[mb][2] = A.acc[mb][3] = 0.f;
  for (int c = 0; c < nch; ++c) {
    if (c + ST - 1 < nch) {
      issue(c + ST - 1, nxt);
      nxt = row_of(c + ST);
    }
    const int st = c % ST;
    const uint32_t par = (phase >> st) & 1u;
    bool ok = mbar_wait_bounded(&bars[st], par, s.err, (uint64_t)s.wait_timeout_ns);
    if (!ok) ok = mbar_wait_bounded(&bars[st], par, s.err, (uint64_t)s.wait_timeout_ns);  // drain
    phase ^= 1u << st;
    const int nrows = (int)((r1 - (r0 + 16 * c)) < 16 ? (r1 - (r0 + 16 * c)) : 16);
    if (ok) chunk_math<D, ROWW>(sm.rows[warp][st], nrows, qb, qscale, A, lane);
    __syncwarp();  // the stage is refilled by a later chunk
  }

  // the warp's partial {m, l, acc[d]} per head into its own ring region (its copies are
  // all complete): wp[g][D + 2]
  float* wp = reinterpret_cast<float*>(&sm.rows[warp][0][0][0]);
  {
    const int h0 = 2 * tig, h1 = 2 * tig + 1;
#pragma unroll
    for (int mb = 0; mb < D / 16; ++mb) {
      if (h0 < G) {
        wp[h0 * (D + 2) + 2 + mb * 16 + gid] = A.acc[mb][0];
        wp[h0 * (D + 2) + 2 + mb * 16 + gid + 8] = A.acc[mb][2];
      }
      if (h1 < G) {
        wp[h1 * (D + 2) + 2 + mb * 16 + gid] = A.acc[mb][1];
        wp[h1 * (D + 2) + 2 + mb * 16 + gid + 8] = A.acc[mb][3];
      }
    }
    if (gid == 0) {
      if (h0 < G) {
        wp[h0 * (D + 2) + 0] = A.m0;
        wp[h0 * (D + 2) + 1] = A.l0;
      }
      if (h1 < G) {
        wp[h1 * (D + 2) + 0] = A.m1;
        wp[h1 * (D + 2) + 1] = A.l1;
      }
    }
  }
  comp_bar();
  // the split's partial: the 4 warps merged by log-sum-exp (a warp without rows has l = 0)
  {
    float* part = s.part + ((u * s.nsplit + split) * G) * (D + 2);
    const float* w0 = reinterpret_cast<const float*>(&sm.rows[0][0][0][0]);
    constexpr int WSTRIDE = (int)(sizeof(sm.rows[0]) / sizeof(float));
    for (int e = gtid; e < G * (D + 2); e += kCompThreads) {
      const int g = e / (D + 2), j = e % (D + 2);
      float mw[kCompWarps], lw[kCompWarps];
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kCompWarps; ++w) {
        mw[w] = w0[w * WSTRIDE + g * (D + 2)];
        lw[w] = w0[w * WSTRIDE + g * (D + 2) + 1];
        if (lw[w] > 0.f) M = fmaxf(M, mw[w]);
      }
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kCompWarps; ++w) {
        const float sc = lw[w] > 0.f ? exp2f(mw[w] - M) : 0.f;
        v = fmaf(j == 1 ? lw[w] : w0[w * WSTRIDE + g * (D + 2) + j], sc, v);
      }
      part[e] = j == 0 ? M : v;
    }
  }
  __threadfence();
  comp_bar();
  if (gtid == 0) {
    const uint32_t prev = atomicAdd(&s.unit_done[u], 1u);
    sm.last = (prev == (uint32_t)s.nsplit - 1u);
  }
  comp_bar();
  if (!sm.last) return;
  __threadfence();
  // merge: per head, weights w_sp = exp2(m_sp - M) of the splits' partials (into shared
  // memory), then out[j] = sum_sp w_sp acc_sp[j] / sum_sp w_sp l_sp
  const int np = s.nsplit;
  const float* pu = s.part + (u * np) * G * (D + 2);
  float* og = out + (((int64_t)(l - s.q_l0) * s.B + b) * s.Hq + (int64_t)h * G) * D;
  float* w = reinterpret_cast<float*>(&sm.rows[0][0][0][0]);  // np floats
  for (int g = 0; g < G; ++g) {
    float mx = -INFINITY;
    for (int sp = gtid; sp < np; sp += kCompThreads) {
      const float* ps = pu + (sp * G + g) * (D + 2);
      if (__ldcg(ps + 1) > 0.f) mx = fmaxf(mx, __ldcg(ps));
    }
    mx = warp_max(mx);
    if (lane == 0) sm.red[warp] = mx;
    comp_bar();
    const float M = fmaxf(fmaxf(sm.red[0], sm.red[1]), fmaxf(sm.red[2], sm.red[3]));
    float ls = 0.f;
    for (int sp = gtid; sp < np; sp += kCompThreads) {
      const float* ps = pu + (sp * G + g) * (D + 2);
      const float lsp = __ldcg(ps + 1);
      const float ww = lsp > 0.f ? exp2f(__ldcg(ps) - M) : 0.f;
      w[sp] = ww;
      ls = fmaf(lsp, ww, ls);
    }
    ls = warp_sum(ls);
    comp_bar();  // everyone has read sm.red (max)
    if (lane == 0) sm.red[warp] = ls;
    comp_bar();
    const float Lsum = sm.red[0] + sm.red[1] + sm.red[2] + sm.red[3];
    for (int j = gtid; j < D; j += kCompThreads) {
      float O = 0.f;
      for (int sp = 0; sp < np; ++sp) {
        const float ww = w[sp];
        if (ww != 0.f) O = fmaf(__ldcg(pu + (sp * G + g) * (D + 2) + 2 + j), ww, O);
      }
      og[g * D + j] = O / Lsum;
    }
    comp_bar();  // w and sm.red are reused by the next head
  }
  if (gtid == 0) s.unit_done[u] = 0u;
}

// ---- fetch warps -----------------------------------------------------------------------
// A fetch item is one chunk of kChunkRows selected rows of a missed unit.  The chunk's
// indices are checked and staged in shared memory first, so every round trip to host
// memory is a single dependent load; each round keeps kFetchUnroll 16-byte loads per
// lane in flight (with d = 128 one warp-wide load is one whole 512-byte K|V record).
// bf16 records: K|V rows copied as they are (16-byte loads, one record per warp-wide load).
template <int D, int FU>
__device__ __forceinline__ void copy_rows(const DevState& s, int64_t u, int64_t r0, int nr, const int32_t* sidx,
                                          int lane) {
  constexpr int VPR = D / 4;  // 16-byte vectors per K|V record
  const uint4* pool = reinterpret_cast<const uint4*>(s.pool) + u * s.Nmax * VPR;
  uint4* slot = reinterpret_cast<uint4*>(s.slots) + (u * s.kmax + r0) * VPR;
  const int total = nr * VPR;
  for (int e0 = lane; e0 < total; e0 += 32 * FU) {
    uint4 v[FU];
#pragma unroll
    for (int j = 0; j < FU; ++j) {
      const int e = e0 + 32 * j;
      v[j] = make_uint4(0, 0, 0, 0);
      if (e < total) {
        const int t = sidx[e / VPR];
        if (t >= 0) v[j] = ld_nc_v4(pool + (int64_t)t * VPR + (e % VPR));
      }
    }
#pragma unroll
    for (int j = 0; j < FU; ++j) {
      const int e = e0 + 32 * j;
      if (e < total) slot[e] = v[j];
    }
  }
}

// Quantised records: lane (row slot, code vector j) loads one 16-byte code vector from the
// host pool and its group's (scale, min) from HBM, and writes the dequantised bf16 values
// to the slot row.
template <int D, int FU, int BITS>
__device__ __forceinline__ void copy_rows_q(const DevState& s, int64_t u, int64_t r0, int nr, const int32_t* sidx,
                                            int lane) {
  using Q = QRec<D, BITS>;
  constexpr int PV = Q::kCodeVecs;  // lanes per row
  constexpr int RPI = 32 / PV;      // rows per warp-wide round
  const unsigned char* pool = reinterpret_cast<const unsigned char*>(s.pool) + u * s.Nmax * Q::kBytes;
  const float2* params = s.qparams + u * s.Nmax * Q::kGroups;
  uint4* slot = reinterpret_cast<uint4*>(s.slots) + (u * s.kmax + r0) * (D / 4);
  const int rl = lane / PV, j = lane % PV, gi = j / Q::kVecsPerGroup;
  for (int rb = 0; rb < nr; rb += RPI * FU) {
    uint4 cv[FU];
    float2 pp[FU];
#pragma unroll
    for (int f = 0; f < FU; ++f) {
      const int r = rb + f * RPI + rl;
      cv[f] = make_uint4(0, 0, 0, 0);
      pp[f] = make_float2(0.f, 0.f);
      if (r < nr) {
        const int t = sidx[r];
        if (t >= 0) {
          cv[f] = ld_nc_v4(reinterpret_cast<const uint4*>(pool + (int64_t)t * Q::kBytes) + j);
          pp[f] = __ldg(params + (int64_t)t * Q::kGroups + gi);
        }
      }
    }
#pragma unroll
    for (int f = 0; f < FU; ++f) {
      const int r = rb + f * RPI + rl;
      if (r < nr) dequant_vec<BITS>(cv[f], pp[f].x, pp[f].y, slot + (int64_t)r * (D / 4) + j * Q::kOutVecs);
    }
  }
}

template <int D, int FU>
__device__ void fetch_role(const DevState& s, const int* pre_m, int n_miss, int lane, int32_t* sidx) {
  constexpr int kFetchUnroll = FU;
  const int NS = s.nchunk, L = s.L, BH = s.B * s.Hkv;
  const int RS = s.fetch_rows, SUB = kChunkRows / RS;
  const int64_t per_unit = (int64_t)NS * SUB;
  const int64_t n_items = (int64_t)n_miss * per_unit;
  while (true) {
    unsigned item = 0;
    if (lane == 0) item = atomicAdd(&s.queue[0], 1u);
    item = __shfl_sync(0xffffffffu, item, 0);
    if ((int64_t)item >= n_items) break;
    const int p = (int)(item / per_unit);
    const int rest = (int)(item % per_unit);
    const int c = rest / SUB;
    const int l = layer_of(pre_m, L, p);
    const int64_t u = s.miss_list[(int64_t)l * BH + (p - pre_m[l])];
    const int b = (int)((u / s.Hkv) % s.B);
    const int64_t k = s.kcount[b];
    const int64_t N = s.ntok[b];
    const int64_t r0 = (int64_t)c * kChunkRows + (int64_t)(rest % SUB) * RS;
    const int nr = (int)((r0 + RS < k) ? RS : (k - r0 > 0 ? k - r0 : 0));
    if (nr > 0) {
      if (lane == 0) {  // the unit's selection: compute groups, earlier in their queue
        const uint64_t tw = s.timeline ? global_timer_ns() : 0;
        wait_flag(&s.sel_cnt[u], (uint32_t)s.nch_miss, s);
        if (s.timeline) {
          const uint64_t t1 = global_timer_ns();
          atomicAdd(&s.timeline[TL_FETCH_WAIT_NS], t1 - tw);
          atomicCAS(&s.timeline[TL_FETCH_FIRST], 0ull, t1);
        }
      }
      __syncwarp();
      const int32_t* ix = s.idx + u * s.kmax + r0;
      for (int i = lane; i < nr; i += 32) {
        int32_t t = __ldcg(ix + i);
        if (t < 0 || (int64_t)t >= N) {
          atomicOr(s.err, kErrBounds);
          t = -1;
        }
        sidx[i] = t;
      }
      __syncwarp();
      if (s.kv_bits == 16)
        copy_rows<D, kFetchUnroll>(s, u, r0, nr, sidx, lane);
      else if (s.kv_bits == 4)
        copy_rows_q<D, kFetchUnroll, 4>(s, u, r0, nr, sidx, lane);
      else
        copy_rows_q<D, kFetchUnroll, 2>(s, u, r0, nr, sidx, lane);
    }
    __threadfence();
    __syncwarp();  // also: sidx is rewritten by the next item
    if (lane == 0 && l != s.drop_flag_layer) red_release_add_u32(&s.ready[u * NS + c], 1u);
    if (lane == 0 && s.timeline) atomicMax(&s.timeline[TL_FETCH_END], global_timer_ns());
  }
}

// ---- the kernel ------------------------------------------------------------------------
// FW fetch warps + one compute group per CTA; MINB CTAs per SM.
template <int D, int G, int FW, int MINB, int FU = kFetchUnroll>
__global__ void __launch_bounds__(32 * (FW + kCompWarps), MINB)
    k_step_fused(DevState s, const uint16_t* __restrict__ q, float* __restrict__ out) {
  using Smem = CompSmem<D>;
  __shared__ int pre[3][kMaxLayers + 1];  // hit, persistent, missed lists
  __shared__ long long sec_start[6];
  __shared__ int s_item;
  __shared__ unsigned long long s_t0, s_t1;  // start of the group's item, end of its waits (timing mode)
  __shared__ int32_t fidx[FW][kChunkRows];
  // mbarriers of the compute warps' row rings (outside the union: selection items reuse
  // the ring memory, never the barriers)
  __shared__ __align__(8) uint64_t att_bar[kCompWarps][kAttStages];
  extern __shared__ __align__(128) unsigned char dsm[];
  Smem& sm = *reinterpret_cast<Smem*>(dsm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = s.L;
  if (tid == 0) {
    if (s.timeline) atomicCAS(&s.timeline[TL_START], 0ull, global_timer_ns());
    int a[3] = {0, 0, 0};
    for (int j = 0; j < 3; ++j) pre[j][0] = 0;
    for (int l = 0; l < L; ++l)
      for (int j = 0; j < 3; ++j) {
        a[j] += s.lcnt[j * L + l];
        pre[j][l + 1] = a[j];
      }
    // compute queue: selection chunks of the missed units, then of the persistent units
    // (layer by layer, the chunks of a unit next to each other), then attention splits
    // of reused, persistent and missed units
    const long long nh = a[0], np = a[1], nm = a[2], NC = s.nch, NCM = s.nch_miss, NS = s.nsplit;
    const long long size[5] = {nm * NCM, np * NC, nh * NS, np * NS, nm * NS};
    sec_start[0] = 0;
    for (int i = 0; i < 5; ++i) sec_start[i + 1] = sec_start[i] + size[i];
  }
  if (s.step_bytes && s.l1 == s.L && blockIdx.x == 0 && tid == 0) {
    // the step's last launch: its reuse decisions (and every earlier layer's) are counted,
    // so the cumulative byte counters are the totals after this step
    unsigned long long hb = 0, mb = 0;
    for (int i = 0; i < kCtrLanes; ++i) {
      hb += s.total_ctr[C_HOST_BYTES * kCtrLanes + i];
      mb += s.total_ctr[C_HBM_BYTES * kCtrLanes + i];
    }
    const int64_t slot = (s.step_index % kStepHist) * 2;
    s.step_bytes[slot] = hb;
    s.step_bytes[slot + 1] = mb;
  }
  if (s.adapt_active && blockIdx.x == 0) {
    // online thresholds: fold this step's mean adjacent-step cosine of each (layer,
    // kv head) into s_hat; the decide kernel, finished before this launch, summed them
    for (int lh = s.l0 * s.Hkv + tid; lh < s.l1 * s.Hkv; lh += blockDim.x) {
      const uint32_t n = s.cos_cnt[lh];
      if (n) {
        const double sh = (1.0 - s.tau_ema) * s.shat[lh] + s.tau_ema * (s.cos_sum[lh] / (double)n);
        s.shat[lh] = sh;
        s.tau[lh] = (float)(sh - (double)s.tau_offset);
      }
      s.cos_sum[lh] = 0.0;
      s.cos_cnt[lh] = 0u;
    }
  }
  __syncthreads();
  if (warp < FW) {
    fetch_role<D, FU>(s, pre[2], pre[2][L], lane, fidx[warp]);
    return;  // no block-wide barrier after this point
  }
  const int gtid = tid - 32 * FW;
  const int BH = s.B * s.Hkv;
  const int NC = s.nch;
  const long long total = sec_start[5];
  if (lane < kAttStages) mbar_init(&att_bar[gtid >> 5][lane], 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncwarp();
  uint32_t att_phase = 0;  // bit st: parity of the next completion of this warp's stage st
  while (true) {
    if (gtid == 0) s_item = (int)atomicAdd(&s.queue[1], 1u);
    comp_bar();
    const long long item = s_item;
    if (item >= total) break;
    int sec = 0;
    while (item >= sec_start[sec + 1]) ++sec;
    const long long j = item - sec_start[sec];
    const int list = (sec == 0 || sec == 4) ? 2 : ((sec == 1 || sec == 3) ? 1 : 0);
    const int* pl = pre[list];
    const int32_t* lst = list == 2 ? s.miss_list : (list == 1 ? s.pers_list : s.hit_list);
    if (s.timeline && gtid == 0) s_t0 = global_timer_ns();
    if (sec <= 1) {  // selection chunk
      // missed units' chunks first (their fetch waits for them), then persistent units':
      // whole units when they fit one group's shared memory in a large launch, else chunks
      const int nc = sec == 0 ? s.nch_miss : NC;
      const int p = (int)(j / nc), c = (int)(j % nc);
      const int l = layer_of(pl, L, p);
      const int64_t u = lst[(int64_t)l * BH + (p - pl[l])];
      if (sec == 1 && NC == 1 && s.sel_chunk >= s.Nmax)
        sel_unit<G>(s, sm.unit, u, gtid);
      else
        sel_chunk<G>(s, sm.sel, u, c, sec == 0 ? s.sel_chunk_miss : s.sel_chunk, nc, gtid);
      if (s.timeline && gtid == 0) {
        const uint64_t t1 = global_timer_ns();
        atomicMax(&s.timeline[sec == 0 ? TL_SEL_MISS_END : TL_SEL_PERS_END], t1);
        atomicAdd(&s.timeline[TL_SEL_SUM_NS], t1 - s_t0);
        atomicAdd(&s.timeline[TL_SEL_ITEMS], 1ull);
      }
    } else {  // attention split
      const int p = (int)(j / s.nsplit), c = (int)(j % s.nsplit);
      const int l = layer_of(pl, L, p);
      const int64_t u = lst[(int64_t)l * BH + (p - pl[l])];
      const int b = (int)((u / s.Hkv) % s.B);
      const int64_t r0 = (int64_t)c * s.split_rows;
      if (s.timeline && gtid == 0) atomicCAS(&s.timeline[TL_ATT_FIRST], 0ull, s_t0);
      if (sec == 3) {
        if (gtid == 0) wait_flag(&s.sel_cnt[u], (uint32_t)NC, s);
        comp_bar();
      } else if (sec == 4 && r0 < s.kcount[b]) {
        if (gtid == 0) {
          const int kPer = s.split_rows / kChunkRows;  // the fetch chunks this split reads
          const uint32_t subs = (uint32_t)(kChunkRows / s.fetch_rows);  // fetch items per chunk
          for (int fc = c * kPer; fc < (c + 1) * kPer && (int64_t)fc * kChunkRows < s.kcount[b]; ++fc)
            wait_flag(&s.ready[u * s.nchunk + fc], subs, s);
          if (s.timeline) atomicAdd(&s.timeline[TL_ATT_WAIT_NS], global_timer_ns() - s_t0);
        }
        comp_bar();
      }
      if (s.timeline && gtid == 0) s_t1 = global_timer_ns();
      attend_split<D>(s, sm.att, att_bar[gtid >> 5], att_phase, q, out, u, c, gtid);
      if (s.timeline && gtid == 0) {
        const uint64_t t1 = global_timer_ns();
        atomicMax(&s.timeline[TL_COMP_END], t1);
        atomicAdd(&s.timeline[TL_ATT_SUM_NS], t1 - s_t0);
        atomicAdd(&s.timeline[TL_ATT_RUN_NS], t1 - s_t1);
        atomicAdd(&s.timeline[TL_ATT_ITEMS], 1ull);
      }
    }
    // this item's generic shared-memory accesses happen before any later bulk copy into
    // the same memory (the copies are issued after the next comp_bar)
    fence_proxy_async_smem();
    comp_bar();
  }
}

template <int D, int G, int FW, int MINB, int FU>
int fused_grid() {
  static int grid = 0;
  if (grid == 0) {
    auto kern = k_step_fused<D, G, FW, MINB, FU>;
    const int smem = (int)sizeof(CompSmem<D>);
    int dev = 0, sms = 0, per_sm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32 * (FW + kCompWarps), smem);
    grid = sms * (per_sm > 0 ? per_sm : 1);
  }
  return grid;
}

template <int D, int G, int FW, int MINB, int FU = kFetchUnroll>
cudaError_t launch_v(const DevState& s, const uint16_t* q, float* out, cudaStream_t st) {
  k_step_fused<D, G, FW, MINB, FU><<<fused_grid<D, G, FW, MINB, FU>(), 32 * (FW + kCompWarps),
                                   sizeof(CompSmem<D>), st>>>(s, q, out);
  return cudaGetLastError();
}

template <int D, int G>
cudaError_t launch_dg(const DevState& s, const uint16_t* q, float* out, cudaStream_t st) {
  // the selection's waits need all chunks of a unit running at once
  const int nc = s.nch > s.nch_miss ? s.nch : s.nch_miss;
  if (fused_grid<D, G, 1, 3, kFetchUnroll>() < nc) return cudaErrorInvalidConfiguration;
  return launch_v<D, G, 1, 3>(s, q, out, st);
}

template <int D>
cudaError_t launch_d(const DevState& s, const uint16_t* q, float* out, cudaStream_t st) {
  switch (s.G) {
    case 1: return launch_dg<D, 1>(s, q, out, st);
    case 2: return launch_dg<D, 2>(s, q, out, st);
    case 3: return launch_dg<D, 3>(s, q, out, st);
    case 4: return launch_dg<D, 4>(s, q, out, st);
    case 5: return launch_dg<D, 5>(s, q, out, st);
    case 6: return launch_dg<D, 6>(s, q, out, st);
    case 7: return launch_dg<D, 7>(s, q, out, st);
    case 8: return launch_dg<D, 8>(s, q, out, st);
    default: return cudaErrorInvalidValue;
  }
}

// Dequantises the records of tokens [t0, t1) of unit u into bf16 rows at dst.
template <int D, int BITS>
__device__ __forceinline__ void fill_q(const DevState& s, int64_t u, int64_t t0, int64_t t1, uint4* dst) {
  using Q = QRec<D, BITS>;
  const unsigned char* pool = reinterpret_cast<const unsigned char*>(s.pool) + (u * s.Nmax + t0) * Q::kBytes;
  const float2* params = s.qparams + (u * s.Nmax + t0) * Q::kGroups;
  const int64_t n = (t1 - t0) * Q::kCodeVecs;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = e / Q::kCodeVecs;
    const int j = (int)(e % Q::kCodeVecs);
    const unsigned char* rec = pool + t * Q::kBytes;
    const float2 pp = __ldg(params + t * Q::kGroups + j / Q::kVecsPerGroup);
    dequant_vec<BITS>(ld_nc_v4(reinterpret_cast<const uint4*>(rec) + j), pp.x, pp.y,
                      dst + t * (D / 4) + j * Q::kOutVecs);
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
    uint4* dst = reinterpret_cast<uint4*>(s.resident) + ((((int64_t)l * s.B + b) * s.P + p) * s.Nmax + t0) * vpr;
    if (s.kv_bits != 16) {  // quantised pool: dequantise every code vector
      if (s.d == 128)
        s.kv_bits == 4 ? fill_q<128, 4>(s, u, t0, tend, dst) : fill_q<128, 2>(s, u, t0, tend, dst);
      else
        s.kv_bits == 4 ? fill_q<64, 4>(s, u, t0, tend, dst) : fill_q<64, 2>(s, u, t0, tend, dst);
      continue;
    }
    const int64_t n = (tend - t0) * vpr;
    const uint4* src = reinterpret_cast<const uint4*>(s.pool) + (u * s.Nmax + t0) * vpr;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x)
      dst[e] = ld_nc_v4(src + e);
  }
}

}  // namespace

cudaError_t launch_step_fused(const DevState& s, const uint16_t* q, float* out, cudaStream_t st) {
  if (s.L > kMaxLayers || s.nbp > kNBPad) return cudaErrorInvalidValue;
  if (s.d == 128) return launch_d<128>(s, q, out, st);
  if (s.d == 64) return launch_d<64>(s, q, out, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_resident_fill(const DevState& s, int64_t t0, int64_t t1, cudaStream_t st) {
  if (s.P <= 0 || s.resident == nullptr || t1 <= t0) return cudaSuccess;
  const int64_t U = (int64_t)s.L * s.B * s.Hkv;
  dim3 grid(64, (unsigned)(U < 65535 ? U : 65535));
  k_resident_fill<<<grid, 256, 0, st>>>(s, t0, t1);
  return cudaGetLastError();
}

}  // namespace clo
