// One persistent, warp-specialised kernel per decode step: selection of the
// persistent units, zero-copy fetch of missed heads' rows and split-K sparse
// attention, ordered by device-side flags only.  (Missed units are selected by the
// launch just before, so their fetch can start as soon as this kernel does.)
//
// Each CTA holds one fetch warp and one 4-warp compute group (6 CTAs per SM).  One
// fetch warp per CTA keeps enough host-link requests in flight to saturate the link
// without queueing so many that the HBM traffic of the compute groups waits behind
// them.
//   * The compute group takes items from one queue, in this order:
//       1. selection of the persistent units, layer by layer:
//          score chunk  -> histogram of the chunk's scores (codes streamed into shared
//                          memory by 1-D bulk copies on the TMA engine);
//          finalize     -> threshold score T of the unit and each chunk's output offset
//                          and tie quota (ties go to the lowest token index);
//          compact chunk-> recompute the scores, write the chunk's selected indices in
//                          ascending order;
//       2. attention splits: reused units, persistent units, then missed units in layer
//          order.
//     score[t] = sum_g (128 - popc(qcode_g ^ kcode_t)) (HATA hash scorer, "CLO
//     (2511.14510) - L3 Per-Paper Synthesis", section 3.2); k = 10 % of the context
//     (section 2.2); out_g = sum_r softmax_r(q_g . k_r / sqrt(d)) v_r over the rows.
//   * Fetch warps copy the selected K|V rows of missed units from pinned host memory
//     into the units' on-GPU cache slots with 16-byte loads, chunk by chunk in layer
//     order, and release one ready flag per chunk (CLO abstract, feature (3):
//     zero-copy transfer engine and GPU-centric synchronisation; the fetch runs
//     ahead of the attention that consumes it, as CLO prefetches a layer ahead,
//     section 5.6).
// Every wait targets work that sits earlier in the compute queue (or a fetch, which
// itself waits only on earlier compute items), so the waits form no cycle; each
// wait is bounded by the context's timeout and reports CLO_ERR_TIMEOUT.
#include "clo_internal.cuh"

namespace clo {

namespace {

constexpr int kFetchWarps = 1;
constexpr int kCompWarps = 4;
constexpr int kCompThreads = 32 * kCompWarps;
constexpr int kFThreads = 32 * (kFetchWarps + kCompWarps);
constexpr int kFetchUnroll = 8;
constexpr int kAttTile = 32;
constexpr int kSelTile = 512;  // tokens per bulk copy (8 KB)
constexpr int kSelStages = 3;
constexpr int kMaxChunks = (int)(kMaxTokens / kSelChunk);
constexpr uint64_t kMbarLimitNs = 2000000000ull;

__device__ __forceinline__ void comp_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kCompThreads) : "memory"); }

// Barrier of the compute group that also ANDs a predicate over its threads, so a
// decision taken per thread (a bounded wait that may time out) becomes uniform.
__device__ __forceinline__ bool comp_bar_and(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred a, b;\n\t"
      "setp.ne.u32 a, %1, 0;\n\t"
      "bar.red.and.pred b, 1, %2, a;\n\t"
      "selp.u32 %0, 1, 0, b;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)p), "n"(kCompThreads)
      : "memory");
  return r != 0;
}

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

// Bounded wait until *flag >= target (acquire); on timeout: error word + counter.
__device__ void wait_flag(const uint32_t* flag, uint32_t target, const DevState& s) {
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
    if (ns < 2048) ns <<= 1;
  }
}

template <int D>
struct AttSmem {
  static constexpr int ROWW = 2 * D + 8;  // bf16 per smem row, padded by 16 bytes
  static constexpr int NG = kCompThreads / D;
  float qs[kMaxG][D];
  uint16_t rows[kAttTile][ROWW];
  float sc[kMaxG][kAttTile];
  float m_run[kMaxG], l_run[kMaxG], alpha[kMaxG];
  float red[NG > 1 ? NG : 1][kMaxG][D];
  int last;
};

struct SelSmem {
  uint4 ring[kSelStages][kSelTile];
  uint32_t hist[kNBPad];
  int cgt[kMaxChunks], ceq[kMaxChunks];
  int wc[kCompWarps][2];
  int misc[4];
};

template <int D>
union CompSmem {
  AttSmem<D> att;
  SelSmem sel;
};

struct Ring {
  uint64_t* bar;
  uint32_t n;  // tiles consumed so far by this group (uniform over the group)
};

// Streams tiles of a unit's chunk of codes through the ring; calls f(tile_index, tile_ptr, ntok).
template <class F>
__device__ void stream_codes(const DevState& s, SelSmem& sm, Ring& ring, const uint4* src, int len, int gtid, F f) {
  const int ntiles = (len + kSelTile - 1) / kSelTile;
  const uint32_t n0 = ring.n;
  // the ring shares shared memory with the attention buffers written by generic stores
  fence_proxy_async_smem();
  comp_bar();
  if (gtid == 0) {
    for (int i = 0; i < kSelStages && i < ntiles; ++i) {
      const int st = (int)((n0 + i) % kSelStages);
      const int n = (len - i * kSelTile) < kSelTile ? (len - i * kSelTile) : kSelTile;
      mbar_arrive_expect_tx(&ring.bar[st], (uint32_t)n * 16u);
      bulk_copy_g2s(&sm.ring[st][0], src + (int64_t)i * kSelTile, (uint32_t)n * 16u, &ring.bar[st]);
    }
  }
  for (int i = 0; i < ntiles; ++i) {
    const uint32_t tn = n0 + i;
    const int st = (int)(tn % kSelStages);
    const int n = (len - i * kSelTile) < kSelTile ? (len - i * kSelTile) : kSelTile;
    const bool ok = comp_bar_and(mbar_wait_bounded(&ring.bar[st], (tn / kSelStages) & 1u, s.err, kMbarLimitNs));
    if (ok) f(i, &sm.ring[st][0], n);  // uniform: f may use group barriers
    comp_bar();
    if (gtid == 0 && i + kSelStages < ntiles) {
      const int j = i + kSelStages;
      const int nj = (len - j * kSelTile) < kSelTile ? (len - j * kSelTile) : kSelTile;
      mbar_arrive_expect_tx(&ring.bar[st], (uint32_t)nj * 16u);
      bulk_copy_g2s(&sm.ring[st][0], src + (int64_t)j * kSelTile, (uint32_t)nj * 16u, &ring.bar[st]);
    }
  }
  ring.n = n0 + ntiles;
}

template <int G>
__device__ __forceinline__ int score_of(const uint4 c, const uint64_t* qw) {
  const uint64_t k0 = (uint64_t)c.x | ((uint64_t)c.y << 32);
  const uint64_t k1 = (uint64_t)c.z | ((uint64_t)c.w << 32);
  int sc = 128 * G;
#pragma unroll
  for (int g = 0; g < G; ++g) sc -= __popcll(k0 ^ qw[2 * g]) + __popcll(k1 ^ qw[2 * g + 1]);
  return sc;
}

template <int G>
__device__ __forceinline__ void load_qcodes(const DevState& s, int64_t u, uint64_t* qw) {
  const int h = (int)(u % s.Hkv);
  const int b = (int)((u / s.Hkv) % s.B);
  const int l = (int)(u / ((int64_t)s.Hkv * s.B));
  const uint4* qc = s.qcodes + ((int64_t)l * s.B + b) * s.Hq + (int64_t)h * G;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const uint4 v = qc[g];
    qw[2 * g] = (uint64_t)v.x | ((uint64_t)v.y << 32);
    qw[2 * g + 1] = (uint64_t)v.z | ((uint64_t)v.w << 32);
  }
}

// ---- selection items ----------------------------------------------------------------
template <int G>
__device__ void sel_score(const DevState& s, SelSmem& sm, Ring& ring, int64_t u, int c, int gtid) {
  const int b = (int)((u / s.Hkv) % s.B);
  const int64_t N = s.ntok[b];
  const int64_t t0 = (int64_t)c * kSelChunk;
  const int len = (int)(N - t0 <= 0 ? 0 : (N - t0 < kSelChunk ? N - t0 : kSelChunk));
  for (int i = gtid; i < s.nbp; i += kCompThreads) sm.hist[i] = 0;
  uint64_t qw[2 * G];
  load_qcodes<G>(s, u, qw);
  comp_bar();
  stream_codes(s, sm, ring, s.codes + u * s.Nmax + t0, len, gtid, [&](int, const uint4* tile, int n) {
    for (int t = gtid; t < n; t += kCompThreads) atomicAdd(&sm.hist[score_of<G>(tile[t], qw)], 1u);
  });
  uint32_t* H = s.sel_hist + (u * s.nch + c) * s.nbp;
  for (int i = gtid; i < s.nbp; i += kCompThreads) H[i] = sm.hist[i];
  __threadfence();
  comp_bar();
  if (gtid == 0) red_release_add_u32(&s.score_done[u], 1u);
}

template <int G>
__device__ void sel_finalize(const DevState& s, SelSmem& sm, int64_t u, int gtid) {
  constexpr int NB = 128 * G + 1;
  const int b = (int)((u / s.Hkv) % s.B);
  const int64_t k = s.kcount[b];
  const int nch = s.nch;
  if (gtid == 0) wait_flag(&s.score_done[u], (uint32_t)nch, s);
  if (gtid < 4) sm.misc[gtid] = 0;
  comp_bar();
  const uint32_t* H = s.sel_hist + u * nch * s.nbp;
  for (int bin = gtid; bin < NB; bin += kCompThreads) {
    uint32_t t = 0;
    for (int c = 0; c < nch; ++c) t += __ldcg(H + c * s.nbp + bin);
    sm.hist[bin] = t;
  }
  comp_bar();
  if (gtid < 32) {  // threshold: largest T with count(score >= T) >= k
    const int lane = gtid;
    const int seg = (NB + 31) / 32;
    const int hi = NB - lane * seg;
    const int lo = hi - seg > 0 ? hi - seg : 0;
    int segsum = 0;
    for (int bin = lo; bin < hi; ++bin) segsum += (int)sm.hist[bin];
    int incl = segsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const int excl = incl - segsum;
    if (excl < k && incl >= k) {
      int run = excl;
      for (int bin = hi - 1; bin >= lo; --bin) {
        if (run + (int)sm.hist[bin] >= k) {
          sm.misc[0] = bin;
          sm.misc[1] = run;
          break;
        }
        run += (int)sm.hist[bin];
      }
    }
  }
  comp_bar();
  const int T = sm.misc[0], n_gt = sm.misc[1];
  for (int c = gtid; c < nch; c += kCompThreads) {
    int gt = 0;
    for (int bin = T + 1; bin < NB; ++bin) gt += (int)__ldcg(H + c * s.nbp + bin);
    sm.cgt[c] = gt;
    sm.ceq[c] = (int)__ldcg(H + c * s.nbp + T);
  }
  comp_bar();
  if (gtid == 0) {
    const int quota = (int)k - n_gt;
    int off = 0, eqb = 0;
    for (int c = 0; c < nch; ++c) {
      int take = quota - eqb;
      take = take < 0 ? 0 : (take > sm.ceq[c] ? sm.ceq[c] : take);
      s.sel_meta[u * nch + c] = make_int4(off, take, T, 0);
      off += sm.cgt[c] + take;
      eqb += sm.ceq[c];
    }
  }
  __threadfence();
  comp_bar();
  if (gtid == 0) red_release_add_u32(&s.fin_done[u], 1u);
}

template <int G>
__device__ void sel_compact(const DevState& s, SelSmem& sm, Ring& ring, int64_t u, int c, int gtid) {
  const int b = (int)((u / s.Hkv) % s.B);
  const int64_t N = s.ntok[b];
  const int64_t k = s.kcount[b];
  const int64_t t0 = (int64_t)c * kSelChunk;
  const int len = (int)(N - t0 <= 0 ? 0 : (N - t0 < kSelChunk ? N - t0 : kSelChunk));
  if (gtid == 0) wait_flag(&s.fin_done[u], 1u, s);
  uint64_t qw[2 * G];
  load_qcodes<G>(s, u, qw);
  comp_bar();
  const int4 meta = __ldcg(&s.sel_meta[u * s.nch + c]);
  const int off = meta.x, take = meta.y, T = meta.z;
  const int warp = gtid >> 5, lane = gtid & 31;
  const uint32_t lt = (1u << lane) - 1u;
  int32_t* out = s.idx + u * s.kmax;
  int run_eq = 0, run_sel = 0;  // chunk-local, uniform over the group
  stream_codes(s, sm, ring, s.codes + u * s.Nmax + t0, len, gtid, [&](int ti, const uint4* tile, int n) {
    int sc[4];
    int gt = 0, eq = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = 128 * warp + 32 * i + lane;
      sc[i] = t < n ? score_of<G>(tile[t], qw) : -1;
      gt += __popc(__ballot_sync(0xffffffffu, sc[i] > T));
      eq += __popc(__ballot_sync(0xffffffffu, sc[i] == T));
    }
    if (lane == 0) {
      sm.wc[warp][0] = gt;
      sm.wc[warp][1] = eq;
    }
    comp_bar();
    int eqb = run_eq, selb = run_sel, eq_all = 0, sel_all = 0;
    for (int w = 0; w < kCompWarps; ++w) {
      int tk = take - (run_eq + eq_all);
      tk = tk < 0 ? 0 : (tk > sm.wc[w][1] ? sm.wc[w][1] : tk);
      const int selw = sm.wc[w][0] + tk;
      if (w < warp) {
        eqb += sm.wc[w][1];
        selb += selw;
      }
      eq_all += sm.wc[w][1];
      sel_all += selw;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const bool is_eq = sc[i] == T;
      const uint32_t beq = __ballot_sync(0xffffffffu, is_eq);
      const int rank = eqb + __popc(beq & lt);
      const bool sel = sc[i] > T || (is_eq && rank < take);
      const uint32_t bsel = __ballot_sync(0xffffffffu, sel);
      if (sel) {
        const int pos = off + selb + __popc(bsel & lt);
        if (pos < k)
          out[pos] = (int32_t)(t0 + (int64_t)ti * kSelTile + 128 * warp + 32 * i + lane);
        else
          atomicOr(s.err, kErrBounds);
      }
      eqb += __popc(beq);
      selb += __popc(bsel);
    }
    run_eq += eq_all;
    run_sel += sel_all;
  });
  __threadfence();
  comp_bar();
  if (gtid == 0) red_release_add_u32(&s.sel_cnt[u], 1u);
}

// ---- attention split -----------------------------------------------------------------
template <int D>
__device__ void attend_split(const DevState& s, AttSmem<D>& sm, const uint16_t* __restrict__ q,
                             float* __restrict__ out, int64_t u, int split, int gtid) {
  constexpr int VPR = D / 4;
  constexpr int NG = AttSmem<D>::NG;
  const int h = (int)(u % s.Hkv);
  const int b = (int)((u / s.Hkv) % s.B);
  const int l = (int)(u / ((int64_t)s.Hkv * s.B));
  const int G = s.G;
  const int warp = gtid >> 5, lane = gtid & 31;
  const int64_t N = s.ntok[b];
  const int64_t k = s.kcount[b];
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
  const float qscale = 1.4426950408889634f * rsqrtf((float)D);  // scores in log2 units
  const uint16_t* qg = q + (((int64_t)l * s.B + b) * s.Hq + (int64_t)h * G) * D;
  for (int e = gtid; e < G * D; e += kCompThreads) sm.qs[e / D][e % D] = bf16_bits_to_f32(qg[e]) * qscale;
  if (gtid < kMaxG) {
    sm.m_run[gtid] = -INFINITY;
    sm.l_run[gtid] = 0.f;
  }
  float acc[kMaxG];
#pragma unroll
  for (int g = 0; g < kMaxG; ++g) acc[g] = 0.f;
  const int dj = gtid % D;
  const int rg = gtid / D;
  comp_bar();

  for (int64_t rb = r0; rb < r1; rb += kAttTile) {
    const int nrows = (int)((r1 - rb) < kAttTile ? (r1 - rb) : kAttTile);
    for (int e = gtid; e < nrows * VPR; e += kCompThreads) {
      const int r = e / VPR, c = e % VPR;
      int64_t srow = rb + r;
      if (persistent) {
        srow = __ldcg(ix + rb + r);
        if (srow < 0 || srow >= N) {
          atomicOr(s.err, kErrBounds);
          srow = 0;
        }
      }
      cp_async16(&sm.rows[r][c * 8], src + srow * VPR + c);
    }
    cp_async_commit();
    cp_async_wait<0>();
    comp_bar();
    for (int p = gtid; p < G * kAttTile; p += kCompThreads) {
      const int g = p / kAttTile, r = p % kAttTile;
      float dot = -INFINITY;
      if (r < nrows) {
        dot = 0.f;
        const uint4* kr = reinterpret_cast<const uint4*>(&sm.rows[r][0]);
#pragma unroll 4
        for (int i = 0; i < D / 8; ++i) {
          const uint4 w = kr[i];
          const float4 qa = *reinterpret_cast<const float4*>(&sm.qs[g][8 * i]);
          const float4 qb = *reinterpret_cast<const float4*>(&sm.qs[g][8 * i + 4]);
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
      sm.sc[g][r] = dot;
    }
    comp_bar();
    for (int g = warp; g < G; g += kCompWarps) {
      const float v = sm.sc[g][lane];
      const float mx = warp_max(v);
      const float mo = sm.m_run[g];
      const float mn = fmaxf(mo, mx);
      const float pv = exp2f(v - mn);
      const float ps = warp_sum(pv);
      sm.sc[g][lane] = pv;
      if (lane == 0) {
        const float a = exp2f(mo - mn);
        sm.alpha[g] = a;
        sm.l_run[g] = sm.l_run[g] * a + ps;
        sm.m_run[g] = mn;
      }
    }
    comp_bar();
#pragma unroll
    for (int g = 0; g < kMaxG; ++g)
      if (g < G) acc[g] *= sm.alpha[g];
    for (int r = rg; r < nrows; r += NG) {
      const float v = bf16_bits_to_f32(sm.rows[r][D + dj]);
#pragma unroll
      for (int g = 0; g < kMaxG; ++g)
        if (g < G) acc[g] = fmaf(sm.sc[g][r], v, acc[g]);
    }
    comp_bar();
  }

  if (NG > 1) {
#pragma unroll
    for (int g = 0; g < kMaxG; ++g)
      if (g < G) sm.red[rg][g][dj] = acc[g];
    comp_bar();
  }
  float* part = s.part + ((u * s.nsplit + split) * G) * (D + 2);
  if (gtid < D) {
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) {
      if (g < G) {
        float a = acc[g];
        if (NG > 1) {
          a = 0.f;
          for (int r = 0; r < NG; ++r) a += sm.red[r][g][gtid];
        }
        part[g * (D + 2) + 2 + gtid] = a;
      }
    }
  }
  if (gtid < G) {
    part[gtid * (D + 2) + 0] = sm.m_run[gtid];
    part[gtid * (D + 2) + 1] = sm.l_run[gtid];
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
  const float* pu = s.part + (u * s.nsplit) * G * (D + 2);
  float* og = out + (((int64_t)l * s.B + b) * s.Hq + (int64_t)h * G) * D;
  for (int e = gtid; e < G * D; e += kCompThreads) {
    const int g = e / D, j = e % D;
    float M = -INFINITY;
    for (int sp = 0; sp < s.nsplit; ++sp) M = fmaxf(M, __ldcg(pu + (sp * G + g) * (D + 2)));
    float Lsum = 0.f, O = 0.f;
    for (int sp = 0; sp < s.nsplit; ++sp) {
      const float* ps = pu + (sp * G + g) * (D + 2);
      const float ls = __ldcg(ps + 1);
      if (ls > 0.f) {
        const float w = exp2f(__ldcg(ps) - M);
        Lsum = fmaf(ls, w, Lsum);
        O = fmaf(__ldcg(ps + 2 + j), w, O);
      }
    }
    og[g * D + j] = O / Lsum;
  }
  if (gtid == 0) s.unit_done[u] = 0u;
}

// ---- fetch warps -----------------------------------------------------------------------
template <int D>
__device__ void fetch_role(const DevState& s, const int* pre_m, int n_miss, int lane) {
  constexpr int VPR = D / 4;  // 16-byte vectors per K|V record
  const int NS = s.nsplit, RS = s.split_rows, L = s.L, BH = s.B * s.Hkv;
  const int64_t n_items = (int64_t)n_miss * NS;
  while (true) {
    unsigned item = 0;
    if (lane == 0) item = atomicAdd(&s.queue[0], 1u);
    item = __shfl_sync(0xffffffffu, item, 0);
    if ((int64_t)item >= n_items) break;
    const int p = (int)(item / NS), c = (int)(item % NS);
    const int l = layer_of(pre_m, L, p);
    const int64_t u = s.miss_list[(int64_t)l * BH + (p - pre_m[l])];
    const int b = (int)((u / s.Hkv) % s.B);
    const int64_t k = s.kcount[b];
    const int64_t N = s.ntok[b];
    const int64_t r0 = (int64_t)c * RS;
    const int64_t r1 = (r0 + RS < k) ? r0 + RS : k;
    if (r0 < r1) {
      // missed units were selected by the launch before this one
      if (lane == 0 && s.timeline) atomicCAS(&s.timeline[TL_FETCH_FIRST], 0ull, global_timer_ns());
      const uint4* pool = reinterpret_cast<const uint4*>(s.pool) + u * s.Nmax * VPR;
      uint4* slot = reinterpret_cast<uint4*>(s.slots) + u * s.kmax * VPR;
      const int32_t* ix = s.idx + u * s.kmax;
      const int64_t total = (r1 - r0) * VPR;
      for (int64_t e0 = lane; e0 < total; e0 += 32 * kFetchUnroll) {
        uint4 v[kFetchUnroll];
#pragma unroll
        for (int j = 0; j < kFetchUnroll; ++j) {
          const int64_t e = e0 + 32 * j;
          if (e < total) {
            const int64_t t = __ldcg(ix + r0 + e / VPR);
            if (t >= 0 && t < N) {
              v[j] = ld_nc_v4(pool + t * VPR + (e % VPR));
            } else {
              atomicOr(s.err, kErrBounds);
              v[j] = make_uint4(0, 0, 0, 0);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < kFetchUnroll; ++j) {
          const int64_t e = e0 + 32 * j;
          if (e < total) slot[r0 * VPR + e] = v[j];
        }
      }
    }
    __threadfence();
    __syncwarp();
    if (lane == 0 && l != s.drop_flag_layer) red_release_add_u32(&s.ready[u * NS + c], 1u);
    if (lane == 0 && s.timeline) atomicMax(&s.timeline[TL_FETCH_END], global_timer_ns());
  }
}

// ---- the kernel ------------------------------------------------------------------------
template <int D, int G>
__global__ void __launch_bounds__(kFThreads, 6) k_step_fused(DevState s, const uint16_t* __restrict__ q,
                                                             float* __restrict__ out) {
  __shared__ int pre[3][kMaxLayers + 1];  // hit, persistent, missed lists
  __shared__ long long sec_start[6];
  __shared__ uint64_t ring_bar[kSelStages];
  __shared__ int s_item;
  __shared__ __align__(128) CompSmem<D> sm;
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
    // compute queue: selections of the persistent units (per layer: the layer's chunk
    // scores, finalizes, chunk compactions), then attention splits of reused,
    // persistent and missed units
    const long long nh = a[0], np = a[1], nm = a[2], SB = 2LL * s.nch + 1, NS = s.nsplit;
    const long long size[5] = {0, np * SB, nh * NS, np * NS, nm * NS};
    sec_start[0] = 0;
    for (int i = 0; i < 5; ++i) sec_start[i + 1] = sec_start[i] + size[i];
    for (int i = 0; i < kSelStages; ++i) mbar_init(&ring_bar[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (warp < kFetchWarps) {
    fetch_role<D>(s, pre[2], pre[2][L], lane);
    return;  // no block-wide barrier after this point
  }
  const int gtid = tid - 32 * kFetchWarps;
  const int BH = s.B * s.Hkv;
  const int NC = s.nch;
  Ring ring{ring_bar, 0u};
  const long long total = sec_start[5];
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
    if (sec <= 1) {  // selection block of one layer
      const long long SB = 2LL * NC + 1;
      const int l = layer_of(pl, L, (int)(j / SB));
      const int n = pl[l + 1] - pl[l];
      const long long r = j - (long long)pl[l] * SB;
      const int32_t* ll = lst + (int64_t)l * BH;
      if (r < (long long)n * NC) {
        sel_score<G>(s, sm.sel, ring, ll[r / NC], (int)(r % NC), gtid);
      } else if (r < (long long)n * NC + n) {
        sel_finalize<G>(s, sm.sel, ll[r - (long long)n * NC], gtid);
      } else {
        const long long r2 = r - (long long)n * NC - n;
        sel_compact<G>(s, sm.sel, ring, ll[r2 / NC], (int)(r2 % NC), gtid);
      }
      if (s.timeline && gtid == 0) atomicMax(&s.timeline[sec == 0 ? TL_SEL_MISS_END : TL_SEL_PERS_END], global_timer_ns());
    } else {  // attention split
      const int p = (int)(j / s.nsplit), c = (int)(j % s.nsplit);
      const int l = layer_of(pl, L, p);
      const int64_t u = lst[(int64_t)l * BH + (p - pl[l])];
      const int b = (int)((u / s.Hkv) % s.B);
      const int64_t r0 = (int64_t)c * s.split_rows;
      if (s.timeline && gtid == 0) atomicCAS(&s.timeline[TL_ATT_FIRST], 0ull, global_timer_ns());
      if (sec == 3) {
        if (gtid == 0) wait_flag(&s.sel_cnt[u], (uint32_t)NC, s);
        comp_bar();
      } else if (sec == 4 && r0 < s.kcount[b]) {
        if (gtid == 0) {
          const uint64_t t0 = s.timeline ? global_timer_ns() : 0;
          wait_flag(&s.ready[u * s.nsplit + c], 1u, s);
          if (s.timeline) atomicAdd(&s.timeline[TL_ATT_WAIT_NS], global_timer_ns() - t0);
        }
        comp_bar();
      }
      attend_split<D>(s, sm.att, q, out, u, c, gtid);
      if (s.timeline && gtid == 0) atomicMax(&s.timeline[TL_COMP_END], global_timer_ns());
    }
    comp_bar();
  }
}

template <int D, int G>
int fused_grid() {
  static int grid = 0;
  if (grid == 0) {
    int dev = 0, sms = 0, per_sm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_step_fused<D, G>, kFThreads, 0);
    grid = sms * (per_sm > 0 ? per_sm : 1);
  }
  return grid;
}

template <int D, int G>
cudaError_t launch_dg(const DevState& s, const uint16_t* q, float* out, cudaStream_t st) {
  k_step_fused<D, G><<<fused_grid<D, G>(), kFThreads, 0, st>>>(s, q, out);
  return cudaGetLastError();
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
    const int64_t n = (tend - t0) * vpr;
    const uint4* src = reinterpret_cast<const uint4*>(s.pool) + (u * s.Nmax + t0) * vpr;
    uint4* dst = reinterpret_cast<uint4*>(s.resident) + ((((int64_t)l * s.B + b) * s.P + p) * s.Nmax + t0) * vpr;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x)
      dst[e] = ld_nc_v4(src + e);
  }
}

}  // namespace

cudaError_t launch_step_fused(const DevState& s, const uint16_t* q, float* out, cudaStream_t st) {
  if (s.L > kMaxLayers || s.nch > kMaxChunks || s.nbp > kNBPad) return cudaErrorInvalidValue;
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
