// Hash-code scoring and top-k selection of the units that missed, one unit per
// thread-block cluster (runs before the fused step kernel, so the zero-copy fetch of
// their rows can start at once; persistent units are selected inside the fused
// kernel, under the fetch).
//
// score[t] = sum_g (128 - popcount(qcode_g ^ kcode_t)) over the G query heads of
// the GQA group; the k = ceil(10 % of N) best tokens are kept, ties going to the
// lower token index, and written in ascending index order (top-k = 10 %: "CLO
// (2511.14510) - L3 Per-Paper Synthesis", section 2.2; HATA scorer: section 3.2).
//
// Scores are small integers (0 .. 128*G), so the selection is one histogram digit:
//   1. each CTA of the cluster owns a contiguous chunk of the unit's tokens, streams
//      its 16-byte codes into shared memory with 1-D bulk copies (TMA engine, a ring
//      of stages on mbarriers), keeps the scores in shared memory and builds a
//      shared-memory histogram;
//   2. after a cluster barrier every CTA sums the cluster's histograms through
//      distributed shared memory and finds the threshold score T with
//      count(score > T) < k <= count(score >= T);
//   3. ordered compaction: tokens with score > T, plus the first (k - count(>T))
//      tokens with score == T in index order across the cluster's chunks.
#include <cooperative_groups.h>

#include "clo_internal.cuh"

namespace cg = cooperative_groups;

namespace clo {

namespace {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelTile = 512;  // tokens per bulk copy (8 KB)
constexpr int kSelStages = 4;
constexpr uint64_t kMbarLimitNs = 2000000000ull;

__host__ __device__ inline int hist_bins_padded(int G) { return ((128 * G + 1) + 31) / 32 * 32; }

struct SelSmem {
  uint4* ring;
  uint16_t* scores;
  uint32_t* hist;
  uint32_t* tot;
  uint64_t* bar;
  int* misc;  // [0] T, [1] n_gt, [2..2+8) gt per rank, [10..18) eq per rank
  int* wcnt;  // [kSelWarps][2] gt, eq per warp; then [kSelWarps][2] offsets
};

__device__ inline SelSmem carve(unsigned char* base, int G, int64_t chunk) {
  SelSmem m;
  size_t off = 0;
  m.ring = reinterpret_cast<uint4*>(base + off);
  off += (size_t)kSelStages * kSelTile * 16;
  m.bar = reinterpret_cast<uint64_t*>(base + off);
  off += kSelStages * 8;
  const int nb = hist_bins_padded(G);
  m.hist = reinterpret_cast<uint32_t*>(base + off);
  off += (size_t)nb * 4;
  m.tot = reinterpret_cast<uint32_t*>(base + off);
  off += (size_t)nb * 4;
  m.misc = reinterpret_cast<int*>(base + off);
  off += 32 * 4;
  m.wcnt = reinterpret_cast<int*>(base + off);
  off += 4 * kSelWarps * 4;
  m.scores = reinterpret_cast<uint16_t*>(base + off);
  return m;
}

template <int G>
__global__ void __launch_bounds__(kSelThreads) k_select(DevState s, int64_t chunk) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int64_t u = blockIdx.y;
  const int dec = s.decision[u];
  if (dec != CLO_DEC_MISS) return;  // uniform over the cluster

  const int h = (int)(u % s.Hkv);
  const int b = (int)((u / s.Hkv) % s.B);
  const int l = (int)(u / ((int64_t)s.Hkv * s.B));
  const int64_t N = s.ntok[b];
  const int64_t k = s.kcount[b];
  const int64_t c0 = (int64_t)rank * chunk;
  const int64_t c1 = (c0 + chunk < N) ? c0 + chunk : N;
  const int len = (int)(c1 > c0 ? c1 - c0 : 0);
  const int NB = 128 * G + 1;

  SelSmem m = carve(smem_raw, G, chunk);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < hist_bins_padded(G); i += kSelThreads) m.hist[i] = 0;
  if (tid == 0) {
    for (int i = 0; i < kSelStages; ++i) mbar_init(&m.bar[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  uint64_t qw[2 * G];
  {
    const uint4* qc = s.qcodes + ((int64_t)l * s.B + b) * s.Hq + (int64_t)h * G;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const uint4 v = qc[g];
      qw[2 * g] = (uint64_t)v.x | ((uint64_t)v.y << 32);
      qw[2 * g + 1] = (uint64_t)v.z | ((uint64_t)v.w << 32);
    }
  }
  __syncthreads();

  const int ntiles = (len + kSelTile - 1) / kSelTile;
  const uint4* src = s.codes + u * s.Nmax + c0;
  if (tid == 0) {
    for (int i = 0; i < kSelStages && i < ntiles; ++i) {
      const int n = (len - i * kSelTile) < kSelTile ? (len - i * kSelTile) : kSelTile;
      mbar_arrive_expect_tx(&m.bar[i], (uint32_t)n * 16u);
      bulk_copy_g2s(m.ring + (size_t)i * kSelTile, src + (int64_t)i * kSelTile, (uint32_t)n * 16u, &m.bar[i]);
    }
  }
  for (int i = 0; i < ntiles; ++i) {
    const int st = i % kSelStages;
    const uint32_t par = (uint32_t)((i / kSelStages) & 1);
    const int n = (len - i * kSelTile) < kSelTile ? (len - i * kSelTile) : kSelTile;
    const bool ok = mbar_wait_bounded(&m.bar[st], par, s.err, kMbarLimitNs);
    if (ok && tid < n) {
      const uint4 c = m.ring[(size_t)st * kSelTile + tid];
      const uint64_t k0 = (uint64_t)c.x | ((uint64_t)c.y << 32);
      const uint64_t k1 = (uint64_t)c.z | ((uint64_t)c.w << 32);
      int sc = 128 * G;
#pragma unroll
      for (int g = 0; g < G; ++g) sc -= __popcll(k0 ^ qw[2 * g]) + __popcll(k1 ^ qw[2 * g + 1]);
      m.scores[i * kSelTile + tid] = (uint16_t)sc;
      atomicAdd(&m.hist[sc], 1u);
    }
    __syncthreads();
    if (tid == 0 && i + kSelStages < ntiles) {
      const int j = i + kSelStages;
      const int nj = (len - j * kSelTile) < kSelTile ? (len - j * kSelTile) : kSelTile;
      mbar_arrive_expect_tx(&m.bar[st], (uint32_t)nj * 16u);
      bulk_copy_g2s(m.ring + (size_t)st * kSelTile, src + (int64_t)j * kSelTile, (uint32_t)nj * 16u, &m.bar[st]);
    }
  }
  cluster.sync();  // every CTA's histogram is complete and visible

  for (int bin = tid; bin < NB; bin += kSelThreads) {
    uint32_t t = 0;
    for (int c = 0; c < C; ++c) t += cluster.map_shared_rank(m.hist, c)[bin];
    m.tot[bin] = t;
  }
  __syncthreads();

  // threshold T: largest score with count(score >= T) >= k
  if (warp == 0) {
    const int seg = (NB + 31) / 32;
    const int hi = NB - lane * seg;
    const int lo = hi - seg > 0 ? hi - seg : 0;
    int segsum = 0;
    for (int bin = lo; bin < hi; ++bin) segsum += (int)m.tot[bin];
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
        if (run + (int)m.tot[bin] >= k) {
          m.misc[0] = bin;
          m.misc[1] = run;
          break;
        }
        run += (int)m.tot[bin];
      }
    }
  }
  __syncthreads();
  const int T = m.misc[0];
  const int n_gt = m.misc[1];
  if (warp < C) {
    const uint32_t* hr = cluster.map_shared_rank(m.hist, warp);
    int gt = 0;
    for (int bin = T + 1 + lane; bin < NB; bin += 32) gt += (int)hr[bin];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) gt += __shfl_xor_sync(0xffffffffu, gt, o);
    if (lane == 0) {
      m.misc[2 + warp] = gt;
      m.misc[10 + warp] = (int)hr[T];
    }
  }
  __syncthreads();
  const int quota = (int)k - n_gt;  // ties to take, cluster-wide, lowest index first
  int out_base = 0, eq_before = 0;
  for (int c = 0; c < rank; ++c) {
    const int eqc = m.misc[10 + c];
    int take = quota - eq_before;
    take = take < 0 ? 0 : (take > eqc ? eqc : take);
    out_base += m.misc[2 + c] + take;
    eq_before += eqc;
  }
  int take_eq = quota - eq_before;
  take_eq = take_eq < 0 ? 0 : (take_eq > m.misc[10 + rank] ? m.misc[10 + rank] : take_eq);

  // ordered compaction of this CTA's chunk: warps own contiguous segments
  const int wseg = ((len + kSelWarps - 1) / kSelWarps + 31) / 32 * 32;
  const int w0 = warp * wseg;
  const int w1 = (w0 + wseg < len) ? w0 + wseg : len;
  {
    int gt = 0, eq = 0;
    for (int t = w0 + lane; t < w1; t += 32) {
      const int sc = m.scores[t];
      gt += sc > T;
      eq += sc == T;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      gt += __shfl_xor_sync(0xffffffffu, gt, o);
      eq += __shfl_xor_sync(0xffffffffu, eq, o);
    }
    if (lane == 0) {
      m.wcnt[2 * warp] = gt;
      m.wcnt[2 * warp + 1] = eq;
    }
  }
  __syncthreads();
  if (tid == 0) {
    int off = out_base, eqb = 0;
    for (int w = 0; w < kSelWarps; ++w) {
      const int gt = m.wcnt[2 * w], eq = m.wcnt[2 * w + 1];
      m.wcnt[2 * kSelWarps + 2 * w] = off;
      m.wcnt[2 * kSelWarps + 2 * w + 1] = eqb;
      int take = take_eq - eqb;
      take = take < 0 ? 0 : (take > eq ? eq : take);
      off += gt + take;
      eqb += eq;
    }
  }
  __syncthreads();
  {
    const int off = m.wcnt[2 * kSelWarps + 2 * warp];
    const int eqb = m.wcnt[2 * kSelWarps + 2 * warp + 1];
    const uint32_t lt = (1u << lane) - 1u;
    int run_sel = 0, run_eq = 0;
    int32_t* out = s.idx + u * s.kmax;
    for (int base = w0; base < w1; base += 32) {
      const int t = base + lane;
      const int sc = t < w1 ? (int)m.scores[t] : -1;
      const bool is_eq = sc == T;
      const uint32_t beq = __ballot_sync(0xffffffffu, is_eq);
      const int eq_rank = eqb + run_eq + __popc(beq & lt);
      const bool sel = (sc > T) || (is_eq && eq_rank < take_eq);
      const uint32_t bsel = __ballot_sync(0xffffffffu, sel);
      if (sel) {
        const int pos = off + run_sel + __popc(bsel & lt);
        if (pos < k)
          out[pos] = (int32_t)(c0 + t);
        else
          atomicOr(s.err, kErrBounds);
      }
      run_eq += __popc(beq);
      run_sel += __popc(bsel);
    }
  }
  cluster.sync();  // peers may still be reading this CTA's histogram
}

template <int G>
cudaError_t launch_select_g(const DevState& s, int cluster, int64_t chunk, cudaStream_t st) {
  const size_t smem = select_smem_bytes(G, chunk);
  cudaError_t e = cudaFuncSetAttribute(k_select<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t U = (int64_t)s.L * s.B * s.Hkv;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cluster, (unsigned)U, 1);
  cfg.blockDim = dim3(kSelThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_select<G>, s, chunk);
}

}  // namespace

size_t select_smem_bytes(int G, int64_t chunk) {
  size_t off = (size_t)kSelStages * kSelTile * 16 + kSelStages * 8 + 2 * (size_t)hist_bins_padded(G) * 4 + 32 * 4 +
               4 * kSelWarps * 4;
  return off + (size_t)((chunk * 2 + 15) / 16 * 16);
}

cudaError_t launch_select(const DevState& s, int cluster, int64_t chunk, cudaStream_t st) {
  switch (s.G) {
    case 1: return launch_select_g<1>(s, cluster, chunk, st);
    case 2: return launch_select_g<2>(s, cluster, chunk, st);
    case 3: return launch_select_g<3>(s, cluster, chunk, st);
    case 4: return launch_select_g<4>(s, cluster, chunk, st);
    case 5: return launch_select_g<5>(s, cluster, chunk, st);
    case 6: return launch_select_g<6>(s, cluster, chunk, st);
    case 7: return launch_select_g<7>(s, cluster, chunk, st);
    case 8: return launch_select_g<8>(s, cluster, chunk, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace clo
