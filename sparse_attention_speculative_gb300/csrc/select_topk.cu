// select_topk.cu -- aggregated-logit top-k with a protected budget on sm_103a.
//
// What it computes: the Vegas selection (technical summary sec. 2.A: the prefix set
// T with |T| = k maximising the logits summed over the collected rows and all query
// heads -- a separable objective, so the k highest scores) under the Dustin budget
// rule (Methodology sec. 1: attention sinks and the recent window are kept first,
// the rest of the budget is filled by score).  Equal scores go to the lower position;
// the output is in ascending position order.
//
// How (GB300 design).  The step is short and latency-bound, so the design minimises
// dependent rounds between the SMs: one thread-block cluster per row (layer x
// sequence), each CTA owning a contiguous slice of the prefix, and four cluster
// barriers in the common case (two from a scored input; one more on rows longer than
// 32768 positions).  Scores become
// order-preserving uint32 keys.
//   A. Every CTA sums the per-KV-group partial scores of its slice (fp32, groups in
//      order), keeps the keys in shared memory and builds a 4096-bin histogram of
//      the top 12 key bits of its candidates (positions outside the protected sink
//      and recent windows).
//   B. Every CTA adds its non-zero bins into rank 0's histogram (distributed shared
//      memory atomics).  Cluster barrier.
//   C. Rank 0 finds the boundary bin, the one that holds the r-th largest candidate
//      key (r = k - |protected|), and writes it into every CTA.  Cluster barrier.  If
//      that bin holds more keys than rank 0 can take, the next 10 bits are
//      histogrammed the same way (rare; at most two more levels).
//   D. Every CTA builds its words of a position bitmap (its candidates above the
//      boundary bin), sends its count of them to every CTA (rows of up to 32768
//      positions: also the words themselves to rank 0), and appends its boundary-bin
//      keys (with positions) to rank 0's buffer.  Cluster barrier.
//   E. Rank 0 resolves the remaining key bits and the tie cut (equal keys go to the
//      lower position) on the gathered keys with block-local passes.  Short rows: it
//      marks the winners and writes the whole row (sinks, candidates in order by a
//      block scan over the bitmap, recent window, -1 padding).  Longer rows: it counts
//      the winners per owning CTA and hands every CTA the cut and where its candidates
//      start (cluster barrier), and
//   F. every CTA marks its boundary keys that made the cut and writes its candidates
//      in position order from its own bitmap words; rank 0 adds the sinks, the recent
//      window and the padding.
// Scored input (the fused verification has already summed the groups and counted the
// level-0 histogram of every prefix position): A reads one score per position, and
// every CTA copies the row's histogram, takes the sinks and the recent window out of
// it and finds the boundary bin itself, so B and C (two cluster barriers) are skipped.
// Results are deterministic; no global workspace.  The kernel is launched as a
// programmatic dependent: its launch overlaps the tail of the verification kernels.
#include <cooperative_groups.h>

#include <climits>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace vsd {
namespace {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kMaxSelCluster = 16;
constexpr int kChunkQuantum = 4 * kSelThreads;  // keys per CTA come in multiples of this
constexpr int kMaxChunk = 16384;
constexpr int kBins0 = 4096;                     // level 0: top 12 bits
constexpr int kBinsL = 1024;                     // levels 1, 2: 10 bits each
constexpr int kGatherCap = 8192;                 // boundary-bin keys rank 0 can hold
// Rows of up to this many bitmap words (32768 positions) are written by rank 0 alone,
// two rounds of its threads; longer rows by every CTA in parallel, which costs one more
// cluster barrier.
constexpr int kShortRowWords = 2 * kSelThreads;

enum Mode : int { kModeWhole = 0, kModeGather = 1, kModeTie = 2 };

struct SelParams {
  const float* partial;
  const int32_t* prefix_len;
  int32_t* idx;
  int32_t* n_sel;
  float* scores_out;
  unsigned* status;
  int Hkv, P_max, k, n_sink, n_recent, chunk;
  // hybrid budget (Dustin Methodology sec. 1), both passes optional:
  int m_limit;                  // >= 0: take at most this many candidates by score
  const uint32_t* pre_bitmap;   // [n_rows][bm_words]: candidates chosen beforehand
  const int32_t* pre_count;     // [n_rows]: how many
  uint32_t* out_bitmap;         // [n_rows][bm_words]: this pass's chosen candidates
  int32_t* out_count;           // [n_rows]
  int bm_words;                 // words per row of those bitmaps: ceil(P_max / 32)
  const uint32_t* hist;         // scored input: level-0 histogram of all prefix positions
};

struct SelShared {
  uint32_t scan[kSelWarps];
  uint32_t tmp[kMaxSelCluster];
  int f_bin, f_rem, f_cnt;  // result of a bin search
  uint32_t gcount;          // rank 0: gathered boundary keys
  uint32_t cnt[kMaxSelCluster];    // candidates each CTA chose before the boundary cut
  uint32_t taken[kMaxSelCluster];  // rank 0: boundary keys taken, per owning CTA
  int out_base;                    // long rows: where this CTA's candidates start
  uint32_t thr_prefix, thr_mask;   // long rows: the boundary cut (from rank 0)
  int thr_cut;
};

// Dynamic shared memory of one CTA (the rank-0-only parts are laid out everywhere).
struct SelLayout {
  uint2* gbuf;       // [kGatherCap] rank 0: boundary-bin (key, position)
  uint32_t* keys;    // [chunk]
  uint32_t* hist;    // [kBins0] this CTA's histogram (rank 0's scratch in E)
  uint32_t* loc;     // [kBins0] this CTA's words of the selection bitmap
  uint32_t* ghist;   // [kBins0 + 2 * kBinsL] rank 0: cluster histograms of the levels
  uint32_t* bitmap;  // [kShortRowWords] rank 0, short rows: the row's candidate bitmap
};

__device__ __forceinline__ SelLayout sel_layout(uint8_t* base, int chunk) {
  SelLayout L;
  L.gbuf = reinterpret_cast<uint2*>(base);
  L.keys = reinterpret_cast<uint32_t*>(base + static_cast<size_t>(kGatherCap) * 8);
  L.hist = L.keys + chunk;
  L.loc = L.hist + kBins0;
  L.ghist = L.loc + kBins0;
  L.bitmap = L.ghist + kBins0 + 2 * kBinsL;
  return L;
}

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Exclusive prefix sum over the threads of the block in thread order; *total gets
// the block sum.  Two __syncthreads; `scratch` is reusable afterwards.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* scratch,
                                                    uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  uint32_t base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) {
    const uint32_t s = scratch[w];
    base += (w < warp) ? s : 0u;
    tot += s;
  }
  *total = tot;
  __syncthreads();
  return base + x - v;
}

// Among bins cnt[0..n) (ascending key order) find the bin b holding the r-th largest
// element (1 <= r <= sum): S(b+1) < r <= S(b) with S(b) = sum of cnt[b..n).
// Result in sh.f_bin, sh.f_rem (= r - S(b+1)) and sh.f_cnt (= cnt[b]).
__device__ void find_bin(const uint32_t* cnt, int n, int r, SelShared& sh) {
  const int E = (n + kSelThreads - 1) / kSelThreads;
  const int hi = n - 1 - static_cast<int>(threadIdx.x) * E;  // this thread: bins hi .. hi-E+1
  uint32_t s = 0;
  for (int e = 0; e < E; ++e)
    if (hi - e >= 0) s += cnt[hi - e];
  uint32_t tot;
  const uint32_t before = block_excl_scan(s, sh.scan, &tot);
  const uint32_t ur = static_cast<uint32_t>(r);
  if (before < ur && ur <= before + s) {
    uint32_t acc = before;
    for (int e = 0; e < E; ++e) {
      const int b = hi - e;
      const uint32_t c = cnt[b];
      if (acc + c >= ur) {
        sh.f_bin = b;
        sh.f_rem = static_cast<int>(ur - acc);
        sh.f_cnt = static_cast<int>(c);
        break;
      }
      acc += c;
    }
  }
  __syncthreads();
}

// The same search from the low end: the bin holding the r-th smallest element.
__device__ void find_bin_low(const uint32_t* cnt, int n, int r, SelShared& sh) {
  const int E = (n + kSelThreads - 1) / kSelThreads;
  const int lo = static_cast<int>(threadIdx.x) * E;
  uint32_t s = 0;
  for (int e = 0; e < E; ++e)
    if (lo + e < n) s += cnt[lo + e];
  uint32_t tot;
  const uint32_t before = block_excl_scan(s, sh.scan, &tot);
  const uint32_t ur = static_cast<uint32_t>(r);
  if (before < ur && ur <= before + s) {
    uint32_t acc = before;
    for (int e = 0; e < E; ++e) {
      const int b = lo + e;
      const uint32_t c = cnt[b];
      if (acc + c >= ur) {
        sh.f_bin = b;
        sh.f_rem = static_cast<int>(ur - acc);
        sh.f_cnt = static_cast<int>(c);
        break;
      }
      acc += c;
    }
  }
  __syncthreads();
}

// Set this thread's selected positions (bit q of `sel` = position my0 + q) in the
// bitmap `bm`, one atomic per word.
__device__ __forceinline__ void mark_bits(uint32_t* bm, int my0, uint64_t sel) {
  while (sel) {
    const int q = __ffsll(static_cast<long long>(sel)) - 1;
    const int pos = my0 + q;
    const int span = 32 - (pos & 31);  // positions of this word from pos on
    const uint64_t m = (span >= 64 - q) ? (~0ull << q) : (((1ull << span) - 1) << q);
    const uint64_t part = sel & m;
    atomicOr(bm + (pos >> 5), static_cast<uint32_t>((part >> q) << (pos & 31)));
    sel &= ~m;
  }
}

// Resolve the boundary bin on the n_in gathered (key, position) pairs: the remaining
// key bits level by level, then -- when every bit is fixed and fewer equal keys are
// taken than there are -- the position cut (equal keys go to the lower position;
// positions are below 2^20: two 10-bit passes).  Winners: (key & mask) > prefix, or
// == prefix at a position <= cut.  `h` is 1024 words of scratch.
__device__ void resolve_boundary(const uint2* gbuf, int n_in, uint32_t* h, SelShared& sh,
                                 uint32_t& prefix, uint32_t& mask, int r_rem, int& cut) {
  const int t = threadIdx.x;
  const int start_level = (mask == 0xFFF00000u) ? 1 : ((mask == 0xFFFFFC00u) ? 2 : 3);
  for (int level = start_level; level < 3; ++level) {
    const int shift = level == 1 ? 10 : 0;
    for (int i = t; i < kBinsL; i += kSelThreads) h[i] = 0u;
    __syncthreads();
    for (int i = t; i < n_in; i += kSelThreads) {
      const uint32_t key = gbuf[i].x;
      if ((key & mask) == prefix) atomicAdd(&h[(key >> shift) & (kBinsL - 1)], 1u);
    }
    __syncthreads();
    find_bin(h, kBinsL, r_rem, sh);
    const bool whole = sh.f_rem == sh.f_cnt;
    prefix |= static_cast<uint32_t>(sh.f_bin) << shift;
    mask |= static_cast<uint32_t>(kBinsL - 1) << shift;
    r_rem = sh.f_rem;
    __syncthreads();
    if (whole) break;
  }
  cut = INT_MAX;
  if (mask == 0xFFFFFFFFu) {
    uint32_t n_eq = 0;
    for (int i = t; i < n_in; i += kSelThreads) n_eq += gbuf[i].x == prefix ? 1u : 0u;
    uint32_t tot_eq;
    (void)block_excl_scan(n_eq, sh.scan, &tot_eq);
    if (tot_eq > static_cast<uint32_t>(r_rem)) {
      uint32_t pos_prefix = 0, pos_mask = 0;
      int rr = r_rem;
      for (int pl = 0; pl < 2; ++pl) {
        const int shift = pl == 0 ? 10 : 0;
        for (int i = t; i < kBinsL; i += kSelThreads) h[i] = 0u;
        __syncthreads();
        for (int i = t; i < n_in; i += kSelThreads) {
          const uint2 e = gbuf[i];
          if (e.x == prefix && (e.y & pos_mask) == pos_prefix)
            atomicAdd(&h[(e.y >> shift) & (kBinsL - 1)], 1u);
        }
        __syncthreads();
        find_bin_low(h, kBinsL, rr, sh);
        pos_prefix |= static_cast<uint32_t>(sh.f_bin) << shift;
        pos_mask |= static_cast<uint32_t>(kBinsL - 1) << shift;
        rr = sh.f_rem;
        __syncthreads();
      }
      cut = static_cast<int>(pos_prefix);
    }
  }
}

__global__ void __launch_bounds__(kSelThreads, 1) select_topk_kernel(const SelParams a) {
  extern __shared__ __align__(16) uint8_t sel_smem[];
  __shared__ SelShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int row = blockIdx.y;
  const int t = threadIdx.x;
  const int chunk = a.chunk;
  const int KPT = chunk / kSelThreads;  // 4, 8, 16 or 32 positions per thread
  const SelLayout L = sel_layout(sel_smem, chunk);

  // rank 0's cluster-wide arrays start at zero before anyone adds to them
  if (rank == 0)
    for (int i = t; i < kBins0 + 2 * kBinsL; i += kSelThreads) L.ghist[i] = 0u;
  if (t == 0) sh.gcount = 0u;
  for (int i = t; i < kBins0; i += kSelThreads) L.hist[i] = 0u;
  __syncthreads();
  cluster_arrive();  // this CTA's shared memory is ready; waited on before remote use
  ptx::pdl_wait_primary();  // the partial scores come from the preceding kernels
  ptx::pdl_launch_dependents();

  // Sums of 4 consecutive positions over the KV groups (fp32, groups in order).  Every
  // position below P_max is valid memory, so the first group of 4 is loaded before
  // the prefix length is known; positions at or past P are masked afterwards.
  const float* base = a.partial + static_cast<size_t>(row) * a.Hkv * a.P_max;
  const bool vec = (a.P_max & 3) == 0;
  auto sum4 = [&](int j, float (&s)[4]) {
    s[0] = s[1] = s[2] = s[3] = 0.f;
    if (vec && j + 3 < a.P_max) {
      int g = 0;
      for (; g + 8 <= a.Hkv; g += 8) {
        float4 x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          x[u] = __ldcg(reinterpret_cast<const float4*>(base + static_cast<size_t>(g + u) * a.P_max + j));
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          s[0] += x[u].x;
          s[1] += x[u].y;
          s[2] += x[u].z;
          s[3] += x[u].w;
        }
      }
      for (; g < a.Hkv; ++g) {
        const float4 x =
            __ldcg(reinterpret_cast<const float4*>(base + static_cast<size_t>(g) * a.P_max + j));
        s[0] += x.x;
        s[1] += x.y;
        s[2] += x.z;
        s[3] += x.w;
      }
    } else {
      for (int g = 0; g < a.Hkv; ++g)
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (j + u < a.P_max) s[u] += __ldcg(base + static_cast<size_t>(g) * a.P_max + j + u);
    }
  };
  const int my0 = rank * chunk + t * KPT;  // this thread's positions [my0, my0 + KPT)
  float s_first[4];
  sum4(my0, s_first);
  // scored input: the row's level-0 histogram is an input too -- its loads go out now
  constexpr int kHistPerThread = kBins0 / kSelThreads;
  uint32_t h_pre[kHistPerThread];
  if (a.hist != nullptr) {
#pragma unroll
    for (int i = 0; i < kHistPerThread; ++i)
      h_pre[i] = __ldcg(a.hist + static_cast<size_t>(row) * kBins0 + t + i * kSelThreads);
  }

  int P = __ldcg(a.prefix_len + row);
  if (P < 0 || P > a.P_max) {
    if (t == 0 && rank == 0) flag_status(a.status, VSD_DEV_BAD_LENGTH);
    P = 0;
  }
  const int n = a.k < P ? a.k : P;
  const int sink_end = a.n_sink < P ? a.n_sink : P;
  const int rb0 = P - a.n_recent > 0 ? P - a.n_recent : 0;
  const int rb = rb0 > sink_end ? rb0 : sink_end;  // candidates: [sink_end, rb)
  // scored input: the scores of the positions that are not ranked (sinks, recent
  // window) are taken out of the histogram below; the first 512 of them load now
  const int n_prot = sink_end + (P - rb);
  uint32_t prot_key = 0u;
  if (a.hist != nullptr && t < n_prot) {
    const int j = t < sink_end ? t : rb + (t - sink_end);
    prot_key = order_key(__ldcg(base + j));
  }
  // candidates chosen beforehand (first pass of the hybrid budget) are always taken
  // and not ranked; this thread's KPT positions sit in one word of that bitmap
  uint32_t pre_bits = 0u;
  int n_pre = 0;
  if (a.pre_bitmap != nullptr) {
    const int wi = my0 >> 5;
    if (wi < a.bm_words) {
      const uint32_t wv = __ldcg(a.pre_bitmap + static_cast<size_t>(row) * a.bm_words + wi);
      pre_bits = (wv >> (my0 & 31)) & (KPT >= 32 ? 0xFFFFFFFFu : ((1u << KPT) - 1u));
    }
    n_pre = __ldcg(a.pre_count + row);
  }
  const int n_cand = rb - sink_end - n_pre;  // rankable candidates
  int r_need = n - (P - (rb - sink_end)) - n_pre;
  if (a.m_limit >= 0 && r_need > a.m_limit) r_need = a.m_limit;
  const bool take_all = r_need >= n_cand;
  const bool ranking = r_need > 0 && !take_all;
  auto rankable = [&](int jj, int q) {
    return jj >= sink_end && jj < rb && !((pre_bits >> q) & 1u);
  };

  // ---- A. keys and the level-0 histogram of the candidates
  if (ranking || a.scores_out != nullptr) {
    auto finish4 = [&](int q, const float (&s)[4]) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int jj = my0 + q + u;
        const uint32_t key = jj < P ? order_key(s[u]) : 0u;
        L.keys[t * KPT + q + u] = key;
        if (jj < P && a.scores_out != nullptr)
          a.scores_out[static_cast<size_t>(row) * a.P_max + jj] = s[u];
        if (ranking && a.hist == nullptr && rankable(jj, q + u))
          atomicAdd(&L.hist[key >> 20], 1u);
      }
    };
    finish4(0, s_first);
    // the rest two groups of 4 per round, both groups' loads in flight together
    for (int q = 4; q < KPT; q += 8) {
      float s0[4], s1[4];
      sum4(my0 + q, s0);
      if (q + 4 < KPT) sum4(my0 + q + 4, s1);
      finish4(q, s0);
      if (q + 4 < KPT) finish4(q + 4, s1);
    }
  }
  __syncthreads();
  cluster_wait();  // every CTA's shared memory is ready

  uint32_t prefix = 0u, mask = 0u;
  int r_rem = r_need;
  int mode = kModeWhole;
  int level_bin = 0;
  if (ranking) {
    // ---- B/C. cluster histograms, level by level, until the boundary bin is small
    mode = kModeTie;
    for (int level = 0; level < 3; ++level) {
      const int nb = level == 0 ? kBins0 : kBinsL;
      const int shift = level == 0 ? 20 : (level == 1 ? 10 : 0);
      const uint32_t dmask = static_cast<uint32_t>(nb - 1);
      uint32_t* gh_local = L.ghist + (level == 0 ? 0 : kBins0 + (level - 1) * kBinsL);
      if (level > 0) {
        for (int i = t; i < nb; i += kSelThreads) L.hist[i] = 0u;
        __syncthreads();
        for (int q = 0; q < KPT; ++q) {
          const int j = my0 + q;
          const uint32_t key = L.keys[t * KPT + q];
          if (rankable(j, q) && (key & mask) == prefix)
            atomicAdd(&L.hist[(key >> shift) & dmask], 1u);
        }
        __syncthreads();
      }
      if (level == 0 && a.hist != nullptr) {
        // scored input: the histogram of every prefix position came with the scores;
        // each CTA takes the positions that are not ranked (sinks, recent window) out
        // of its own copy and searches it -- no cluster round
#pragma unroll
        for (int i = 0; i < kHistPerThread; ++i) gh_local[t + i * kSelThreads] = h_pre[i];
        if (t == 0) {
          // a histogram that does not hold r_rem candidates (not the one written with
          // these scores) finds no bin: take bin 0 whole, and flag it
          sh.f_bin = 0;
          sh.f_rem = 0;
          sh.f_cnt = -1;
        }
        __syncthreads();
        if (t < n_prot) atomicSub(&gh_local[prot_key >> 20], 1u);
        for (int i = t + kSelThreads; i < n_prot; i += kSelThreads) {
          const int j = i < sink_end ? i : rb + (i - sink_end);
          atomicSub(&gh_local[order_key(__ldcg(base + j)) >> 20], 1u);
        }
        __syncthreads();
        find_bin(gh_local, nb, r_rem, sh);
        if (sh.f_cnt < 0) {
          if (t == 0 && rank == 0) flag_status(a.status, VSD_DEV_BAD_LENGTH);
          __syncthreads();
          if (t == 0) {
            sh.f_rem = 1;
            sh.f_cnt = 1;
          }
          __syncthreads();
        }
      } else {
        uint32_t* gh0 = cluster.map_shared_rank(gh_local, 0);
        for (int b = t; b < nb; b += kSelThreads) {
          const uint32_t c = L.hist[b];
          if (c) atomicAdd(gh0 + b, c);
        }
        cluster_arrive();
        cluster_wait();  // rank 0's histogram of this level is complete
        if (rank == 0) {
          // rank 0 searches its histogram and hands the result to every CTA
          find_bin(gh_local, nb, r_rem, sh);
          if (t < static_cast<int>(cluster.num_blocks())) {
            SelShared* d = cluster.map_shared_rank(&sh, t);
            d->f_bin = sh.f_bin;
            d->f_rem = sh.f_rem;
            d->f_cnt = sh.f_cnt;
          }
        }
        cluster_arrive();
        cluster_wait();  // every CTA has the boundary bin of this level
      }
      const int bin = sh.f_bin;
      const int c_star = sh.f_cnt;
      r_rem = sh.f_rem;
      prefix |= static_cast<uint32_t>(bin) << shift;
      mask |= dmask << shift;
      level_bin = bin;
      __syncthreads();  // sh.f_* is written again by the next level
      if (r_rem == c_star) {
        mode = kModeWhole;  // the whole boundary bin is taken
        break;
      }
      if (c_star <= kGatherCap) {
        mode = kModeGather;
        break;
      }
      // level 2 fixes all 32 bits: more than kGatherCap keys equal to one value
    }
  }

  // ---- D. mark the sure winners, hand the boundary bin to rank 0
  uint32_t* lbm = L.loc;
  const int nw_cta = chunk / 32;
  const bool short_row = static_cast<int>(cluster.num_blocks()) * nw_cta <= kShortRowWords;
  uint64_t inbin_kept = 0;  // gather mode: this thread's boundary-bin positions
  {
    uint64_t sure = static_cast<uint64_t>(pre_bits), inbin = 0;
    for (int q = 0; q < KPT; ++q) {
      const int j = my0 + q;
      if (rankable(j, q)) {
        if (take_all) {
          sure |= 1ull << q;
        } else if (ranking) {
          const uint32_t km = L.keys[t * KPT + q] & mask;
          if (km > prefix) sure |= 1ull << q;
          else if (km == prefix) inbin |= 1ull << q;
        }
      }
    }
    if (mode == kModeWhole) {
      sure |= inbin;
      inbin = 0;
    } else if (mode == kModeTie) {
      // every boundary key equals the threshold: the first r_rem of them in position
      // order are taken; this CTA's share follows from the lower ranks' counts
      if (t < rank) sh.tmp[t] = *cluster.map_shared_rank(L.hist + level_bin, t);
      __syncthreads();
      long long before = 0;
      for (int r = 0; r < rank; ++r) before += sh.tmp[r];
      uint32_t tot_in;
      const int cnt = __popcll(inbin);
      const uint32_t pre = block_excl_scan(static_cast<uint32_t>(cnt), sh.scan, &tot_in);
      const long long left = static_cast<long long>(r_rem) - before - pre;
      uint64_t take = inbin;
      if (left <= 0) {
        take = 0;
      } else if (left < cnt) {
        for (int drop = cnt - static_cast<int>(left); drop > 0; --drop)
          take &= ~(1ull << (63 - __clzll(static_cast<long long>(take))));  // the highest
      }
      sure |= take;
      inbin = 0;
    }
    // this CTA's words of the position bitmap (short rows: also stored to rank 0); its
    // count goes to every CTA
    for (int i = t; i < nw_cta; i += kSelThreads) lbm[i] = 0u;
    __syncthreads();
    mark_bits(lbm, t * KPT, sure);
    uint32_t n_sure;
    (void)block_excl_scan(static_cast<uint32_t>(__popcll(sure)), sh.scan, &n_sure);
    if (t < static_cast<int>(cluster.num_blocks()))
      cluster.map_shared_rank(&sh, t)->cnt[rank] = n_sure;
    if (short_row) {
      uint32_t* bm0 = cluster.map_shared_rank(L.bitmap, 0);
      for (int i = t; i < nw_cta; i += kSelThreads) bm0[rank * nw_cta + i] = lbm[i];
    }
    if (mode == kModeGather) {
      // append (key, position) of the boundary bin to rank 0's buffer, one atomic per warp
      const int lane = t & 31;
      const uint32_t mine = static_cast<uint32_t>(__popcll(inbin));
      uint32_t incl = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t wtot = __shfl_sync(0xffffffffu, incl, 31);
      uint32_t wbase = 0;
      if (lane == 31 && wtot) wbase = atomicAdd(cluster.map_shared_rank(&sh.gcount, 0), wtot);
      wbase = __shfl_sync(0xffffffffu, wbase, 31);
      uint2* gb0 = cluster.map_shared_rank(L.gbuf, 0);
      uint32_t o = wbase + incl - mine;
      inbin_kept = inbin;
      while (inbin) {
        const int q = __ffsll(static_cast<long long>(inbin)) - 1;
        inbin &= inbin - 1;
        gb0[o++] = make_uint2(L.keys[t * KPT + q], static_cast<uint32_t>(my0 + q));
      }
    }
  }
  cluster_arrive();
  cluster_wait();  // every CTA has every count; rank 0 holds every boundary key
  const int CS = static_cast<int>(cluster.num_blocks());
  int32_t* dst = a.idx + static_cast<size_t>(row) * a.k;
  const int n_recent_kept = P - rb;

  if (short_row) {
    // ---- E/F (short rows). Rank 0 alone: resolve the boundary bin, mark the winners
    //      in its row bitmap, write the row from the bitmap
    if (rank != 0) return;
    if (mode == kModeGather) {
      const int n_in = static_cast<int>(sh.gcount);
      int cut;
      resolve_boundary(L.gbuf, n_in, L.hist, sh, prefix, mask, r_rem, cut);
      for (int i = t; i < n_in; i += kSelThreads) {
        const uint2 e = L.gbuf[i];
        const uint32_t km = e.x & mask;
        if (km > prefix || (km == prefix && static_cast<int>(e.y) <= cut))
          atomicOr(&L.bitmap[e.y >> 5], 1u << (e.y & 31));
      }
      __syncthreads();
    }
    const int nw_row = CS * nw_cta;
    uint32_t o_base = static_cast<uint32_t>(sink_end);
    for (int w0 = 0; w0 < nw_row; w0 += kSelThreads) {
      const int w = w0 + t;
      uint32_t bits = w < nw_row ? L.bitmap[w] : 0u;
      if (a.out_bitmap != nullptr && w < a.bm_words)
        a.out_bitmap[static_cast<size_t>(row) * a.bm_words + w] = bits;
      uint32_t r_tot;
      uint32_t o = o_base + block_excl_scan(static_cast<uint32_t>(__popc(bits)), sh.scan, &r_tot);
      while (bits) {
        const int bit = __ffs(bits) - 1;
        bits &= bits - 1;
        if (o < static_cast<uint32_t>(n)) dst[o] = w * 32 + bit;
        ++o;
      }
      o_base += r_tot;
    }
    if (a.out_count != nullptr && t == 0) a.out_count[row] = static_cast<int>(o_base) - sink_end;
    for (int i = t; i < sink_end; i += kSelThreads) dst[i] = i;
    for (int i = t; i < n_recent_kept; i += kSelThreads) dst[n - n_recent_kept + i] = rb + i;
    for (int m = n + t; m < a.k; m += kSelThreads) dst[m] = -1;
    if (t == 0) a.n_sel[row] = n;
    return;
  }

  // ---- E (long rows, gather mode): rank 0 resolves the boundary bin, counts the
  //      winners per owning CTA and hands every CTA the cut and where its candidates
  //      start in the row
  int out_base = sink_end;
  uint32_t total = 0;  // candidates chosen in the row (rank 0)
  if (mode == kModeGather) {
    if (rank == 0) {
      const int n_in = static_cast<int>(sh.gcount);
      int cut;
      resolve_boundary(L.gbuf, n_in, L.hist, sh, prefix, mask, r_rem, cut);
      if (t < CS) sh.taken[t] = 0u;
      __syncthreads();
      for (int i = t; i < n_in; i += kSelThreads) {
        const uint2 e = L.gbuf[i];
        const uint32_t km = e.x & mask;
        if (km > prefix || (km == prefix && static_cast<int>(e.y) <= cut))
          atomicAdd(&sh.taken[static_cast<int>(e.y) / chunk], 1u);
      }
      __syncthreads();
      if (t < CS) {
        uint32_t before = 0;
        for (int r = 0; r < t; ++r) before += sh.cnt[r] + sh.taken[r];
        SelShared* d = cluster.map_shared_rank(&sh, t);
        d->out_base = sink_end + static_cast<int>(before);
        d->thr_prefix = prefix;
        d->thr_mask = mask;
        d->thr_cut = cut;
      }
      for (int r = 0; r < CS; ++r) total += sh.cnt[r] + sh.taken[r];
    }
    cluster_arrive();
    cluster_wait();  // every CTA has the cut and its start
    // this CTA's boundary-bin positions that made the cut
    const uint32_t tp = sh.thr_prefix, tm = sh.thr_mask;
    const int tc = sh.thr_cut;
    uint64_t take = 0;
    for (uint64_t m = inbin_kept; m; m &= m - 1) {
      const int q = __ffsll(static_cast<long long>(m)) - 1;
      const uint32_t km = L.keys[t * KPT + q] & tm;
      if (km > tp || (km == tp && my0 + q <= tc)) take |= 1ull << q;
    }
    mark_bits(lbm, t * KPT, take);
    out_base = sh.out_base;
    __syncthreads();
  } else {
    for (int r = 0; r < CS; ++r) {
      if (r < rank) out_base += static_cast<int>(sh.cnt[r]);
      total += sh.cnt[r];
    }
  }

  // ---- F. every CTA writes its candidates in position order from its bitmap words
  //      (one word per thread per round, a block scan of the words' counts); rank 0
  //      writes the sinks, the recent window and the padding
  uint32_t o_base = static_cast<uint32_t>(out_base);
  for (int w0 = 0; w0 < nw_cta; w0 += kSelThreads) {
    const int w = w0 + t;
    uint32_t bits = w < nw_cta ? lbm[w] : 0u;
    if (a.out_bitmap != nullptr && w < nw_cta) {
      // this pass's chosen candidates, for the next pass of the hybrid budget
      const int gw = rank * nw_cta + w;
      if (gw < a.bm_words) a.out_bitmap[static_cast<size_t>(row) * a.bm_words + gw] = bits;
    }
    uint32_t r_tot;
    uint32_t o = o_base + block_excl_scan(static_cast<uint32_t>(__popc(bits)), sh.scan, &r_tot);
    while (bits) {
      const int bit = __ffs(bits) - 1;
      bits &= bits - 1;
      if (o < static_cast<uint32_t>(n)) dst[o] = rank * chunk + w * 32 + bit;
      ++o;
    }
    o_base += r_tot;
  }
  if (rank != 0) return;
  if (a.out_count != nullptr && t == 0) a.out_count[row] = static_cast<int>(total);
  for (int i = t; i < sink_end; i += kSelThreads) dst[i] = i;
  for (int i = t; i < n_recent_kept; i += kSelThreads) dst[n - n_recent_kept + i] = rb + i;
  for (int m = n + t; m < a.k; m += kSelThreads) dst[m] = -1;
  if (t == 0) a.n_sel[row] = n;
}


}  // namespace

int select_cluster_size(int P_max, int n_rows) {
  int cs = (P_max + kChunkQuantum - 1) / kChunkQuantum;
  if (cs < 1) cs = 1;
  const int cap = n_rows > 7 ? 8 : kMaxSelCluster;  // 16-CTA clusters: few fit at once
  if (cs > cap) cs = cap;
  int p2 = 1;
  while (p2 < cs) p2 <<= 1;
  return p2 > cap ? cap : p2;
}

int select_chunk(int P_max, int cs) {
  int chunk = (P_max + cs - 1) / cs;
  chunk = ((chunk + kChunkQuantum - 1) / kChunkQuantum) * kChunkQuantum;
  if (chunk < kChunkQuantum) chunk = kChunkQuantum;
  return chunk > kMaxChunk ? -1 : chunk;
}

size_t select_smem_bytes(int chunk, int cs) {
  (void)cs;
  return static_cast<size_t>(kGatherCap) * 8 +
         (static_cast<size_t>(chunk) + 2 * kBins0 + kBins0 + 2 * kBinsL + kShortRowWords) * 4;
}

cudaError_t launch_select(const SelectArgs& sa, cudaStream_t stream) {
  if (sa.n_rows == 0) return cudaSuccess;
  const int CS = select_cluster_size(sa.P_max, sa.n_rows);
  const int chunk = select_chunk(sa.P_max, CS);
  if (chunk < 0) return cudaErrorInvalidValue;
  SelParams p;
  p.partial = sa.partial;
  p.prefix_len = sa.prefix_len;
  p.idx = sa.idx;
  p.n_sel = sa.n_sel;
  p.scores_out = sa.scores_out;
  p.status = sa.status;
  p.Hkv = sa.Hkv;
  p.P_max = sa.P_max;
  p.k = sa.k;
  p.n_sink = sa.n_sink;
  p.n_recent = sa.n_recent;
  p.chunk = chunk;
  p.m_limit = sa.m_limit;
  p.pre_bitmap = sa.pre_bitmap;
  p.pre_count = sa.pre_count;
  p.out_bitmap = sa.out_bitmap;
  p.out_count = sa.out_count;
  p.bm_words = (sa.P_max + 31) / 32;
  p.hist = sa.hist;
  const size_t smem = select_smem_bytes(chunk, CS);
  cudaError_t e = cudaFuncSetAttribute(select_topk_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (CS > 8) {
    e = cudaFuncSetAttribute(select_topk_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed,
                             1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CS, sa.n_rows, 1);
  cfg.blockDim = dim3(kSelThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, select_topk_kernel, p);
}

}  // namespace vsd
