// select_topk.cu -- aggregated-logit top-k with a protected budget on sm_103a.
//
// What it computes: the Vegas selection (technical summary sec. 2.A: the prefix set
// T with |T| = k maximising the logits summed over the collected rows and all query
// heads -- a separable objective, so the k highest scores) under the Dustin budget
// rule (Methodology sec. 1: attention sinks and the recent window are kept first,
// the rest of the budget is filled by score).  Equal scores go to the lower position;
// the output is in ascending position order.
//
// How (GB300 design).  One thread-block cluster per row (layer x sequence), each CTA
// owning a contiguous slice of the prefix, each thread a contiguous run of KPT
// positions.  Scores become order-preserving uint32 keys; the task is to find the
// threshold key T and the tie cut c such that exactly r = k - |protected| candidates
// satisfy  key > T  or  (key == T and position <= c).
//   A. Every CTA sums the per-KV-group partial scores of its slice (fp32, groups in
//      order; the partials are L2-resident after verification), keeps the keys in
//      shared memory and builds a 4096-bin histogram of their top 12 bits.
//   B. Cluster barrier.  CTA i adds up bins [i n/CS, (i+1) n/CS) of all CTAs'
//      histograms (distributed shared memory, all loads in flight at once).
//   C. Cluster barrier.  Every CTA finds the slice, then the bin, holding the r-th
//      largest key.  If that bin still holds more than the gather capacity, the
//      next 10 bits are histogrammed the same way (rare; at most two more levels).
//   D. Every CTA copies its keys of the boundary bin, in position order, to rank 0
//      (offsets from the per-CTA bin counts) and reports its counts.
//   E. Cluster barrier.  Rank 0 alone resolves the remaining bits and the tie cut on
//      the gathered keys with block-local passes, then writes T, c and the output
//      offset of every CTA into that CTA's shared memory.
//   F. Cluster barrier.  Every CTA writes its selected positions in order.
// Four cluster barriers in the common case, no global workspace, no atomics on
// results, and deterministic output.  The kernel is launched as a programmatic
// dependent: its launch overlaps the tail of the verification kernels.
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
constexpr int kMaxChunk = 32768;
constexpr int kBins0 = 4096;                     // level 0: top 12 bits
constexpr int kBinsL = 1024;                     // levels 1, 2: 10 bits each
constexpr int kGatherCap = 8192;                 // boundary-bin keys rank 0 can hold

enum Mode : int { kModeWhole = 0, kModeGather = 1, kModeTie = 2 };

struct SelParams {
  const float* partial;
  const int32_t* prefix_len;
  int32_t* idx;
  int32_t* n_sel;
  float* scores_out;
  unsigned* status;
  int Hkv, P_max, k, n_sink, n_recent, chunk;
};

struct SelShared {
  uint32_t scan[kSelWarps];
  uint32_t slice_tot;
  uint32_t tmp[kSelWarps];
  // result of a bin search
  int f_bin;
  int f_rem;
  int f_cnt;
  // counts reported to rank 0 by every CTA
  uint32_t above[kMaxSelCluster];
  uint32_t inbin[kMaxSelCluster];
  uint32_t sel_in[kMaxSelCluster];
  uint32_t stot[kMaxSelCluster];
  // decision broadcast by rank 0
  uint32_t T;
  int cut;
  uint32_t out_off;
};

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum over the threads of the block in thread order; *total gets
// the block sum.  Contains two __syncthreads and leaves `scratch` reusable.
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

// Among bins cnt[0..n) (ascending key order) find the bin b holding the r-th
// largest element (1 <= r <= sum): S(b+1) < r <= S(b) with S(b) = sum of cnt[b..n).
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

__global__ void __launch_bounds__(kSelThreads, 1) select_topk_kernel(const SelParams a) {
  extern __shared__ __align__(16) uint8_t sel_smem[];
  __shared__ SelShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int CS = static_cast<int>(cluster.num_blocks());
  const int row = blockIdx.y;
  const int t = threadIdx.x;
  const int chunk = a.chunk;
  const int KPT = chunk / kSelThreads;
  uint32_t* keys = reinterpret_cast<uint32_t*>(sel_smem);           // [chunk]
  uint32_t* hist = keys + chunk;                                      // [kBins0]
  uint32_t* red = hist + kBins0;                                      // [kBins0 / CS]
  uint32_t* loc = red + kBins0 / CS;                                  // [kBins0 / CS]
  uint2* gather = reinterpret_cast<uint2*>(loc + kBins0 / CS);       // [kGatherCap]

  ptx::pdl_launch_dependents();
  ptx::pdl_wait_primary();  // the partial scores come from the preceding kernels

  int P = __ldg(a.prefix_len + row);
  if (P < 0 || P > a.P_max) {
    if (t == 0 && rank == 0) flag_status(a.status, VSD_DEV_BAD_LENGTH);
    P = 0;
  }
  const int n = a.k < P ? a.k : P;
  const int sink_end = a.n_sink < P ? a.n_sink : P;
  const int rb0 = P - a.n_recent > 0 ? P - a.n_recent : 0;
  const int rb = rb0 > sink_end ? rb0 : sink_end;  // candidates: [sink_end, rb)
  const int n_cand = rb - sink_end;
  const int r_need = n - (P - n_cand);
  const int lo = rank * chunk;
  const int my0 = lo + t * KPT;  // this thread's positions [my0, my0 + KPT)

  // protected positions in [x0, x1)
  auto prot_in = [&](int x0, int x1) {
    const int a0 = max(x0, 0), a1 = min(x1, sink_end);
    const int b0 = max(x0, rb), b1 = min(x1, P);
    return max(a1 - a0, 0) + max(b1 - b0, 0);
  };
  auto cand_in = [&](int x0, int x1) {
    return max(min(x1, rb) - max(x0, sink_end), 0);
  };
  const bool all_or_none = r_need <= 0 || r_need >= n_cand;

  if (!all_or_none)
    for (int i = t; i < kBins0; i += kSelThreads) hist[i] = 0u;
  if (!all_or_none || a.scores_out != nullptr) {
    if (!all_or_none) __syncthreads();
    // ---- A. aggregated scores, keys and the level-0 histogram
    const float* base = a.partial + static_cast<size_t>(row) * a.Hkv * a.P_max;
    const bool vec = (a.P_max & 3) == 0;
    for (int q = 0; q < KPT; q += 4) {
      const int j = my0 + q;
      float s[4] = {0.f, 0.f, 0.f, 0.f};
      if (vec && j + 3 < P) {
        int g = 0;
        for (; g + 8 <= a.Hkv; g += 8) {
          float4 x[8];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            x[u] = __ldg(reinterpret_cast<const float4*>(base + static_cast<size_t>(g + u) * a.P_max + j));
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            s[0] += x[u].x;
            s[1] += x[u].y;
            s[2] += x[u].z;
            s[3] += x[u].w;
          }
        }
        for (; g < a.Hkv; ++g) {
          const float4 x = __ldg(reinterpret_cast<const float4*>(base + static_cast<size_t>(g) * a.P_max + j));
          s[0] += x.x;
          s[1] += x.y;
          s[2] += x.z;
          s[3] += x.w;
        }
      } else {
        for (int g = 0; g < a.Hkv; ++g)
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (j + u < P) s[u] += __ldg(base + static_cast<size_t>(g) * a.P_max + j + u);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int jj = j + u;
        const uint32_t key = jj < P ? order_key(s[u]) : 0u;
        keys[t * KPT + q + u] = key;
        if (jj < P && a.scores_out != nullptr)
          a.scores_out[static_cast<size_t>(row) * a.P_max + jj] = s[u];
        if (!all_or_none && jj >= sink_end && jj < rb) atomicAdd(&hist[key >> 20], 1u);
      }
    }
  }

  uint32_t T = 0u;
  int cut = INT_MAX;
  uint32_t out_off = 0;
  if (all_or_none) {
    // nothing to rank: every candidate or none of them is taken
    T = r_need <= 0 ? 0xFFFFFFFFu : 0u;
    cut = r_need <= 0 ? -1 : INT_MAX;
    out_off = prot_in(0, lo) + (r_need <= 0 ? 0 : cand_in(0, lo));
  } else {
    // ---- B/C. cluster histogram levels until the boundary bin is small enough
    uint32_t prefix = 0u, mask = 0u;
    int r_rem = r_need;
    int mode = kModeTie;
    int level_bin = 0;  // bin of the final level (index into every CTA's hist)
    for (int level = 0; level < 3; ++level) {
      const int nb = level == 0 ? kBins0 : kBinsL;
      const int shift = level == 0 ? 20 : (level == 1 ? 10 : 0);
      const uint32_t dmask = static_cast<uint32_t>(nb - 1);
      if (level > 0) {
        // every CTA has read the previous level's histograms (barrier below), so
        // they can be rebuilt for this level's digit
        for (int i = t; i < nb; i += kSelThreads) hist[i] = 0u;
        __syncthreads();
        for (int q = 0; q < KPT; ++q) {
          const int j = my0 + q;
          const uint32_t key = keys[t * KPT + q];
          if (j >= sink_end && j < rb && (key & mask) == prefix)
            atomicAdd(&hist[(key >> shift) & dmask], 1u);
        }
      }
      cluster.sync();  // all histograms of this level complete
      const int sl = nb / CS;
      const int sbase = rank * sl;
      uint32_t part = 0;
      for (int b = t; b < sl; b += kSelThreads) {
        uint32_t v[kMaxSelCluster];
#pragma unroll
        for (int r = 0; r < kMaxSelCluster; ++r)
          v[r] = r < CS ? *cluster.map_shared_rank(hist + sbase + b, r) : 0u;
        uint32_t s = 0;
#pragma unroll
        for (int r = 0; r < kMaxSelCluster; ++r) s += v[r];
        red[b] = s;
        part += s;
      }
      uint32_t tot;
      (void)block_excl_scan(part, sh.scan, &tot);
      if (t == 0) sh.slice_tot = tot;
      cluster.sync();  // all slices reduced
      // slice holding the r_rem-th largest: read every CTA's slice total
      if (t < CS) sh.stot[t] = *cluster.map_shared_rank(&sh.slice_tot, t);
      __syncthreads();
      int s_star = 0;
      uint32_t above = 0;
      for (int r = CS - 1; r >= 0; --r) {
        const uint32_t c = sh.stot[r];
        if (above + c >= static_cast<uint32_t>(r_rem)) {
          s_star = r;
          break;
        }
        above += c;
      }
      // copy that slice locally, then search it
      for (int b = t; b < sl; b += kSelThreads)
        loc[b] = *cluster.map_shared_rank(red + b, s_star);
      __syncthreads();
      find_bin(loc, sl, r_rem - static_cast<int>(above), sh);
      const int b_local = sh.f_bin;
      const int bin = s_star * sl + b_local;
      const int c_star = sh.f_cnt;
      r_rem = sh.f_rem;
      prefix |= static_cast<uint32_t>(bin) << shift;
      mask |= dmask << shift;
      level_bin = bin;
      __syncthreads();  // sh.f_* and loc are written again by the next level
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

    // ---- D. counts (and the boundary-bin keys) to rank 0
    uint32_t c_above = 0, c_in = 0;
    for (int q = 0; q < KPT; ++q) {
      const int j = my0 + q;
      if (j >= sink_end && j < rb) {
        const uint32_t km = keys[t * KPT + q] & mask;
        c_above += km > prefix ? 1u : 0u;
        c_in += km == prefix ? 1u : 0u;
      }
    }
    uint32_t tot_above, tot_in;
    const uint32_t packed = c_above | (c_in << 16);  // both below 2^16 per CTA
    uint32_t tot_packed;
    const uint32_t pre = block_excl_scan(packed, sh.scan, &tot_packed);
    tot_above = tot_packed & 0xFFFFu;
    tot_in = tot_packed >> 16;
    if (mode == kModeGather) {
      // this CTA's first slot: boundary-bin keys of the lower ranks
      if (t < rank) sh.tmp[t] = *cluster.map_shared_rank(hist + level_bin, t);
      __syncthreads();
      uint32_t base = 0;
      for (int r = 0; r < rank; ++r) base += sh.tmp[r];
      uint2* dst = cluster.map_shared_rank(gather, 0);
      uint32_t o = base + (pre >> 16);
      for (int q = 0; q < KPT; ++q) {
        const int j = my0 + q;
        const uint32_t key = keys[t * KPT + q];
        if (j >= sink_end && j < rb && (key & mask) == prefix) {
          dst[o] = make_uint2(key, static_cast<uint32_t>(j));
          ++o;
        }
      }
    }
    if (t == 0) {
      *cluster.map_shared_rank(&sh.above[rank], 0) = tot_above;
      *cluster.map_shared_rank(&sh.inbin[rank], 0) = tot_in;
    }
    cluster.sync();  // gathered keys and counts are at rank 0

    // ---- E. rank 0 resolves the threshold and the output offsets
    if (rank == 0) {
      uint32_t n_in = 0;
      for (int r = 0; r < CS; ++r) n_in += sh.inbin[r];
      if (t < kMaxSelCluster) sh.sel_in[t] = 0u;
      if (t == 0) sh.cut = INT_MAX;
      if (mode == kModeWhole) {
        T = prefix;
        cut = INT_MAX;
        if (t < CS) sh.sel_in[t] = sh.inbin[t];
      } else if (mode == kModeGather) {
        // remaining digits of the gathered keys
        int start_level = 1;
        if ((mask & 0x000FFC00u) != 0) start_level = 2;
        if (mask == 0xFFFFFFFFu) start_level = 3;
        for (int level = start_level; level < 3; ++level) {
          const int shift = level == 1 ? 10 : 0;
          for (int i = t; i < kBinsL; i += kSelThreads) hist[i] = 0u;
          __syncthreads();
          for (uint32_t i = t; i < n_in; i += kSelThreads) {
            const uint32_t key = gather[i].x;
            if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & (kBinsL - 1)], 1u);
          }
          __syncthreads();
          find_bin(hist, kBinsL, r_rem, sh);
          prefix |= static_cast<uint32_t>(sh.f_bin) << shift;
          mask |= static_cast<uint32_t>(kBinsL - 1) << shift;
          const bool whole = sh.f_rem == sh.f_cnt;
          r_rem = sh.f_rem;
          __syncthreads();
          if (whole) break;
        }
        // T = prefix.  If the mask is complete, r_rem keys equal to T are taken in
        // position order; otherwise the whole bin below the mask is taken.
        T = prefix;
        const bool full = mask == 0xFFFFFFFFu;
        const int E = (static_cast<int>(n_in) + kSelThreads - 1) / kSelThreads;
        const int i0 = t * E;
        const int i1 = min(i0 + E, static_cast<int>(n_in));
        if (full) {
          uint32_t ce = 0;
          for (int i = i0; i < i1; ++i) ce += gather[i].x == T ? 1u : 0u;
          uint32_t tot_eq;
          const uint32_t before = block_excl_scan(ce, sh.scan, &tot_eq);
          const uint32_t ur = static_cast<uint32_t>(r_rem);
          if (before < ur && ur <= before + ce) {
            uint32_t acc = before;
            for (int i = i0; i < i1; ++i) {
              if (gather[i].x == T && ++acc == ur) {
                sh.cut = static_cast<int>(gather[i].y);
                break;
              }
            }
          }
          __syncthreads();
          cut = sh.cut;
        } else {
          T = prefix;  // smallest key with this prefix: every key of the bin is >= T
          cut = INT_MAX;
        }
        for (int i = i0; i < i1; ++i) {
          const uint32_t key = gather[i].x;
          const int j = static_cast<int>(gather[i].y);
          const bool sel = full ? (key > T || (key == T && j <= cut)) : ((key & mask) >= prefix);
          if (sel) atomicAdd(&sh.sel_in[j / chunk], 1u);
        }
      } else {
        // kModeTie: every boundary key equals T; take the first r_rem in position order
        T = prefix;
        int rc = 0;
        uint32_t before_rc = 0;
        for (int r = 0; r < CS; ++r) {
          const uint32_t c = sh.inbin[r];
          if (before_rc + c >= static_cast<uint32_t>(r_rem)) {
            rc = r;
            break;
          }
          before_rc += c;
        }
        const uint32_t e = static_cast<uint32_t>(r_rem) - before_rc;  // 1-based within rc
        const uint32_t* rkeys = cluster.map_shared_rank(keys, rc);
        const int base_j = rc * chunk + t * KPT;
        uint32_t ce = 0;
        for (int q = 0; q < KPT; ++q) {
          const int j = base_j + q;
          ce += (j >= sink_end && j < rb && rkeys[t * KPT + q] == T) ? 1u : 0u;
        }
        uint32_t tot_eq;
        const uint32_t before = block_excl_scan(ce, sh.scan, &tot_eq);
        if (before < e && e <= before + ce) {
          uint32_t acc = before;
          for (int q = 0; q < KPT; ++q) {
            const int j = base_j + q;
            if (j >= sink_end && j < rb && rkeys[t * KPT + q] == T && ++acc == e) {
              sh.cut = j;
              break;
            }
          }
        }
        __syncthreads();
        cut = sh.cut;
        if (t < CS) {
          uint32_t bef = 0;
          for (int r = 0; r < t; ++r) bef += sh.inbin[r];
          const int left = r_rem - static_cast<int>(bef);
          sh.sel_in[t] = static_cast<uint32_t>(min(max(left, 0), static_cast<int>(sh.inbin[t])));
        }
      }
      __syncthreads();
      if (t < CS) {
        uint32_t off = 0;
        for (int r = 0; r < t; ++r) off += prot_in(r * chunk, (r + 1) * chunk) + sh.above[r] + sh.sel_in[r];
        SelShared* dst = cluster.map_shared_rank(&sh, t);
        dst->T = T;
        dst->cut = cut;
        dst->out_off = off;
      }
    }
    cluster.sync();  // every CTA has its threshold and offset
    T = sh.T;
    cut = sh.cut;
    out_off = sh.out_off;
  }

  // ---- F. selected positions of this slice, in order
  uint32_t cs = 0;
  for (int q = 0; q < KPT; ++q) {
    const int j = my0 + q;
    if (j >= P) break;
    bool sel;
    if (j < sink_end || j >= rb) {
      sel = true;
    } else {
      const uint32_t key = all_or_none ? 0u : keys[t * KPT + q];
      sel = all_or_none ? (r_need > 0) : (key > T || (key == T && j <= cut));
    }
    cs += sel ? 1u : 0u;
  }
  uint32_t cs_total;
  uint32_t o = out_off + block_excl_scan(cs, sh.scan, &cs_total);
  int32_t* dst = a.idx + static_cast<size_t>(row) * a.k;
  for (int q = 0; q < KPT; ++q) {
    const int j = my0 + q;
    if (j >= P) break;
    bool sel;
    if (j < sink_end || j >= rb) {
      sel = true;
    } else {
      const uint32_t key = all_or_none ? 0u : keys[t * KPT + q];
      sel = all_or_none ? (r_need > 0) : (key > T || (key == T && j <= cut));
    }
    if (sel) {
      if (o < static_cast<uint32_t>(n)) dst[o] = j;
      ++o;
    }
  }
  // unused slots and the count
  for (int m = n + rank * kSelThreads + t; m < a.k; m += CS * kSelThreads) dst[m] = -1;
  if (rank == 0 && t == 0) a.n_sel[row] = n;
}

}  // namespace

int select_cluster_size(int P_max, int n_rows) {
  int cs = (P_max + kChunkQuantum - 1) / kChunkQuantum;
  if (cs < 1) cs = 1;
  const int cap = n_rows > 7 ? 8 : kMaxSelCluster;  // 16-CTA clusters: few fit at once
  if (cs > cap) cs = cap;
  // power of two, so every slice of the histograms has the same size
  int p2 = 1;
  while (p2 < cs) p2 <<= 1;
  cs = p2 > cap ? cap : p2;
  return cs;
}

int select_chunk(int P_max, int cs) {
  int chunk = (P_max + cs - 1) / cs;
  chunk = ((chunk + kChunkQuantum - 1) / kChunkQuantum) * kChunkQuantum;
  if (chunk < kChunkQuantum) chunk = kChunkQuantum;
  return chunk > kMaxChunk ? -1 : chunk;
}

size_t select_smem_bytes(int chunk, int cs) {
  return static_cast<size_t>(chunk) * 4 + kBins0 * 4 + static_cast<size_t>(kBins0 / cs) * 8 +
         static_cast<size_t>(kGatherCap) * 8;
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
