// select_scored.cu -- the protected top-k selection from an aggregated score (the
// scored path: the fused verification has already summed the collected logits over
// the KV groups and counted the level-0 histogram of every prefix position).
//
// What it computes: the Vegas selection (technical summary sec. 2.A: the k prefix
// positions with the highest logits summed over the collected rows and all query heads)
// under the Dustin budget rule (Methodology sec. 1: the attention sinks and the recent
// window are kept first, the rest of the budget goes by score).  Equal scores go to the
// lower position; the row is written in ascending position order.  The index sets are
// bit for bit those of the selection that aggregates the partial scores itself.
//
// How (GB300 design).  The step is short and bound by the latency of its dependent
// rounds.  A row is split into slices of 4K-32K positions, one CTA (512 threads) each,
// the CTAs of a row forming one cluster; a slice stays in registers as order-preserving
// keys for the whole kernel.
//   1. Every CTA loads its slice and the row's level-0 histogram (top 12 key bits) of
//      the candidates (the verification call leaves the sinks and the recent window
//      out of it; a histogram of every prefix position has them taken out here, from
//      the scores) and finds the boundary bin, the one holding the r-th largest
//      candidate key (r = the budget left after the protected positions).  Every CTA
//      reaches the same bin without an exchange.  Rank 0 writes the protected part of
//      the row and its padding after the exchange.
//   2. Common case (the boundary bin holds at most 4096 keys): every CTA appends its
//      boundary-bin keys, with their positions, to every CTA's list and posts its count
//      of keys above the bin -- one cluster barrier -- and then resolves the cut on the
//      full list by itself: the remaining 20 key bits in two 10-bit histogram rounds,
//      then, among keys equal to the cut, the lowest positions (two 10-bit rounds on the
//      positions).  From the list it also knows how many of each CTA's keys are taken,
//      so it knows where its own output starts: no further exchange.
//      Otherwise (a bin of more than 4096 keys: long runs of equal scores) the next 10
//      key bits are histogrammed over the cluster's registers, one barrier per level,
//      and the equal keys at the cut are ranked by a scan and a final exchange.
//   3. Every CTA writes its taken positions in order: one block scan of its taken
//      counts in position order.
// The kernel is a programmatic dependent: its launch overlaps the tail of the
// verification kernels and it waits for their results before reading any.
#include <cooperative_groups.h>

#include <climits>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace vsd {
namespace {

constexpr int kScThreads = 512;
constexpr int kScWarps = kScThreads / 32;
constexpr int kScBins0 = 4096;  // level 0: top 12 key bits (the histogram given)
constexpr int kScBinsL = 1024;  // later levels: 10 bits each
constexpr int kScMaxCluster = 16;
constexpr int kScMaxGroups = 16;  // float4 groups a thread: up to 64 positions
constexpr int kScListCap = 4096;  // boundary-bin entries every CTA can hold
// dynamic shared memory: the level-0 histogram, the boundary-bin list and (clusters of
// two or more: segments of at most half the list) the staging copy of this CTA's entries
constexpr int kScDynBytes = kScBins0 * 4 + kScListCap * 8 + kScListCap / 2 * 8;

struct ScParams {
  const float* score;    // [n_rows][P_max]
  const uint32_t* hist;  // [n_rows][4096]
  const int32_t* prefix_len;
  int32_t* idx;          // [n_rows][k]
  int32_t* n_sel;
  unsigned* status;
  int P_max, k, n_sink, n_recent;
};

struct ScShared {
  uint32_t hl[2][kScBinsL];           // levels path: this CTA's counts
  uint32_t hs[2][kScBinsL];           // levels path: the cluster's sums
  uint32_t hr[4][kScBinsL];           // list resolution rounds (zeroed up front)
  uint64_t bar_list;                  // list path: every CTA's entries have arrived
  uint32_t tot[kScMaxCluster];        // levels path: per CTA, above | equal << 16
  uint32_t above[kScMaxCluster];      // list path: per CTA, keys above the boundary bin
  uint32_t real[kScMaxCluster];       // list path: per CTA, its boundary-bin entries
  uint32_t taken[kScMaxCluster];      // list path: per CTA, boundary-bin keys taken
  uint32_t wsum[kScMaxGroups][kScWarps];
  uint32_t gtot[kScMaxGroups];
  uint32_t scan[kScWarps];
  int f_bin, f_rem, f_cnt;
  uint32_t f_tot;
};

__device__ __forceinline__ uint32_t sc_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ void sc_cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void sc_cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The same shared-memory variable in cluster CTA `rank` (a shared::cluster address).
__device__ __forceinline__ uint32_t sc_peer(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(ptx::smem_u32(p)), "r"(rank));
  return r;
}

// Arrive on a peer CTA's barrier announcing `bytes` of bulk copy to it.  Relaxed: all
// the peer reads after its wait arrives by the bulk copy itself, so nothing else has
// to be ordered (a release would also wait for this CTA's pending global stores).
__device__ __forceinline__ void sc_peer_arrive_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void sc_cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

// Bulk copy of `bytes` (a multiple of 16) from this CTA's shared memory into a peer's,
// completing on the peer's barrier.
__device__ __forceinline__ void sc_bulk_to_peer(uint32_t dst, const void* src, uint32_t bytes,
                                                uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "r"(ptx::smem_u32(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// Wait (bounded) for phase 0 of a local barrier that peers arrive on.
__device__ __forceinline__ bool sc_wait_peers(uint64_t* bar) {
  const uint32_t a = ptx::smem_u32(bar);
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(a), "r"(0u)
        : "memory");
    if (done) return true;
    if (it == 0) t0 = ptx::global_timer_ns();
    if ((it & 63u) == 63u && ptx::global_timer_ns() - t0 > VSD_WAIT_LIMIT_NS) return false;
  }
}

// Exclusive prefix sum of v over the block's threads in thread order; *total gets the
// block sum.  The 16 warp totals are scanned by shuffles in every warp.
__device__ __forceinline__ uint32_t sc_block_scan(uint32_t v, uint32_t* scratch,
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
  uint32_t w = lane < kScWarps ? scratch[lane] : 0u;
#pragma unroll
  for (int o = 1; o < kScWarps; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
    if (lane >= o) w += y;
  }
  const uint32_t incl = __shfl_sync(0xffffffffu, w, warp);
  const uint32_t wtot = __shfl_sync(0xffffffffu, x, 31);
  *total = __shfl_sync(0xffffffffu, w, kScWarps - 1);
  __syncthreads();  // scratch reusable
  return incl - wtot + x - v;
}

// The bin holding the r-th element of n bins (cnt), counted from the top (descending)
// or from the bottom: sh.f_bin (-1 when the bins hold fewer than r), sh.f_rem = r minus
// the elements before that bin, sh.f_cnt = its count, sh.f_tot = the bins' sum.
template <bool kFromTop>
__device__ void sc_find_bin(const uint32_t* cnt, int n, uint32_t r, ScShared& sh) {
  const int E = n / kScThreads;  // 8 or 2 bins a thread, contiguous
  const int t = threadIdx.x;
  // the thread's bins in search order: first, then first -/+ 1, ...
  const int first = kFromTop ? n - 1 - t * E : t * E;
  uint32_t s = 0;
  for (int e = 0; e < E; ++e) s += cnt[kFromTop ? first - e : first + e];
  if (t == 0) sh.f_bin = -1;
  uint32_t tot;
  const uint32_t before = sc_block_scan(s, sh.scan, &tot);  // its syncs order the reset
  if (t == 0) sh.f_tot = tot;
  if (before < r && r <= before + s) {
    uint32_t acc = before;
    for (int e = 0; e < E; ++e) {
      const int b = kFromTop ? first - e : first + e;
      const uint32_t c = cnt[b];
      if (acc + c >= r) {
        sh.f_bin = b;
        sh.f_rem = static_cast<int>(r - acc);
        sh.f_cnt = static_cast<int>(c);
        break;
      }
      acc += c;
    }
  }
  __syncthreads();
}

// Calls f(entry) for every list entry: CTA q's entries sit at
// [q * segcap + 2, q * segcap + 2 + real[q]).  Warp q walks segment q (a cluster has at
// most 16 CTAs, a CTA 16 warps); a single CTA's one segment is walked by all threads.
template <typename F>
__device__ __forceinline__ void sc_for_entries(const uint2* list, int CS, uint32_t segcap,
                                               const ScShared& sh, F&& f) {
  const int t = threadIdx.x;
  if (CS == 1) {
    const int n = static_cast<int>(sh.real[0]);
    for (int i = t; i < n; i += kScThreads) f(list[2 + i]);
  } else {
    const int w = t >> 5;
    if (w < CS) {
      const uint2* seg = list + w * segcap + 2;
      const int n = static_cast<int>(sh.real[w]);
      for (int i = t & 31; i < n; i += 32) f(seg[i]);
    }
  }
}

// The cut among the list entries (key, position) of boundary bin b0: `need` of them
// (1 <= need <= all) are taken, those with key > T or key == T at a position <= cut.
// Every CTA holding the same entries reaches the same (T, cut).  The four rounds use
// the zeroed sh.hr[0..3].
__device__ void sc_resolve_list(const uint2* list, int CS, uint32_t segcap, uint32_t b0,
                                int need, int all, ScShared& sh, uint32_t& T, int& cut) {
  uint32_t prefix = b0 << 20, mask = 0xFFF00000u;
  int rem = need, cnt = all;
  for (int level = 0; level < 2; ++level) {
    const int shift = level == 0 ? 10 : 0;
    uint32_t* h = sh.hr[level];
    sc_for_entries(list, CS, segcap, sh, [&](uint2 e) {
      if ((e.x & mask) == prefix) atomicAdd(&h[(e.x >> shift) & (kScBinsL - 1)], 1u);
    });
    __syncthreads();
    sc_find_bin<true>(h, kScBinsL, static_cast<uint32_t>(rem), sh);
    if (sh.f_bin < 0) break;  // cannot happen for a list that holds the whole bin
    prefix |= static_cast<uint32_t>(sh.f_bin) << shift;
    mask |= static_cast<uint32_t>(kScBinsL - 1) << shift;
    rem = sh.f_rem;
    cnt = sh.f_cnt;
    if (rem == cnt && prefix != 0u) {  // the bin is taken whole: every key >= prefix
      T = prefix - 1u;
      cut = -1;
      return;
    }
  }
  T = prefix;
  if (rem >= cnt) {
    cut = INT_MAX;
    return;
  }
  // the rem lowest positions among the keys equal to T (positions are below 2^20)
  uint32_t pp = 0u, pm = 0u;
  for (int level = 0; level < 2; ++level) {
    const int shift = level == 0 ? 10 : 0;
    uint32_t* h = sh.hr[2 + level];
    const uint32_t tk = T;
    sc_for_entries(list, CS, segcap, sh, [&](uint2 e) {
      if (e.x == tk && (e.y & pm) == pp) atomicAdd(&h[(e.y >> shift) & (kScBinsL - 1)], 1u);
    });
    __syncthreads();
    sc_find_bin<false>(h, kScBinsL, static_cast<uint32_t>(rem), sh);
    if (sh.f_bin < 0) break;
    pp |= static_cast<uint32_t>(sh.f_bin) << shift;
    pm |= static_cast<uint32_t>(kScBinsL - 1) << shift;
    rem = sh.f_rem;
  }
  cut = static_cast<int>(pp);
}

// Exclusive scan of v over (group i, thread t) in i-major order -- position order of
// the slice; returns the CTA total.
template <int NG>
__device__ __forceinline__ uint32_t sc_group_scan(uint32_t (&v)[NG], ScShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int i = 0; i < NG; ++i) {
    uint32_t x = v[i];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) sh.wsum[i][warp] = x;
    v[i] = x - v[i];
  }
  __syncthreads();
  if (warp < NG) {  // warp i scans group i's warp totals
    const uint32_t s = lane < kScWarps ? sh.wsum[warp][lane] : 0u;
    uint32_t x = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane < kScWarps) sh.wsum[warp][lane] = x - s;
    if (lane == 31) sh.gtot[warp] = x;
  }
  __syncthreads();
  uint32_t run = 0u;
#pragma unroll
  for (int i = 0; i < NG; ++i) {
    v[i] += sh.wsum[i][warp] + run;
    run += sh.gtot[i];
  }
  return run;
}

template <int NG>
__global__ void __launch_bounds__(kScThreads, (NG <= 4 ? 2 : 1))
    select_scored_kernel(const ScParams a) {
  extern __shared__ __align__(16) uint8_t sc_dyn[];
  __shared__ ScShared sh;
  uint32_t* h0 = reinterpret_cast<uint32_t*>(sc_dyn);             // [4096]
  uint2* list = reinterpret_cast<uint2*>(sc_dyn + kScBins0 * 4);  // [kScListCap]
  constexpr int kChunk = NG * 4 * kScThreads;
  const int CS = static_cast<int>(gridDim.x);  // the cluster spans the row
  const int rank = static_cast<int>(blockIdx.x);
  const int row = blockIdx.y;
  const int t = threadIdx.x;

  for (int i = t; i < 2 * kScBinsL; i += kScThreads) {
    (&sh.hl[0][0])[i] = 0u;
    (&sh.hs[0][0])[i] = 0u;
  }
  for (int i = t; i < 4 * kScBinsL; i += kScThreads) (&sh.hr[0][0])[i] = 0u;
  if (t < kScMaxCluster) {
    sh.tot[t] = 0u;
    sh.above[t] = 0u;
    sh.real[t] = 0u;
    sh.taken[t] = 0u;
  }
  if (t == 0) {
    if (CS > 1) {
      ptx::mbar_init(&sh.bar_list, static_cast<uint32_t>(CS));  // one arrival per CTA
      ptx::fence_mbarrier_init();
    }
  }
  __syncthreads();
  // zeroed before any CTA writes into them: every CTA waits on this arrival before its
  // first write into another CTA's shared memory
  bool arrived = CS > 1;
  bool done_arrived = false;  // list path: arrived after the last shared-memory exchange
  if (arrived) sc_cluster_arrive();
  ptx::pdl_wait_primary();  // the scores and the histogram come from the preceding kernels
  ptx::pdl_launch_dependents();

  const int P_raw = __ldcg(a.prefix_len + row);
  const float* srow = a.score + static_cast<size_t>(row) * a.P_max;
  const int cb = rank * kChunk;
  // The slice: group i of thread t holds positions cb + (i * 512 + t) * 4 + {0..3}.
  // Straight-line loads (no branch between them, so all are in flight at once);
  // positions past the row are clamped to its last valid entry and masked below.
  uint32_t key[NG][4];
  if ((a.P_max & 3) == 0 && a.P_max >= 4) {
    const int jmax = a.P_max - 4;
#pragma unroll
    for (int i = 0; i < NG; ++i) {
      const int j = cb + (i * kScThreads + t) * 4;
      const float4 x = __ldcg(reinterpret_cast<const float4*>(srow + (j < jmax ? j : jmax)));
      key[i][0] = sc_key(x.x);
      key[i][1] = sc_key(x.y);
      key[i][2] = sc_key(x.z);
      key[i][3] = sc_key(x.w);
    }
  } else if (a.P_max > 0) {  // rows not 16-byte aligned: scalar loads
    const int jmax = a.P_max - 1;
#pragma unroll
    for (int i = 0; i < NG; ++i) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = cb + (i * kScThreads + t) * 4 + e;
        key[i][e] = sc_key(__ldcg(srow + (j < jmax ? j : jmax)));
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < NG; ++i) key[i][0] = key[i][1] = key[i][2] = key[i][3] = 0u;
  }
  const uint32_t* hrow = a.hist + static_cast<size_t>(row) * kScBins0;
#pragma unroll
  for (int u = 0; u < kScBins0 / kScThreads; ++u)
    h0[u * kScThreads + t] = __ldcg(hrow + u * kScThreads + t);

  const bool bad_len = P_raw < 0 || P_raw > a.P_max;
  const int P = bad_len ? 0 : P_raw;
  const int n = P < a.k ? P : a.k;
  const int sink_end = a.n_sink < P ? a.n_sink : P;
  const int rb = (P - a.n_recent) > sink_end ? (P - a.n_recent) : sink_end;  // recent start
  const int n_cand = rb - sink_end;
  const int r = n - sink_end - (P - rb);  // candidates to take
  const bool thresh = r > 0 && r < n_cand;

  // rank 0: the protected part of the row and the padding (independent of the cut)
  int32_t* dst = a.idx + static_cast<size_t>(row) * a.k;
  // rank 0 also writes the protected part of the row and its padding, after the last
  // cluster release (a release would wait for these stores)
  bool protected_done = false;
  auto write_protected = [&]() {
    if (protected_done) return;
    protected_done = true;
    if (rank != 0) return;
    const int n_recent_kept = P - rb;
    for (int i = t; i < sink_end; i += kScThreads) dst[i] = i;
    for (int i = t; i < n_recent_kept; i += kScThreads) dst[n - n_recent_kept + i] = rb + i;
    for (int m = n + t; m < a.k; m += kScThreads) dst[m] = -1;
    if (t == 0) {
      a.n_sel[row] = n;
      if (bad_len) flag_status(a.status, VSD_DEV_BAD_LENGTH);
    }
  };
  __syncthreads();  // h0 copied

  // Candidate keys become >= 1, every other position 0 (never taken: the cut is >= 1).
#pragma unroll
  for (int i = 0; i < NG; ++i) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = cb + (i * kScThreads + t) * 4 + e;
      const bool cand = j >= sink_end && j < rb;
      key[i][e] = cand ? (key[i][e] > 1u ? key[i][e] : 1u) : 0u;
    }
  }

  // The cut.  List rule: taken iff key > T, or key == T at a position <= cut.
  uint32_t T = 0u;
  int cut = -1;
  int base = sink_end;  // where this CTA's taken positions start in the row
  bool take_all = r >= n_cand;
  bool levels = false;
  uint32_t b0 = 0u;
  int need = 0, cnt0 = 0;
  if (thresh) {
    sc_find_bin<true>(h0, kScBins0, static_cast<uint32_t>(r), sh);
    if (sh.f_tot != static_cast<uint32_t>(n_cand) && sh.f_tot == static_cast<uint32_t>(P)) {
      // a histogram of every prefix position (a verification call told no sink or
      // recent window): take the protected positions out, from the scores, and search
      // again
      const int n_prot = sink_end + (P - rb);
      for (int q = t; q < n_prot; q += kScThreads) {
        const int j = q < sink_end ? q : rb + (q - sink_end);
        atomicSub(&h0[sc_key(__ldcg(srow + j)) >> 20], 1u);
      }
      __syncthreads();
      sc_find_bin<true>(h0, kScBins0, static_cast<uint32_t>(r), sh);
    }
    if (sh.f_bin < 0 || sh.f_tot != static_cast<uint32_t>(n_cand)) {
      // a histogram that does not count these scores: the row is unspecified
      if (rank == 0 && t == 0) flag_status(a.status, VSD_DEV_BAD_LENGTH);
      take_all = true;
    } else {
      b0 = static_cast<uint32_t>(sh.f_bin);
      need = sh.f_rem;
      cnt0 = sh.f_cnt;
      levels = cnt0 > kScListCap;
    }
  }
  if (!thresh || take_all) {
    T = take_all ? 0u : 0xFFFFFFFFu;
    cut = -1;
    if (take_all) {  // the candidates of the slices before this one
      const int hi = rb < cb ? rb : cb;
      base += hi > sink_end ? hi - sink_end : 0;
    }
  } else if (!levels) {
    // ---- list path: every CTA gathers the boundary bin and resolves the cut itself
    uint32_t nb = 0u, na = 0u;
#pragma unroll
    for (int i = 0; i < NG; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t bin = key[i][e] >> 20;
        na += bin > b0 ? 1u : 0u;
        nb += (bin == b0 && key[i][e] != 0u) ? 1u : 0u;
      }
    uint32_t tot;
    const uint32_t off = sc_block_scan(nb | (na << 16), sh.scan, &tot);
    const uint32_t my_off = off & 0xFFFFu;
    const uint32_t n_mine = tot & 0xFFFFu;
    // CTA q's segment of every CTA's list: slots [q * segcap, (q + 1) * segcap), a
    // header (its entry count and its count above the bin) and padding, then its entries
    const uint32_t segcap = (static_cast<uint32_t>(kScListCap) / static_cast<uint32_t>(CS)) & ~1u;
    const uint32_t room = segcap - 2u;
    if (CS > 1) {
      // stage the segment (an even number of slots: 16-byte copies), then one bulk copy
      // into every CTA's list, announced on that CTA's barrier
      uint2* stage = list + kScListCap;
      uint32_t k_i = 0u;
#pragma unroll
      for (int i = 0; i < NG; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if ((key[i][e] >> 20) == b0 && key[i][e] != 0u) {
            const uint32_t slot = my_off + k_i;
            if (slot < room)
              stage[2 + slot] =
                  make_uint2(key[i][e], static_cast<uint32_t>(cb + (i * kScThreads + t) * 4 + e));
            ++k_i;
          }
        }
      const uint32_t padded = n_mine + (n_mine & 1u);
      const bool fits = padded <= room;
      if (t == 0) {
        stage[0] = make_uint2(n_mine, tot >> 16);
        stage[1] = make_uint2(0u, 0xFFFFFFFFu);
        if (fits && (n_mine & 1u)) stage[2 + n_mine] = make_uint2(0u, 0xFFFFFFFFu);
      }
      ptx::fence_proxy_async_smem();  // the staged segment, for the bulk copies
      __syncthreads();
      if (arrived) sc_cluster_wait();  // every CTA's barrier is initialised
      arrived = false;
      if (t < CS) {
        const uint32_t q = static_cast<uint32_t>(t);
        const uint32_t bytes = (fits ? 2u + padded : 2u) * 8u;  // the header at least
        const uint32_t bar = sc_peer(&sh.bar_list, q);
        sc_peer_arrive_tx(bar, bytes);
        sc_bulk_to_peer(sc_peer(list + rank * segcap, q), stage, bytes, bar);
      }
      if (!sc_wait_peers(&sh.bar_list) && t == 0) flag_status(a.status, VSD_DEV_TIMEOUT);
      if (t < CS) {
        const uint2 hd = list[t * segcap];
        sh.real[t] = hd.x;
        sh.above[t] = hd.y;
      }
      __syncthreads();
      // every copy into this CTA has landed; once all CTAs have arrived here, every copy
      // out of this CTA has landed too (waited on before exit)
      sc_cluster_arrive_relaxed();
      done_arrived = true;
      write_protected();  // no release follows: the stores need not complete before it
    } else {
      uint32_t k_i = 0u;
#pragma unroll
      for (int i = 0; i < NG; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if ((key[i][e] >> 20) == b0 && key[i][e] != 0u) {
            const uint32_t slot = my_off + k_i;
            if (slot < room)
              list[2 + slot] =
                  make_uint2(key[i][e], static_cast<uint32_t>(cb + (i * kScThreads + t) * 4 + e));
            ++k_i;
          }
        }
      if (t == 0) sh.real[0] = n_mine;
      __syncthreads();
      write_protected();
    }
    uint32_t n_real = 0u;
    bool over = false;
    for (int q = 0; q < CS; ++q) {
      n_real += sh.real[q];
      over = over || sh.real[q] + (sh.real[q] & 1u) > room;
    }
    if (n_real != static_cast<uint32_t>(cnt0)) {
      // the histogram's bin count is not the slices' (a foreign histogram)
      if (rank == 0 && t == 0) flag_status(a.status, VSD_DEV_BAD_LENGTH);
      T = 0u;
      cut = -1;
      const int hi = rb < cb ? rb : cb;
      base += hi > sink_end ? hi - sink_end : 0;
    } else if (over) {
      // one CTA holds more of the bin than its segment: the registers' route instead
      if (done_arrived) sc_cluster_wait();
      done_arrived = false;
      levels = true;
    } else {
      sc_resolve_list(list, CS, segcap, b0, need, static_cast<int>(n_real), sh, T, cut);
      if (CS > 1) {
        // warp q counts how many of CTA q's entries are taken
        const int warp = t >> 5, lane = t & 31;
        if (warp < CS) {
          const uint2* seg = list + warp * segcap + 2;
          const uint32_t n_q = sh.real[warp];
          uint32_t c = 0u;
          for (uint32_t i = lane; i < n_q; i += 32u) {
            const uint2 ent = seg[i];
            c += (ent.x > T || (ent.x == T && static_cast<int>(ent.y) <= cut)) ? 1u : 0u;
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
          if (lane == 0) sh.taken[warp] = c;
        }
        __syncthreads();
        for (int q = 0; q < rank; ++q) base += static_cast<int>(sh.above[q] + sh.taken[q]);
      }
    }
  }

  if (!levels) {
    // ---- write: taken counts in position order, then the positions
    uint32_t v[NG];
    uint64_t tm = 0ull;
#pragma unroll
    for (int i = 0; i < NG; ++i) {
      uint32_t c = 0u;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = cb + (i * kScThreads + t) * 4 + e;
        const uint32_t kk = key[i][e];
        if (kk > T || (kk == T && j <= cut)) {
          tm |= 1ull << (i * 4 + e);
          ++c;
        }
      }
      v[i] = c;
    }
    sc_group_scan<NG>(v, sh);
#pragma unroll
    for (int i = 0; i < NG; ++i) {
      int o = base + static_cast<int>(v[i]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if ((tm >> (i * 4 + e)) & 1ull) {
          if (o < n) dst[o] = cb + (i * kScThreads + t) * 4 + e;
          ++o;
        }
      }
    }
    write_protected();
    if (arrived || done_arrived) sc_cluster_wait();  // no CTA exits while peers may copy
    return;
  }

  // ---- levels path: the next key bits histogrammed over the cluster's registers
  uint32_t prefix = b0 << 20, mask = 0xFFF00000u;
  int t_need = need;
  bool whole = false;
  for (int level = 0; level < 2 && !whole; ++level) {
    const int shift = level == 0 ? 10 : 0;
#pragma unroll
    for (int i = 0; i < NG; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (key[i][e] != 0u && (key[i][e] & mask) == prefix)
          atomicAdd(&sh.hl[level][(key[i][e] >> shift) & (kScBinsL - 1)], 1u);
    __syncthreads();
    const uint32_t* sums = sh.hl[level];
    if (CS > 1) {
      cg::cluster_group cluster = cg::this_cluster();
      if (arrived) sc_cluster_wait();  // every CTA's sums are zeroed
      arrived = false;
      for (int b = t; b < kScBinsL; b += kScThreads) {
        const uint32_t c = sh.hl[level][b];
        if (c != 0u)
          for (int q = 0; q < CS; ++q) atomicAdd(cluster.map_shared_rank(&sh.hs[level][b], q), c);
      }
      sc_cluster_arrive();
      sc_cluster_wait();
      sums = sh.hs[level];
    }
    sc_find_bin<true>(sums, kScBinsL, static_cast<uint32_t>(t_need), sh);
    if (sh.f_bin < 0) {
      if (rank == 0 && t == 0) flag_status(a.status, VSD_DEV_BAD_LENGTH);
      break;  // keep the coarser cut (uniform across the cluster)
    }
    prefix |= static_cast<uint32_t>(sh.f_bin) << shift;
    mask |= static_cast<uint32_t>(kScBinsL - 1) << shift;
    t_need = sh.f_rem;
    whole = sh.f_rem == sh.f_cnt;
  }
  // keys above the cut, and keys equal to it (masked): the equal ones taken in position
  // order
  uint32_t v[NG];
#pragma unroll
  for (int i = 0; i < NG; ++i) {
    uint32_t above = 0u, eq = 0u;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (key[i][e] != 0u) {
        const uint32_t km = key[i][e] & mask;
        above += km > prefix ? 1u : 0u;
        eq += km == prefix ? 1u : 0u;
      }
    }
    v[i] = above | (eq << 16);
  }
  const uint32_t cta_tot = sc_group_scan<NG>(v, sh);
  int take_eq = t_need;  // equal keys this CTA takes (lowest positions first)
  if (CS > 1) {
    cg::cluster_group cluster = cg::this_cluster();
    if (arrived) sc_cluster_wait();
    arrived = false;
    if (t < CS) *cluster.map_shared_rank(&sh.tot[rank], t) = cta_tot;
    sc_cluster_arrive();
    sc_cluster_wait();
    long long eq_before = 0;
    for (int q = 0; q < rank; ++q) {
      const uint32_t tq = sh.tot[q];
      const long long eq_q = tq >> 16;
      long long take_q = static_cast<long long>(t_need) - eq_before;
      take_q = take_q < 0 ? 0 : (take_q > eq_q ? eq_q : take_q);
      base += static_cast<int>((tq & 0xFFFFu) + take_q);
      eq_before += eq_q;
    }
    const long long tk = static_cast<long long>(t_need) - eq_before;
    take_eq = static_cast<int>(tk < 0 ? 0 : (tk > INT_MAX ? INT_MAX : tk));
  }
#pragma unroll
  for (int i = 0; i < NG; ++i) {
    int o = base + static_cast<int>(v[i] & 0xFFFFu);
    int eq_rank = static_cast<int>(v[i] >> 16);
    o += eq_rank < take_eq ? eq_rank : take_eq;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (key[i][e] == 0u) continue;
      const uint32_t km = key[i][e] & mask;
      bool take = km > prefix;
      if (km == prefix) {
        take = eq_rank < take_eq;
        ++eq_rank;
      }
      if (take) {
        if (o < n) dst[o] = cb + (i * kScThreads + t) * 4 + e;
        ++o;
      }
    }
  }
  write_protected();
}

// float4 groups a thread holds for a row of P_max positions: the shortest slices (4K
// positions and up) that cover the row with at most 16 CTAs.  More, shorter slices
// shorten every pass over the keys; the exchange costs about the same for any width.
int scored_groups(int P_max) {
  for (int g = 2; g <= kScMaxGroups; g *= 2)
    if (P_max <= kScMaxCluster * g * 4 * kScThreads) return g;
  return kScMaxGroups;
}

template <int NG>
cudaError_t launch_ng(const ScParams& p, int CS, int n_rows, cudaStream_t stream) {
  auto kern = select_scored_kernel<NG>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kScDynBytes);
  if (e != cudaSuccess) return e;
  if (CS > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(CS), static_cast<unsigned>(n_rows), 1);
  cfg.blockDim = dim3(kScThreads, 1, 1);
  cfg.dynamicSmemBytes = kScDynBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (CS > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = static_cast<unsigned>(CS);
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

int select_scored_cluster(int P_max) {
  if (P_max < 0) return -1;
  const int chunk = scored_groups(P_max) * 4 * kScThreads;
  int cs = (P_max + chunk - 1) / chunk;
  if (cs < 1) cs = 1;
  return cs > kScMaxCluster ? -1 : cs;
}

cudaError_t launch_select_scored(const SelectArgs& sa, cudaStream_t stream) {
  if (sa.n_rows == 0) return cudaSuccess;
  const int CS = select_scored_cluster(sa.P_max);
  if (CS < 0 || sa.n_rows > 65535) return cudaErrorInvalidValue;
  ScParams p;
  p.score = sa.partial;
  p.hist = sa.hist;
  p.prefix_len = sa.prefix_len;
  p.idx = sa.idx;
  p.n_sel = sa.n_sel;
  p.status = sa.status;
  p.P_max = sa.P_max;
  p.k = sa.k;
  p.n_sink = sa.n_sink;
  p.n_recent = sa.n_recent;
  switch (scored_groups(sa.P_max)) {
    case 2: return launch_ng<2>(p, CS, sa.n_rows, stream);
    case 4: return launch_ng<4>(p, CS, sa.n_rows, stream);
    case 8: return launch_ng<8>(p, CS, sa.n_rows, stream);
    default: return launch_ng<16>(p, CS, sa.n_rows, stream);
  }
}

}  // namespace vsd
