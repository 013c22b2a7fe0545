// select_topk.cu -- aggregated-logit top-k with a protected budget on sm_103a.
//
// What it computes: the Vegas selection (technical summary sec. 2.A: the prefix set
// T with |T| = k maximising the logits summed over the collected rows and all query
// heads -- a separable objective, so the k highest scores) under the Dustin budget
// rule (Methodology sec. 1: attention sinks and the recent window are kept first,
// the rest of the budget is filled by score).  Equal scores go to the lower position;
// the output is in ascending position order.
//
// How (GB300 design): one thread-block cluster per row (layer x sequence), up to 16
// CTAs, each owning a contiguous slice of the prefix.  Each CTA
//   1. sums the per-KV-group partial scores of its slice (fp32, fixed order) and
//      keeps order-preserving uint32 keys of the candidates in shared memory;
//   2. runs an MSB-first radix select, 8 bits per pass: shared-memory histograms
//      built with warp match/ballot aggregation, summed across the cluster through
//      distributed shared memory, then a suffix scan picks the digit holding the
//      r-th largest key; a pass whose bucket is taken whole ends the search early;
//   3. compacts: selected = protected, or key above the threshold, or equal to it
//      with tie rank (in position order across the cluster) below the remainder;
//      output slots come from block scans plus the counts of lower-ranked CTAs.
// One launch covers all rows; no global workspace, no atomics on results.
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"

namespace cg = cooperative_groups;

namespace vsd {
namespace {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kMaxSelCluster = 16;
constexpr int kMaxChunk = 16384;

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
  uint32_t hist[2][256];
  uint32_t tot[256];
  uint32_t scan[kSelWarps];
  uint32_t cnt[3];  // protected, above threshold, equal to threshold (this CTA)
  int bin;
  int rrem;
  int done;
};

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum over the threads of the block, in thread order; also returns
// the block total through *total.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* scratch,
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
  if (warp == 0) {
    uint32_t w = lane < kSelWarps ? scratch[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kSelWarps) scratch[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const uint32_t warp_base = warp > 0 ? scratch[warp - 1] : 0u;
  *total = scratch[kSelWarps - 1];
  const uint32_t res = warp_base + x - v;
  __syncthreads();  // scratch is reused by the caller's next scan
  return res;
}

__global__ void __launch_bounds__(kSelThreads, 1) select_topk_kernel(const SelParams a) {
  extern __shared__ uint32_t keys[];  // [chunk]
  __shared__ SelShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int CS = static_cast<int>(cluster.num_blocks());
  const int row = blockIdx.y;
  const int t = threadIdx.x, lane = t & 31;

  int P = __ldg(a.prefix_len + row);
  if (P < 0 || P > a.P_max) {
    if (t == 0 && rank == 0) flag_status(a.status, VSD_DEV_BAD_LENGTH);
    P = 0;
  }
  const int n = a.k < P ? a.k : P;
  const int sink_end = a.n_sink < P ? a.n_sink : P;
  const int recent_begin = P - a.n_recent > 0 ? P - a.n_recent : 0;
  const int rb = recent_begin > sink_end ? recent_begin : sink_end;
  const int n_prot = sink_end + (P - rb);
  const int r_need = n - n_prot > 0 ? n - n_prot : 0;
  const int lo = rank * a.chunk;
  // candidate = unprotected prefix position
  auto is_cand = [&](int j) { return j >= sink_end && j < rb; };
  auto is_prot = [&](int j) { return j < P && (j < sink_end || j >= rb); };

  // ---- 1. aggregated scores and order-preserving keys of the slice
  for (int i = t; i < a.chunk; i += kSelThreads) {
    const int j = lo + i;
    uint32_t key = 0u;
    if (j < P) {
      float s = 0.f;
      const float* src = a.partial + static_cast<size_t>(row) * a.Hkv * a.P_max + j;
      for (int g = 0; g < a.Hkv; ++g) s += __ldg(src + static_cast<size_t>(g) * a.P_max);
      if (a.scores_out) a.scores_out[static_cast<size_t>(row) * a.P_max + j] = s;
      key = order_key(s);
    }
    keys[i] = key;
  }
  if (t < 256) {
    sh.hist[0][t] = 0u;
    sh.hist[1][t] = 0u;
  }
  __syncthreads();

  // ---- 2. radix select of the r_need-th largest candidate key
  uint32_t pv = 0u, mask = 0u;
  int r_rem = r_need;
  if (r_need > 0) {
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      uint32_t* hb = sh.hist[pass & 1];
      for (int base = 0; base < a.chunk; base += kSelThreads) {
        const int i = base + t;
        const int j = lo + i;
        bool part = false;
        uint32_t bin = 0u;
        if (i < a.chunk && is_cand(j)) {
          const uint32_t key = keys[i];
          if ((key & mask) == pv) {
            part = true;
            bin = (key >> shift) & 0xFFu;
          }
        }
        const unsigned act = __ballot_sync(0xffffffffu, part);
        if (part) {
          const unsigned same = __match_any_sync(act, bin);
          if (lane == __ffs(same) - 1) atomicAdd(&hb[bin], static_cast<uint32_t>(__popc(same)));
        }
      }
      cluster.sync();
      if (t < 256) {
        uint32_t s = 0u;
        for (int r = 0; r < CS; ++r) {
          const SelShared* other = cluster.map_shared_rank(&sh, r);
          s += other->hist[pass & 1][t];
        }
        sh.tot[t] = s;
        sh.hist[(pass + 1) & 1][t] = 0u;  // every CTA finished reading it last pass
      }
      __syncthreads();
      if (t < 256) {
        // suffix sums over bins: thread t holds bin 255 - t
        const int bidx = t >> 5;
        const uint32_t mine = sh.tot[255 - t];
        uint32_t x = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        if (lane == 31) sh.scan[bidx] = x;
        asm volatile("bar.sync 2, 256;" ::: "memory");
        uint32_t off = 0u;
        for (int w = 0; w < bidx; ++w) off += sh.scan[w];
        const uint32_t incl = off + x;
        const uint32_t gt = incl - mine;
        if (gt < static_cast<uint32_t>(r_rem) && static_cast<uint32_t>(r_rem) <= incl) {
          sh.bin = 255 - t;
          sh.rrem = r_rem - static_cast<int>(gt);
          sh.done = (mine == static_cast<uint32_t>(r_rem) - gt) ? 1 : 0;
        }
      }
      __syncthreads();
      pv |= static_cast<uint32_t>(sh.bin) << shift;
      mask |= 0xFFu << shift;
      r_rem = sh.rrem;
      const int done = sh.done;
      __syncthreads();
      if (done) break;
    }
  }

  // ---- 3. counts of this slice, exchanged across the cluster
  const int pt = (a.chunk + kSelThreads - 1) / kSelThreads;
  const int i0 = t * pt;
  const int i1 = min(i0 + pt, a.chunk);
  uint32_t cp = 0u, cgt = 0u, ceq = 0u;
  for (int i = i0; i < i1; ++i) {
    const int j = lo + i;
    if (is_prot(j)) {
      ++cp;
    } else if (j < P) {
      const uint32_t kk = keys[i] & mask;
      if (kk > pv) ++cgt;
      else if (kk == pv) ++ceq;
    }
  }
  uint32_t tot_p, tot_g, tot_e;
  const uint32_t pre_eq = block_exclusive_scan(ceq, sh.scan, &tot_e);
  (void)block_exclusive_scan(cp, sh.scan, &tot_p);
  (void)block_exclusive_scan(cgt, sh.scan, &tot_g);
  if (t == 0) {
    sh.cnt[0] = tot_p;
    sh.cnt[1] = tot_g;
    sh.cnt[2] = tot_e;
  }
  cluster.sync();
  uint32_t before_pg = 0u, eq_before = 0u;
  for (int r = 0; r < rank; ++r) {
    const SelShared* other = cluster.map_shared_rank(&sh, r);
    before_pg += other->cnt[0] + other->cnt[1];
    eq_before += other->cnt[2];
  }
  const uint32_t rr = static_cast<uint32_t>(r_rem);
  // selected positions of this thread's range, in order
  uint32_t tie = eq_before + pre_eq;
  uint32_t cs = 0u;
  for (int i = i0; i < i1; ++i) {
    const int j = lo + i;
    bool sel = false;
    if (is_prot(j)) {
      sel = true;
    } else if (j < P) {
      const uint32_t kk = keys[i] & mask;
      if (kk > pv) sel = true;
      else if (kk == pv) sel = (tie++ < rr);
    }
    cs += sel ? 1u : 0u;
  }
  uint32_t cs_total;
  const uint32_t cs_pre = block_exclusive_scan(cs, sh.scan, &cs_total);
  uint32_t out = before_pg + (eq_before < rr ? eq_before : rr) + cs_pre;
  tie = eq_before + pre_eq;
  int32_t* dst = a.idx + static_cast<size_t>(row) * a.k;
  for (int i = i0; i < i1; ++i) {
    const int j = lo + i;
    bool sel = false;
    if (is_prot(j)) {
      sel = true;
    } else if (j < P) {
      const uint32_t kk = keys[i] & mask;
      if (kk > pv) sel = true;
      else if (kk == pv) sel = (tie++ < rr);
    }
    if (sel) {
      if (out < static_cast<uint32_t>(n)) dst[out] = j;
      ++out;
    }
  }
  // unused slots and the count
  for (int m = n + rank * kSelThreads + t; m < a.k; m += CS * kSelThreads) dst[m] = -1;
  if (rank == 0 && t == 0) a.n_sel[row] = n;
  cluster.sync();  // keep shared memory alive until every CTA has read the counts
}

}  // namespace

int select_cluster_size(int P_max) {
  int cs = (P_max + 2047) / 2048;
  if (cs < 1) cs = 1;
  if (cs > kMaxSelCluster) cs = kMaxSelCluster;
  while ((P_max + cs - 1) / cs > kMaxChunk) return -1;  // slice does not fit
  return cs;
}

cudaError_t launch_select(const SelectArgs& sa, cudaStream_t stream) {
  if (sa.n_rows == 0) return cudaSuccess;
  const int CS = select_cluster_size(sa.P_max);
  if (CS < 1) return cudaErrorInvalidValue;
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
  p.chunk = (sa.P_max + CS - 1) / CS;
  if (p.chunk < 1) p.chunk = 1;
  const size_t smem = static_cast<size_t>(p.chunk) * sizeof(uint32_t);
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
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, select_topk_kernel, p);
}

}  // namespace vsd
