// sparse_decode.cu -- sparse draft-step attention on sm_103a.
//
// What it computes ("Vegas" technical summary, sec. 2 drafting phase and sec. 3
// sparse execution): one query row per head attends only the selected positions
// (paged attention with page size 1 whose page indices are the selected token
// indices) plus the tokens appended after the selection (dense tail).
//
// How (GB300 design).  The step moves a few MB to tens of MB of randomly placed
// 256-byte rows; at one sequence it is bound by the latency of its dependent loads
// (index -> block table -> K and V rows), at large batches by how many gathers stay in
// flight.  The attended list of one (sequence, KV head) pair, idx[0 .. n_sel) followed
// by [tail_start, seq_len), is cut into splits of 128 positions (more per split only
// when the list is very long).  A pair with a single split writes its output directly;
// otherwise each split writes (m, l, o) to the workspace and the pair's last split (a
// per-pair counter in the workspace, reset to zero by that split) combines them, every
// load of a round in flight at once, in split order.  Results are bit-reproducible;
// the only atomics are the counters.  Three kernels:
//   * sparse_tc_kernel (splits of one 128-position batch, the common case): one split
//     per CTA of four warps on the 5th-generation tensor cores (below); one CTA per SM
//     when the splits fit one wave, three per SM otherwise.
//   * sparse_ws_kernel (more splits than one wave of it holds): persistent CTAs with a
//     producer warpgroup gathering into three stages and two consumer warpgroups
//     running the same tensor-core steps (below).
//   * sparse_decode_kernel (splits longer than one batch: lists beyond 1024 batches),
//     on the CUDA cores: sixteen warps of 8 positions for up to 4 query heads per KV
//     head, eight warps of 16 beyond; a row of K or V is read by head_dim/8 adjacent
//     lanes, 16 bytes each, all of a warp's loads in flight together (the first index
//     loads issued speculatively, before the list lengths are known); each lane forms
//     partial dot products of its 8 dims with the G queries of the group (fp32, q in
//     shared memory), a shuffle tree over the row's lanes completes the logits, the
//     warp softmax and the P.V product on the lane's 8 dims follow in registers, and
//     the warps merge in shared memory in a fixed order.
#include <cfloat>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace vsd {
namespace {

constexpr int kBatch = 128;  // positions per CTA per batch

// Warps per CTA and keys per warp for G query heads per KV head: sixteen warps of 8
// keys while a warp's G * 8 accumulators leave room (512 threads get 128 registers
// each), eight warps of 16 keys beyond.
template <int G>
struct SCfg {
  static constexpr int kWarps = G <= 4 ? 16 : 8;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kKeysPerWarp = kBatch / kWarps;
};
constexpr int kPageS = 16;
constexpr int kMaxSplits = 1024;

struct SParams {
  const uint16_t* q;
  const uint16_t* k_cache;
  const uint16_t* v_cache;
  const int32_t* block_table;
  const int32_t* idx;
  const int32_t* n_sel;
  const int32_t* tail_start;
  const int32_t* seq_len;
  uint16_t* out;
  float* ws;
  unsigned* counters;  // per pair: splits that have written their partial
  unsigned* status;
  int Hq, Hkv, max_blocks, num_blocks, k_max;
  int split_len;   // positions per split (a multiple of kBatch)
  int max_splits;  // workspace slots per pair
  float scale_log2;
};

// Thread layout of one warp's batch for head dimension D: a K / V row is read by
// LPR = D / 8 lanes (8 dims = 16 bytes each), one instruction covers KPI = 32 / LPR
// rows, and the warp's keys take U = keys / KPI instructions ("slots").
template <int D, int G>
struct SLayout {
  static constexpr int LPR = D / 8;
  static constexpr int KPI = 32 / LPR;
  static constexpr int U = SCfg<G>::kKeysPerWarp / KPI;
};

template <int D, int G>
struct SSmem {
  float q[G][D];
  float wm[SCfg<G>::kWarps][G];
  float wl[SCfg<G>::kWarps][G];
  union {
    float wo[SCfg<G>::kWarps][G][D];
    float merge_scratch[SCfg<G>::kThreads * 6];  // m, l and a float4 o per thread
  };
};

// The attended list of sequence b (false lengths: an empty list, flagged).
struct SList {
  int ns, t0, total;
};

__device__ __forceinline__ SList attended_list(int ns, int t0, int t1, const SParams& a,
                                               bool flag) {
  SList L;
  // the list must fit the launch's splits: a tail longer than the declared max_tail
  // is refused (flagged, nothing attended) rather than partly dropped
  const bool ok = ns >= 0 && ns <= a.k_max && t0 >= 0 && t0 <= t1 &&
                  static_cast<long long>(t1) <= static_cast<long long>(a.max_blocks) * kPageS &&
                  static_cast<long long>(ns) + (t1 - t0) <=
                      static_cast<long long>(a.split_len) * a.max_splits;
  if (!ok && flag) flag_status(a.status, VSD_DEV_BAD_LENGTH);
  L.ns = ok ? ns : 0;
  L.t0 = t0;
  L.total = ok ? ns + (t1 - t0) : 0;
  return L;
}

// One split's partial (m, l, o) in the workspace: the G heads' running max and sum,
// padded so that the G output rows (read as float4 by the merge) start on a 16-byte
// boundary, then the rows.
template <int D, int G>
struct SSlot {
  static constexpr int kO = (2 * G + 3) / 4 * 4;  // floats before the output rows
  static constexpr int kFloats = kO + G * D;
  static_assert(kFloats % 4 == 0 && D % 4 == 0, "16-byte slots");
};

// Combine the n partial (m, l, o) of one pair's splits and write its G output rows.
// Thread t of the kSThreads that run it (`sync` is their barrier) = (float4 group of
// (head, dims), part); part p takes splits p, p + kParts, ... with all loads of a round
// in flight; the parts then combine in shared memory.
// kRound: splits per load round when a thread holds one output group.
template <int D, int G, int kSThreads, int kRound, typename Sync>
__device__ __forceinline__ void merge_splits_by(const SParams& a, float* scratch, int pair, int b,
                                                int g, int n, const int t, Sync sync) {
  constexpr int kQ = D / 4;
  constexpr int NG = G * kQ;                              // float4 groups of the output
  constexpr int kGPT = NG > kSThreads ? NG / kSThreads : 1;  // groups per thread
  constexpr int kParts = NG >= kSThreads ? 1 : kSThreads / NG;
  constexpr int kU = kGPT == 1 ? kRound : (16 / kGPT > 1 ? 16 / kGPT : 1);  // per load round
  static_assert(NG * kParts / kGPT == kSThreads || NG >= kSThreads, "merge layout");
  const int part = kParts > 1 ? t / NG : 0;
  const size_t stride = SSlot<D, G>::kFloats;
  const float* base = a.ws + static_cast<size_t>(pair) * a.max_splits * stride;
  float M[kGPT], L[kGPT];
  float4 O[kGPT];
#pragma unroll
  for (int i = 0; i < kGPT; ++i) {
    M[i] = -INFINITY;
    L[i] = 0.f;
    O[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int k0 = part; k0 < n; k0 += kU * kParts) {
    float mk[kGPT][kU], lk[kGPT][kU];
    float4 ok[kGPT][kU];
#pragma unroll
    for (int i = 0; i < kGPT; ++i) {
      const int gi = (kParts > 1 ? t % NG : t) + i * kSThreads;
      const int hh = gi / kQ, q4 = gi % kQ;
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int k = k0 + u * kParts;
        if (k < n) {
          const float* sl = base + k * stride;
          mk[i][u] = __ldcg(sl + hh);
          lk[i][u] = __ldcg(sl + G + hh);
          ok[i][u] = __ldcg(reinterpret_cast<const float4*>(sl + SSlot<D, G>::kO + hh * D) + q4);
        } else {
          mk[i][u] = -INFINITY;
          lk[i][u] = 0.f;
          ok[i][u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kGPT; ++i) {
      float mn = M[i];
#pragma unroll
      for (int u = 0; u < kU; ++u) mn = fmaxf(mn, mk[i][u]);
      const float sc = (M[i] == -INFINITY) ? 0.f : exp2f(M[i] - mn);
      L[i] *= sc;
      O[i].x *= sc;
      O[i].y *= sc;
      O[i].z *= sc;
      O[i].w *= sc;
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const float w = (mk[i][u] == -INFINITY) ? 0.f : exp2f(mk[i][u] - mn);
        L[i] += w * lk[i][u];
        O[i].x += w * ok[i][u].x;
        O[i].y += w * ok[i][u].y;
        O[i].z += w * ok[i][u].z;
        O[i].w += w * ok[i][u].w;
      }
      M[i] = mn;
    }
  }
  if constexpr (kParts > 1) {
    // parts meet in shared memory: [part][group] of m, l and the float4 o
    float* pm = scratch;  // kSThreads * 6 floats
    float* pl = pm + kParts * NG;
    float4* po = reinterpret_cast<float4*>(pl + kParts * NG);
    const int gi = t % NG;
    pm[part * NG + gi] = M[0];
    pl[part * NG + gi] = L[0];
    po[part * NG + gi] = O[0];
    sync();
    if (part == 0) {
      float mn = -INFINITY;
#pragma unroll
      for (int r = 0; r < kParts; ++r) mn = fmaxf(mn, pm[r * NG + gi]);
      float Lt = 0.f;
      float4 Ot = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int r = 0; r < kParts; ++r) {
        const float mr = pm[r * NG + gi];
        const float w = (mr == -INFINITY) ? 0.f : exp2f(mr - mn);
        const float4 o = po[r * NG + gi];
        Lt += w * pl[r * NG + gi];
        Ot.x += w * o.x;
        Ot.y += w * o.y;
        Ot.z += w * o.z;
        Ot.w += w * o.w;
      }
      L[0] = Lt;
      O[0] = Ot;
    }
    if (part != 0) return;
  }
#pragma unroll
  for (int i = 0; i < kGPT; ++i) {
    const int gi = (kParts > 1 ? t % NG : t) + i * kSThreads;
    const int hh = gi / kQ, q4 = gi % kQ;
    const float inv = L[i] > 0.f ? 1.f / L[i] : 0.f;
    uint2 pk;
    pk.x = pack_bf16x2(O[i].x * inv, O[i].y * inv);
    pk.y = pack_bf16x2(O[i].z * inv, O[i].w * inv);
    *reinterpret_cast<uint2*>(a.out + (static_cast<size_t>(b) * a.Hq + g * G + hh) * D +
                              q4 * 4) = pk;
  }
}

template <int D, int G, int kSThreads, int kRound = 16>
__device__ __forceinline__ void merge_splits(const SParams& a, float* scratch, int pair, int b,
                                             int g, int n) {
  merge_splits_by<D, G, kSThreads, kRound>(a, scratch, pair, b, g, n,
                                           static_cast<int>(threadIdx.x),
                                           [] { __syncthreads(); });
}

template <int D, int G>
__global__ void __launch_bounds__(SCfg<G>::kThreads, 1) sparse_decode_kernel(const SParams a) {
  constexpr int kSWarps = SCfg<G>::kWarps, kSThreads = SCfg<G>::kThreads;
  constexpr int kKeysPerWarp = SCfg<G>::kKeysPerWarp;
  using Lay = SLayout<D, G>;
  constexpr int LPR = Lay::LPR, KPI = Lay::KPI, U = Lay::U;
  extern __shared__ __align__(16) uint8_t sparse_smem[];
  SSmem<D, G>& sm = *reinterpret_cast<SSmem<D, G>*>(sparse_smem);
  const int split = blockIdx.x;
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / LPR;  // which row of an instruction
  const int lr = lane % LPR;   // which 8 dims of the row

  ptx::pdl_launch_dependents();  // the next kernel on the stream may become resident
  ptx::pdl_wait_primary();       // idx / n_sel come from the preceding kernel

  // First round of loads, independent of one another: the list lengths, the first
  // batch's indices (speculatively: used only for positions that turn out to be
  // selected ones) and the queries.
  const int lo = split * a.split_len;
  const int wbase0 = lo + warp * kKeysPerWarp;
  int j_spec[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int pos = wbase0 + u * KPI + sub;
    j_spec[u] = (a.idx != nullptr && pos < a.k_max)
                    ? __ldg(a.idx + static_cast<size_t>(b) * a.k_max + pos)
                    : 0;
  }
  constexpr int kQLoads = (G * D / 8 + kSThreads - 1) / kSThreads;
  uint4 qraw[kQLoads];
#pragma unroll
  for (int u = 0; u < kQLoads; ++u) {
    const int i = threadIdx.x + u * kSThreads;
    if (i < G * D / 8) {
      const int hh = i / (D / 8), c8 = i % (D / 8);
      qraw[u] = *reinterpret_cast<const uint4*>(
          a.q + (static_cast<size_t>(b) * a.Hq + g * G + hh) * D + c8 * 8);
    }
  }
  const int ns_raw = a.n_sel != nullptr ? __ldg(a.n_sel + b) : 0;
  const int t0_raw = __ldg(a.tail_start + b);
  const int t1 = __ldg(a.seq_len + b);
  const SList L = attended_list(ns_raw, t0_raw, t1, a, split == 0 && g == 0 && threadIdx.x == 0);
  if (lo >= L.total && !(split == 0 && L.total == 0)) return;  // no work in this split
  const int hi = min(lo + a.split_len, L.total);
  const int n_splits = (L.total + a.split_len - 1) / a.split_len;

#pragma unroll
  for (int u = 0; u < kQLoads; ++u) {
    const int i = threadIdx.x + u * kSThreads;
    if (i < G * D / 8) {
      const int hh = i / (D / 8), c8 = i % (D / 8);
      const uint4 raw = qraw[u];
      float4 lo4, hi4;
      lo4.x = bf16_lo(raw.x);
      lo4.y = bf16_hi(raw.x);
      lo4.z = bf16_lo(raw.y);
      lo4.w = bf16_hi(raw.y);
      hi4.x = bf16_lo(raw.z);
      hi4.y = bf16_hi(raw.z);
      hi4.z = bf16_lo(raw.w);
      hi4.w = bf16_hi(raw.w);
      *reinterpret_cast<float4*>(&sm.q[hh][c8 * 8]) = lo4;
      *reinterpret_cast<float4*>(&sm.q[hh][c8 * 8 + 4]) = hi4;
    }
  }
  __syncthreads();

  float m[G], lsum[G], acc[G][8];
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    m[hh] = -INFINITY;
    lsum[hh] = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[hh][e] = 0.f;
  }

  for (int wbase = wbase0; wbase < hi; wbase += kBatch) {
    // ---- list position -> token -> cache row, for each slot of this lane's row group
    int row[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int pos = wbase + u * KPI + sub;
      row[u] = -1;
      if (pos < hi) {
        const int j = pos >= L.ns ? L.t0 + (pos - L.ns)
                      : wbase == wbase0 ? j_spec[u]
                                        : __ldg(a.idx + static_cast<size_t>(b) * a.k_max + pos);
        if (j < 0 || j >= t1) {
          if (lr == 0) flag_status(a.status, VSD_DEV_BAD_INDEX);
        } else {
          const int blk =
              __ldg(a.block_table + static_cast<size_t>(b) * a.max_blocks + j / kPageS);
          if (blk < 0 || blk >= a.num_blocks) {
            if (lr == 0) flag_status(a.status, VSD_DEV_BAD_BLOCK);
          } else {
            row[u] = (blk * a.Hkv + g) * kPageS + (j % kPageS);
          }
        }
      }
    }
    // ---- every K and V load of the batch in flight: 16 bytes of each row per lane
    uint4 kr[U], vr[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (row[u] >= 0) {
        const size_t off = static_cast<size_t>(row[u]) * D + lr * 8;
        kr[u] = ldg_stream16(a.k_cache + off);
        vr[u] = ldg_stream16(a.v_cache + off);
      } else {
        kr[u] = make_uint4(0, 0, 0, 0);
        vr[u] = make_uint4(0, 0, 0, 0);
      }
    }
    // ---- logits: partial dot products of the lane's 8 dims, completed over the row
    float z[U][G];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float kf[8];
      kf[0] = bf16_lo(kr[u].x); kf[1] = bf16_hi(kr[u].x);
      kf[2] = bf16_lo(kr[u].y); kf[3] = bf16_hi(kr[u].y);
      kf[4] = bf16_lo(kr[u].z); kf[5] = bf16_hi(kr[u].z);
      kf[6] = bf16_lo(kr[u].w); kf[7] = bf16_hi(kr[u].w);
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        const float4 qa = *reinterpret_cast<const float4*>(&sm.q[hh][lr * 8]);
        const float4 qb = *reinterpret_cast<const float4*>(&sm.q[hh][lr * 8 + 4]);
        float s = qa.x * kf[0];
        s = fmaf(qa.y, kf[1], s); s = fmaf(qa.z, kf[2], s); s = fmaf(qa.w, kf[3], s);
        s = fmaf(qb.x, kf[4], s); s = fmaf(qb.y, kf[5], s);
        s = fmaf(qb.z, kf[6], s); s = fmaf(qb.w, kf[7], s);
        z[u][hh] = s;
      }
    }
#pragma unroll
    for (int o = 1; o < LPR; o <<= 1)
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int hh = 0; hh < G; ++hh) z[u][hh] += __shfl_xor_sync(0xffffffffu, z[u][hh], o);
    // ---- online softmax over the warp's keys (slots x row groups)
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      float bm = -INFINITY;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        z[u][hh] = row[u] >= 0 ? z[u][hh] * a.scale_log2 : -INFINITY;
        bm = fmaxf(bm, z[u][hh]);
      }
#pragma unroll
      for (int o = LPR; o < 32; o <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
      const float mn = fmaxf(m[hh], bm);
      const float alpha = (m[hh] == -INFINITY) ? 0.f : exp2f(m[hh] - mn);
      float ps = 0.f;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float p = (z[u][hh] == -INFINITY) ? 0.f : exp2f(z[u][hh] - mn);
        z[u][hh] = p;
        ps += p;
      }
      lsum[hh] = lsum[hh] * alpha + ps;  // this row group's keys; groups combine at the end
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[hh][e] *= alpha;
      m[hh] = mn;
    }
    // ---- P.V on the lane's 8 dims
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float vf[8];
      vf[0] = bf16_lo(vr[u].x); vf[1] = bf16_hi(vr[u].x);
      vf[2] = bf16_lo(vr[u].y); vf[3] = bf16_hi(vr[u].y);
      vf[4] = bf16_lo(vr[u].z); vf[5] = bf16_hi(vr[u].z);
      vf[6] = bf16_lo(vr[u].w); vf[7] = bf16_hi(vr[u].w);
#pragma unroll
      for (int hh = 0; hh < G; ++hh)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[hh][e] = fmaf(z[u][hh], vf[e], acc[hh][e]);
    }
  }
  // the row groups of the warp hold disjoint keys: add them up
#pragma unroll
  for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      lsum[hh] += __shfl_xor_sync(0xffffffffu, lsum[hh], o);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[hh][e] += __shfl_xor_sync(0xffffffffu, acc[hh][e], o);
    }

  // ---- merge the warps in a fixed order
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    if (lane == 0) {
      sm.wm[warp][hh] = m[hh];
      sm.wl[warp][hh] = lsum[hh];
    }
    if (sub == 0) {
      *reinterpret_cast<float4*>(&sm.wo[warp][hh][lr * 8]) =
          make_float4(acc[hh][0], acc[hh][1], acc[hh][2], acc[hh][3]);
      *reinterpret_cast<float4*>(&sm.wo[warp][hh][lr * 8 + 4]) =
          make_float4(acc[hh][4], acc[hh][5], acc[hh][6], acc[hh][7]);
    }
  }
  __syncthreads();
  const bool direct = n_splits <= 1;
  const int pair = b * a.Hkv + g;
  const size_t slot = static_cast<size_t>(pair) * a.max_splits + split;
  float* wsl = direct ? nullptr : a.ws + slot * SSlot<D, G>::kFloats;
  for (int i = threadIdx.x; i < G * D; i += kSThreads) {
    const int hh = i / D, dim = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kSWarps; ++w) M = fmaxf(M, sm.wm[w][hh]);
    float Lh = 0.f, o = 0.f;
#pragma unroll
    for (int w = 0; w < kSWarps; ++w) {
      const float mw = sm.wm[w][hh];
      const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
      Lh += f * sm.wl[w][hh];
      o += f * sm.wo[w][hh][dim];
    }
    if (direct) {
      const float val = Lh > 0.f ? o / Lh : 0.f;
      const __nv_bfloat16 bv = __float2bfloat16_rn(val);
      a.out[(static_cast<size_t>(b) * a.Hq + g * G + hh) * D + dim] =
          *reinterpret_cast<const uint16_t*>(&bv);
    } else {
      wsl[SSlot<D, G>::kO + hh * D + dim] = o;
      if (dim == 0) {
        wsl[hh] = M;
        wsl[G + hh] = Lh;
      }
    }
  }
  if (direct) return;
  // The last split of the pair to get here combines them all.  The CTA barrier orders
  // every thread's partial stores before thread 0's acquire-release count, which
  // publishes them GPU-wide; the last counter (acquire) sees every other split's, and
  // the barrier after it extends that to the whole CTA.  The counter goes back to
  // zero for the next call.
  __shared__ int s_last;
  __syncthreads();  // also: every thread is done reading sm.wo
  if (threadIdx.x == 0) {
    const unsigned old = ptx::atom_add_acq_rel_gpu(a.counters + pair, 1u);
    const int last = old == static_cast<unsigned>(n_splits - 1);
    if (last) ptx::st_relaxed_gpu(a.counters + pair, 0u);
    s_last = last;
  }
  __syncthreads();
  if (!s_last) return;
  merge_splits<D, G, kSThreads>(a, sm.merge_scratch, pair, b, g, n_splits);
}

// ---------------------------------------------------------------- tensor-core step
// One split of up to 128 attended positions of one (sequence, KV head) pair per CTA of
// four warps, on the 5th-generation tensor cores:
//   * every thread resolves one position (index or tail -> block table -> cache row);
//     the CTA then gathers the 128 K and V rows with 16-byte asynchronous copies, one
//     instruction covering whole rows, straight into the 128-byte-swizzled K-major
//     layout the MMA reads (absent rows are zero-filled), and stages the G query rows
//     (padded to 16) the same way;
//   * one thread issues S^T = K Q^T (M = 128 keys, N = 16, K = head_dim) into TMEM;
//   * thread t owns key t (TMEM lane t): it reads its 16 logits, the CTA forms the
//     per-head max and sum in shared memory, and the thread writes its probabilities
//     as row t of P^T (bf16, swizzled);
//   * one thread issues O^T = V^T P^T (M = 128 >= head_dim, N = 16, K = 128 keys) into TMEM;
//     thread d < head_dim reads dimension d of the G heads and writes the output, or the
//     split's (m, l, o) for the last-split merge shared with the CUDA-core kernel.
constexpr int kTcThreads = 128;
constexpr int kTcNQ = 16;  // MMA N: query heads of the group, padded

template <int D>
struct TcSmem {
  static constexpr int kHalf = kBatch * 128;       // one 64-column half of a K/V tile
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kBatch * D * 2;
  static constexpr int kOffQ = kOffV + kBatch * D * 2;
  static constexpr int kOffRed = kOffQ + (kTcNQ * D * 2 < 2048 ? 2048 : kTcNQ * D * 2);
  static constexpr int kOffBar = kOffRed + 2 * 4 * kTcNQ * 4;  // after [2][4][16] floats
  // P^T reuses the K tile (its QK MMA has completed before P^T is written) and the
  // merge scratch the V tile (after the PV MMA); the PV MMA reads 128 rows of V^T,
  // which for D = 64 run 16 KB past the V tile, still inside this allocation
  static constexpr int kOffP = kOffK;
  static constexpr int kOffScratch = kOffV;
  static constexpr int kUsed = kOffBar + 64 > kOffV + 2 * kHalf ? kOffBar + 64 : kOffV + 2 * kHalf;
  static constexpr int kBytes = kUsed + 1024;  // + alignment slack
  static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0, "swizzle atoms need 1 KB alignment");
  static_assert(kBatch * 128 <= kOffV - kOffK, "P^T fits in the K tile");
  static_assert(kTcThreads * 6 * 4 <= kBatch * D * 2, "merge scratch fits in the V tile");
};

template <int D, int G>
__global__ void __launch_bounds__(kTcThreads) sparse_tc_kernel(const SParams a) {
  using Sm = TcSmem<D>;
  constexpr int LPR = D / 8;        // 16-byte chunks per row
  constexpr int RPI = 32 / LPR;     // rows per warp instruction
  constexpr int QPT = kTcNQ * LPR / kTcThreads;  // query chunks per thread
  static_assert(kTcNQ * LPR % kTcThreads == 0, "query staging");
  extern __shared__ uint8_t tc_smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* k_s = base + Sm::kOffK;
  uint8_t* v_s = base + Sm::kOffV;
  uint8_t* q_s = base + Sm::kOffQ;
  uint8_t* p_s = base + Sm::kOffP;
  float* red = reinterpret_cast<float*>(base + Sm::kOffRed);
  float* scratch = reinterpret_cast<float*>(base + Sm::kOffScratch);
  uint64_t* bar_s = reinterpret_cast<uint64_t*>(base + Sm::kOffBar);
  uint64_t* bar_o = bar_s + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_s + 2);
  __shared__ int s_last;

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  if (t == 0) {
    ptx::mbar_init(bar_s, 1);
    ptx::mbar_init(bar_o, 1);
    ptx::fence_mbarrier_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(tmem_slot, 32);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;  // S^T: columns [0, 16); O^T: columns [16, 32)
  ptx::pdl_launch_dependents();
  ptx::pdl_wait_primary();  // idx / n_sel come from the preceding kernel

  // this thread's index is loaded together with the list lengths (every position
  // below k_max is valid memory; it is used only if the position is a selected one)
  const int lo = split * a.split_len;
  const int j_spec = (a.idx != nullptr && lo + t < a.k_max)
                         ? __ldg(a.idx + static_cast<size_t>(b) * a.k_max + lo + t)
                         : 0;
  const int ns_raw = a.n_sel != nullptr ? __ldg(a.n_sel + b) : 0;
  const int t0_raw = __ldg(a.tail_start + b);
  const int t1 = __ldg(a.seq_len + b);
  uint4 qv[QPT];
#pragma unroll
  for (int u = 0; u < QPT; ++u) {
    const int i = t + u * kTcThreads, r = i / LPR, c = i % LPR;
    qv[u] = make_uint4(0, 0, 0, 0);
    if (r < G)
      qv[u] = *reinterpret_cast<const uint4*>(a.q + (static_cast<size_t>(b) * a.Hq + g * G + r) * D +
                                              c * 8);
  }
  const SList L = attended_list(ns_raw, t0_raw, t1, a, split == 0 && g == 0 && t == 0);
  const bool work = lo < L.total || (split == 0 && L.total == 0);
  const int n_splits = (L.total + a.split_len - 1) / a.split_len;
  const bool direct = n_splits <= 1;
  const int pair = b * a.Hkv + g;
  bool timed_out = false;

  if (work) {
    // ---- this thread's position -> cache row (-1: absent, zero-filled)
    const int pos = lo + t;
    int crow = -1;
    if (pos < L.total && pos < lo + kBatch) {
      const int j = pos >= L.ns ? L.t0 + (pos - L.ns) : j_spec;
      if (j < 0 || j >= t1) {
        flag_status(a.status, VSD_DEV_BAD_INDEX);
      } else {
        const int blk = __ldg(a.block_table + static_cast<size_t>(b) * a.max_blocks + j / kPageS);
        if (blk < 0 || blk >= a.num_blocks)
          flag_status(a.status, VSD_DEV_BAD_BLOCK);
        else
          crow = (blk * a.Hkv + g) * kPageS + (j % kPageS);
      }
    }
    // ---- gather: warp w copies rows 32 w .. 32 w + 31, RPI whole rows per instruction
    const int ch = lane % LPR;
#pragma unroll
    for (int u = 0; u < 32 / RPI; ++u) {
      const int rl = u * RPI + lane / LPR;  // row within the warp
      const int r = warp * 32 + rl;
      const int cr = __shfl_sync(0xffffffffu, crow, rl);
      const size_t src = cr >= 0 ? static_cast<size_t>(cr) * D + ch * 8 : 0;
      const int off = (ch >> 3) * Sm::kHalf + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
      ptx::cp_async16(k_s + off, a.k_cache + src, cr >= 0 ? 16u : 0u);
      ptx::cp_async16(v_s + off, a.v_cache + src, cr >= 0 ? 16u : 0u);
    }
    ptx::cp_async_commit();
    // ---- the group's query rows (loaded with the indices), padded with zeros to 16
#pragma unroll
    for (int u = 0; u < QPT; ++u) {
      const int i = t + u * kTcThreads, r = i / LPR, c = i % LPR;
      *reinterpret_cast<uint4*>(q_s + (c >> 3) * (kTcNQ * 128) + r * 128 +
                                (((c & 7) ^ (r & 7)) << 4)) = qv[u];
    }
    ptx::cp_async_wait_all();
    ptx::fence_proxy_async_smem();  // make the copies and stores visible to the tensor cores
    __syncthreads();

    // ---- S^T = K Q^T
    if (t == 0) {
      ptx::tc_fence_after();
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(128, kTcNQ, 0, 0);
      const uint32_t ka = ptx::smem_u32(k_s), qa = ptx::smem_u32(q_s);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int hh = kk >> 2, w = kk & 3;
        const uint64_t ad = ptx::sdesc_sw128(ka + hh * Sm::kHalf + w * 32, 16, 1024);
        const uint64_t bd = ptx::sdesc_sw128(qa + hh * kTcNQ * 128 + w * 32, 16, 1024);
        ptx::umma_bf16(tmem, ad, bd, idesc, kk > 0 ? 1u : 0u);
      }
      ptx::umma_commit(bar_s);
    }
    if (!ptx::mbar_wait(bar_s, 0)) timed_out = true;
    ptx::tc_fence_after();
    float sv[kTcNQ];
    ptx::tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16), reinterpret_cast<uint32_t(&)[16]>(sv));
    ptx::tmem_wait_ld();
    // ---- softmax over the CTA's keys, per head (log2 units)
    const bool valid = crow >= 0;
    float z[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      z[h] = valid ? sv[h] * a.scale_log2 : -INFINITY;
      float mx = z[h];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      if (lane == 0) red[warp * kTcNQ + h] = mx;
    }
    __syncthreads();
    float m[G], psum[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = fmaxf(fmaxf(red[h], red[kTcNQ + h]), fmaxf(red[2 * kTcNQ + h], red[3 * kTcNQ + h]));
      const float p = (z[h] == -INFINITY) ? 0.f : exp2f(z[h] - m[h]);
      z[h] = p;
      float sp = p;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sp += __shfl_xor_sync(0xffffffffu, sp, o);
      if (lane == 0) red[4 * kTcNQ + warp * kTcNQ + h] = sp;
    }
    // row t of P^T: 16 bf16 (heads >= G are zero) in two swizzled 16-byte chunks
    float pr[kTcNQ];
#pragma unroll
    for (int c = 0; c < kTcNQ; ++c) pr[c] = c < G ? z[c < G ? c : 0] : 0.f;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      uint4 pk;
      pk.x = pack_bf16x2(pr[k * 8 + 0], pr[k * 8 + 1]);
      pk.y = pack_bf16x2(pr[k * 8 + 2], pr[k * 8 + 3]);
      pk.z = pack_bf16x2(pr[k * 8 + 4], pr[k * 8 + 5]);
      pk.w = pack_bf16x2(pr[k * 8 + 6], pr[k * 8 + 7]);
      *reinterpret_cast<uint4*>(p_s + t * 128 + ((k ^ (t & 7)) << 4)) = pk;
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();
#pragma unroll
    for (int h = 0; h < G; ++h)
      psum[h] = red[4 * kTcNQ + h] + red[5 * kTcNQ + h] + red[6 * kTcNQ + h] + red[7 * kTcNQ + h];

    // ---- O^T = V^T P^T
    if (t == 0) {
      ptx::tc_fence_after();
      // M = 128 for either head dimension: with D = 64 the upper 64 rows of A are the
      // next 16 KB of this CTA's shared memory and land in TMEM lanes 64-127, never read
      // (the M = 64 shape keeps its rows in a different TMEM lane layout)
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(128, kTcNQ, 1, 1);
      const uint32_t va = ptx::smem_u32(v_s), pa = ptx::smem_u32(p_s);
#pragma unroll
      for (int kk = 0; kk < kBatch / 16; ++kk) {
        const uint64_t ad = ptx::sdesc_sw128(va + kk * 2048, Sm::kHalf, 1024);
        const uint64_t bd = ptx::sdesc_sw128(pa + kk * 2048, Sm::kHalf, 1024);
        ptx::umma_bf16(tmem + 16, ad, bd, idesc, kk > 0 ? 1u : 0u);
      }
      ptx::umma_commit(bar_o);
    }
    if (!ptx::mbar_wait(bar_o, 0)) timed_out = true;
    ptx::tc_fence_after();
    if (warp < D / 32) {  // TMEM lanes 0 .. D-1 hold the output dimensions
      float o[kTcNQ];
      ptx::tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + 16,
                     reinterpret_cast<uint32_t(&)[16]>(o));
      ptx::tmem_wait_ld();
      const int dim = t;
      if (direct) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float val = psum[h] > 0.f ? o[h] / psum[h] : 0.f;
          const __nv_bfloat16 bv = __float2bfloat16_rn(val);
          a.out[(static_cast<size_t>(b) * a.Hq + g * G + h) * D + dim] =
              *reinterpret_cast<const uint16_t*>(&bv);
        }
      } else {
        float* wsl = a.ws + (static_cast<size_t>(pair) * a.max_splits + split) * SSlot<D, G>::kFloats;
#pragma unroll
        for (int h = 0; h < G; ++h) wsl[SSlot<D, G>::kO + h * D + dim] = o[h];
        if (dim < G) {
          // m and l of head `dim` (every thread holds all heads' values)
#pragma unroll
          for (int h = 0; h < G; ++h) {
            if (h == dim) {
              wsl[h] = m[h];
              wsl[G + h] = psum[h];
            }
          }
        }
      }
    }
    if (timed_out) flag_status(a.status, VSD_DEV_TIMEOUT);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 32);
  }
  if (!work || direct) return;
  // The last split of the pair to get here combines them all (as in the CUDA-core
  // kernel: the barrier above orders every thread's partial stores before thread 0's
  // acquire-release count).
  if (t == 0) {
    const unsigned old = ptx::atom_add_acq_rel_gpu(a.counters + pair, 1u);
    const int last = old == static_cast<unsigned>(n_splits - 1);
    if (last) ptx::st_relaxed_gpu(a.counters + pair, 0u);
    s_last = last;
  }
  __syncthreads();
  if (!s_last) return;
  // 24 splits per round: a head's 2048 selected positions plus its tail (17 splits)
  // merge in one round of loads
  merge_splits<D, G, kTcThreads, 24>(a, scratch, pair, b, g, n_splits);
}

// ---------------------------------------------------------------- warp-specialised step
// An item's position in the launch and its pair's attended list (CTA-uniform).
struct TcItem {
  int pair, b, g, split, lo;
  SList L;
};

// For launches with more splits than one wave of the one-split kernel holds: persistent
// CTAs (one per SM) over contiguous runs of the (pair, split) items, numbered pair-major
// as that kernel's grid.  A producer warpgroup resolves each item's positions (one item
// ahead) and gathers its K / V rows into a ring of three stages; its copies and the
// item's metadata (which rows are present, the list length) complete the stage's `full`
// barrier.  Two consumer warpgroups take alternate items through the one-split kernel's
// tensor-core steps, each with its own TMEM columns, barriers, query block and merge
// scratch, and hand the stage back through its `empty` barrier when the PV product has
// read it.  One item's gather and two items' products are in flight per SM.  A
// consumer counts its run of splits of one pair in one arrival; the pair's last arrival
// merges.
constexpr int kWsStages = 3;
constexpr int kWsThreads = 3 * kTcThreads;

template <int D>
struct WsSmem {
  static constexpr int kHalf = kBatch * 128;
  static constexpr int kTile = kBatch * D * 2;  // one K or V tile; stage s: K at 2 s kTile
  static constexpr int kQBytes = kTcNQ * D * 2 < 2048 ? 2048 : kTcNQ * D * 2;
  static constexpr int kOffQ = 2 * kWsStages * kTile;              // [2] query blocks
  static constexpr int kOffRed = kOffQ + 2 * kQBytes;              // [2][2][4][16] floats
  static constexpr int kOffScratch = kOffRed + 2 * 2 * 4 * kTcNQ * 4;  // [2][128 * 6] floats
  static constexpr int kOffMeta = kOffScratch + 2 * kTcThreads * 6 * 4;  // [S][8] words
  static constexpr int kOffBar = kOffMeta + kWsStages * 8 * 4;
  static constexpr int kBarBytes = (2 * kWsStages + 4) * 8 + 16;  // full, empty, s[2], o[2], slot
  // with D = 64 the PV MMA reads 16 KB past a V tile (rows never read back)
  static constexpr int kUsedA = kOffBar + kBarBytes;
  static constexpr int kUsedB = (2 * kWsStages - 1) * kTile + 2 * kHalf;
  static constexpr int kBytes = (kUsedA > kUsedB ? kUsedA : kUsedB) + 1024;
  static_assert(kTile % 1024 == 0 && kOffQ % 1024 == 0 && kQBytes % 1024 == 0,
                "swizzle atoms need 1 KB alignment");
  static_assert(kBatch * 128 <= kTile, "P^T fits in the K tile");
  static_assert(kOffScratch % 16 == 0 && kOffBar % 8 == 0, "layout");
};

template <int D, int G>
__global__ void __launch_bounds__(kWsThreads, 1)
    sparse_ws_kernel(const SParams a, const int items_per_cta, const int n_items) {
  using Sm = WsSmem<D>;
  constexpr int LPR = D / 8;        // 16-byte chunks per row
  constexpr int RPI = 32 / LPR;     // rows per warp instruction
  constexpr int QPT = kTcNQ * LPR / kTcThreads;  // query chunks per consumer thread
  static_assert(kTcNQ * LPR % kTcThreads == 0, "query staging");
  extern __shared__ uint8_t ws_smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(ws_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint32_t* meta = reinterpret_cast<uint32_t*>(base + Sm::kOffMeta);  // [s][0..3] rows, [s][4] length
  uint64_t* full = reinterpret_cast<uint64_t*>(base + Sm::kOffBar);
  uint64_t* empty = full + kWsStages;
  uint64_t* bar_s = empty + kWsStages;  // [2]
  uint64_t* bar_o = bar_s + 2;          // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_o + 2);
  __shared__ int s_last[2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wg = warp >> 2;  // 0: producer; 1, 2: consumers
  const int first = blockIdx.x * items_per_cta;
  const int n = min(n_items, first + items_per_cta) - first;
  if (tid == 0) {
    for (int s = 0; s < kWsStages; ++s) {
      ptx::mbar_init(&full[s], kTcThreads + 1);  // every producer's copies + the metadata
      ptx::mbar_init(&empty[s], 1);
    }
    for (int c = 0; c < 2; ++c) {
      ptx::mbar_init(&bar_s[c], 1);
      ptx::mbar_init(&bar_o[c], 1);
    }
    ptx::fence_mbarrier_init();
  }
  if (warp == 4) {
    ptx::tmem_alloc(tmem_slot, 64);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  ptx::pdl_launch_dependents();
  ptx::pdl_wait_primary();  // idx / n_sel come from the preceding kernel

  const auto item_of = [&](int it) {
    TcItem w;
    w.pair = it / a.max_splits;
    w.split = it - w.pair * a.max_splits;
    w.b = w.pair / a.Hkv;
    w.g = w.pair - w.b * a.Hkv;
    w.lo = w.split * a.split_len;
    w.L = SList{0, 0, 0};
    return w;
  };
  const auto has_work = [&](const TcItem& w) {
    return w.lo < w.L.total || (w.split == 0 && w.L.total == 0);
  };
  bool timed_out = false;

  if (wg == 0) {
    // ---------------------------------------------------------------- producer
    struct Loads {
      int j_spec, ns, t0, t1;
    };
    const auto load = [&](const TcItem& w) {
      Loads l;
      l.j_spec = (a.idx != nullptr && w.lo + tid < a.k_max)
                     ? __ldg(a.idx + static_cast<size_t>(w.b) * a.k_max + w.lo + tid)
                     : 0;
      l.ns = a.n_sel != nullptr ? __ldg(a.n_sel + w.b) : 0;
      l.t0 = __ldg(a.tail_start + w.b);
      l.t1 = __ldg(a.seq_len + w.b);
      return l;
    };
    TcItem nxt = item_of(first);
    Loads ln = n > 0 ? load(nxt) : Loads{0, 0, 0, 0};
    for (int j = 0; j < n; ++j) {
      TcItem cur = nxt;
      const Loads lc = ln;
      // position tid of the item -> cache row (-1: absent, zero-filled)
      cur.L = attended_list(lc.ns, lc.t0, lc.t1, a, cur.split == 0 && cur.g == 0 && tid == 0);
      int crow = -1;
      const int pos = cur.lo + tid;
      if (pos < cur.L.total && pos < cur.lo + kBatch) {
        const int jj = pos >= cur.L.ns ? cur.L.t0 + (pos - cur.L.ns) : lc.j_spec;
        if (jj < 0 || jj >= lc.t1) {
          flag_status(a.status, VSD_DEV_BAD_INDEX);
        } else {
          const int blk =
              __ldg(a.block_table + static_cast<size_t>(cur.b) * a.max_blocks + jj / kPageS);
          if (blk < 0 || blk >= a.num_blocks)
            flag_status(a.status, VSD_DEV_BAD_BLOCK);
          else
            crow = (blk * a.Hkv + cur.g) * kPageS + (jj % kPageS);
        }
      }
      if (j + 1 < n) {  // the next item's loads go out under this one's
        nxt = item_of(first + j + 1);
        ln = load(nxt);
      }
      const int s = j % kWsStages;
      const uint32_t use = static_cast<uint32_t>(j / kWsStages);
      if (use > 0 && !ptx::mbar_wait(&empty[s], (use - 1) & 1u)) timed_out = true;
      if (has_work(cur)) {
        // warp w copies rows 32 w .. 32 w + 31, RPI whole rows per instruction
        uint8_t* k_s = base + s * 2 * Sm::kTile;
        uint8_t* v_s = k_s + Sm::kTile;
        const int ch = lane % LPR;
#pragma unroll
        for (int u = 0; u < 32 / RPI; ++u) {
          const int rl = u * RPI + lane / LPR;
          const int r = warp * 32 + rl;
          const int cr = __shfl_sync(0xffffffffu, crow, rl);
          const size_t src = cr >= 0 ? static_cast<size_t>(cr) * D + ch * 8 : 0;
          const int off = (ch >> 3) * Sm::kHalf + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
          ptx::cp_async16(k_s + off, a.k_cache + src, cr >= 0 ? 16u : 0u);
          ptx::cp_async16(v_s + off, a.v_cache + src, cr >= 0 ? 16u : 0u);
        }
      }
      ptx::cp_async_mbar_arrive_noinc(&full[s]);
      const unsigned rows = __ballot_sync(0xffffffffu, crow >= 0);
      if (lane == 0) meta[s * 8 + warp] = rows;
      if (tid == 0) meta[s * 8 + 4] = static_cast<uint32_t>(cur.L.total);
      ptx::named_barrier_sync(3, kTcThreads);
      if (tid == 0) ptx::mbar_arrive(&full[s]);  // releases the metadata
    }
    ptx::cp_async_wait_all();
  } else {
    // ---------------------------------------------------------------- consumers
    const int c = wg - 1;
    const int ct = tid - wg * kTcThreads;  // key of the item = TMEM lane
    const int cw = ct >> 5;                // lane quarter
    const uint32_t tm = tmem + 32 * c;     // S^T: columns [0, 16); O^T: [16, 32)
    uint8_t* q_s = base + Sm::kOffQ + c * Sm::kQBytes;
    float* red = reinterpret_cast<float*>(base + Sm::kOffRed) + c * (2 * 4 * kTcNQ);
    float* scratch = reinterpret_cast<float*>(base + Sm::kOffScratch) + c * (kTcThreads * 6);
    const uint32_t bar_id = 1 + c;
    const auto csync = [bar_id] { ptx::named_barrier_sync(bar_id, kTcThreads); };
    int staged_pair = -1;
    int pend_pair = -1, pend_splits = 0, pend_count = 0;  // partials not yet counted
    uint32_t phase = 0;
    const auto flush = [&]() {
      // the barrier orders every thread's partial stores before the acquire-release
      // count; the last arrival of the pair combines its splits
      ptx::tc_fence_before();
      csync();
      if (ct == 0) {
        const unsigned old =
            ptx::atom_add_acq_rel_gpu(a.counters + pend_pair, static_cast<unsigned>(pend_count));
        const int lst =
            old + static_cast<unsigned>(pend_count) == static_cast<unsigned>(pend_splits);
        if (lst) ptx::st_relaxed_gpu(a.counters + pend_pair, 0u);
        s_last[c] = lst;
      }
      csync();
      if (s_last[c]) {
        const int pb = pend_pair / a.Hkv;
        merge_splits_by<D, G, kTcThreads, 24>(a, scratch, pend_pair, pb, pend_pair - pb * a.Hkv,
                                              pend_splits, ct, csync);
      }
      pend_count = 0;
    };
    for (int j = c; j < n; j += 2) {
      const int s = j % kWsStages;
      const uint32_t use = static_cast<uint32_t>(j / kWsStages);
      if (!ptx::mbar_wait(&full[s], use & 1u)) timed_out = true;
      TcItem cur = item_of(first + j);
      cur.L.total = static_cast<int>(meta[s * 8 + 4]);
      const bool valid = (meta[s * 8 + cw] >> (ct & 31)) & 1u;
      const bool work = has_work(cur);
      const int n_splits = (cur.L.total + a.split_len - 1) / a.split_len;
      const bool direct = n_splits <= 1;
      // every consumer thread has read the stage's metadata past this barrier
      if (pend_count > 0 && (cur.pair != pend_pair || !work || direct)) flush();
      if (!work) {
        csync();
        if (ct == 0) ptx::mbar_arrive(&empty[s]);
        continue;
      }
      uint8_t* k_s = base + s * 2 * Sm::kTile;
      uint8_t* v_s = k_s + Sm::kTile;
      uint8_t* p_s = k_s;
      if (cur.pair != staged_pair) {
        // the group's query rows, padded with zeros to 16 (this consumer's previous QK
        // product, the block's last reader, has completed)
#pragma unroll
        for (int u = 0; u < QPT; ++u) {
          const int i = ct + u * kTcThreads, r = i / LPR, cc = i % LPR;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (r < G)
            v = *reinterpret_cast<const uint4*>(
                a.q + (static_cast<size_t>(cur.b) * a.Hq + cur.g * G + r) * D + cc * 8);
          *reinterpret_cast<uint4*>(q_s + (cc >> 3) * (kTcNQ * 128) + r * 128 +
                                    (((cc & 7) ^ (r & 7)) << 4)) = v;
        }
        staged_pair = cur.pair;
      }
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      csync();
      // ---- S^T = K Q^T
      if (ct == 0) {
        ptx::tc_fence_after();
        constexpr uint32_t idesc = ptx::idesc_bf16_f32(128, kTcNQ, 0, 0);
        const uint32_t ka = ptx::smem_u32(k_s), qa = ptx::smem_u32(q_s);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int hh = kk >> 2, w = kk & 3;
          const uint64_t ad = ptx::sdesc_sw128(ka + hh * Sm::kHalf + w * 32, 16, 1024);
          const uint64_t bd = ptx::sdesc_sw128(qa + hh * kTcNQ * 128 + w * 32, 16, 1024);
          ptx::umma_bf16(tm, ad, bd, idesc, kk > 0 ? 1u : 0u);
        }
        ptx::umma_commit(&bar_s[c]);
      }
      if (!ptx::mbar_wait(&bar_s[c], phase)) timed_out = true;
      ptx::tc_fence_after();
      float sv[kTcNQ];
      ptx::tmem_ld16(tm + (static_cast<uint32_t>(cw * 32) << 16),
                     reinterpret_cast<uint32_t(&)[16]>(sv));
      ptx::tmem_wait_ld();
      // ---- softmax over the item's keys, per head (log2 units)
      float z[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        z[h] = valid ? sv[h] * a.scale_log2 : -INFINITY;
        float mx = z[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) red[cw * kTcNQ + h] = mx;
      }
      csync();
      float m[G], psum[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        m[h] = fmaxf(fmaxf(red[h], red[kTcNQ + h]), fmaxf(red[2 * kTcNQ + h], red[3 * kTcNQ + h]));
        const float pv = (z[h] == -INFINITY) ? 0.f : exp2f(z[h] - m[h]);
        z[h] = pv;
        float sp = pv;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sp += __shfl_xor_sync(0xffffffffu, sp, o);
        if (lane == 0) red[4 * kTcNQ + cw * kTcNQ + h] = sp;
      }
      // row ct of P^T: 16 bf16 (heads >= G are zero) in two swizzled 16-byte chunks
      float pr[kTcNQ];
#pragma unroll
      for (int cc = 0; cc < kTcNQ; ++cc) pr[cc] = cc < G ? z[cc < G ? cc : 0] : 0.f;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        uint4 pk;
        pk.x = pack_bf16x2(pr[k * 8 + 0], pr[k * 8 + 1]);
        pk.y = pack_bf16x2(pr[k * 8 + 2], pr[k * 8 + 3]);
        pk.z = pack_bf16x2(pr[k * 8 + 4], pr[k * 8 + 5]);
        pk.w = pack_bf16x2(pr[k * 8 + 6], pr[k * 8 + 7]);
        *reinterpret_cast<uint4*>(p_s + ct * 128 + ((k ^ (ct & 7)) << 4)) = pk;
      }
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      csync();
#pragma unroll
      for (int h = 0; h < G; ++h)
        psum[h] = red[4 * kTcNQ + h] + red[5 * kTcNQ + h] + red[6 * kTcNQ + h] + red[7 * kTcNQ + h];
      // ---- O^T = V^T P^T; its completion also hands the stage back to the producer
      if (ct == 0) {
        ptx::tc_fence_after();
        constexpr uint32_t idesc = ptx::idesc_bf16_f32(128, kTcNQ, 1, 1);
        const uint32_t va = ptx::smem_u32(v_s), pa = ptx::smem_u32(p_s);
#pragma unroll
        for (int kk = 0; kk < kBatch / 16; ++kk) {
          const uint64_t ad = ptx::sdesc_sw128(va + kk * 2048, Sm::kHalf, 1024);
          const uint64_t bd = ptx::sdesc_sw128(pa + kk * 2048, Sm::kHalf, 1024);
          ptx::umma_bf16(tm + 16, ad, bd, idesc, kk > 0 ? 1u : 0u);
        }
        ptx::umma_commit(&bar_o[c]);
        ptx::umma_commit(&empty[s]);
      }
      if (!ptx::mbar_wait(&bar_o[c], phase)) timed_out = true;
      ptx::tc_fence_after();
      phase ^= 1u;
      if (cw < D / 32) {  // TMEM lanes 0 .. D-1 hold the output dimensions
        float o[kTcNQ];
        ptx::tmem_ld16(tm + (static_cast<uint32_t>(cw * 32) << 16) + 16,
                       reinterpret_cast<uint32_t(&)[16]>(o));
        ptx::tmem_wait_ld();
        const int dim = ct;
        if (direct) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float val = psum[h] > 0.f ? o[h] / psum[h] : 0.f;
            const __nv_bfloat16 bv = __float2bfloat16_rn(val);
            a.out[(static_cast<size_t>(cur.b) * a.Hq + cur.g * G + h) * D + dim] =
                *reinterpret_cast<const uint16_t*>(&bv);
          }
        } else {
          float* wsl =
              a.ws + (static_cast<size_t>(cur.pair) * a.max_splits + cur.split) * SSlot<D, G>::kFloats;
#pragma unroll
          for (int h = 0; h < G; ++h) wsl[SSlot<D, G>::kO + h * D + dim] = o[h];
          if (dim < G) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
              if (h == dim) {
                wsl[h] = m[h];
                wsl[G + h] = psum[h];
              }
            }
          }
        }
      }
      if (!direct) {
        pend_pair = cur.pair;
        pend_splits = n_splits;
        ++pend_count;
      }
    }
    if (pend_count > 0) flush();
  }
  if (timed_out) flag_status(a.status, VSD_DEV_TIMEOUT);
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 64);
  }
}

template <int D, int G>
cudaError_t launch_ws(const SParams& p, long long items, int sm_count, cudaStream_t stream) {
  constexpr int smem = WsSmem<D>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(sparse_ws_kernel<D, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  const int per_cta = static_cast<int>((items + sm_count - 1) / sm_count);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((items + per_cta - 1) / per_cta), 1, 1);
  cfg.blockDim = dim3(kWsThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, sparse_ws_kernel<D, G>, p, per_cta, static_cast<int>(items));
}

template <int D, int G>
cudaError_t launch_tc(const SParams& p, int B, int Hkv, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  // When the splits fit one wave at one CTA per SM, each CTA reserves more than half of
  // an SM's shared memory, so that no two share an SM (its load/store pipe and issue
  // slots); beyond that, as many CTAs per SM as fit (three), in waves.
  int dev = 0, sm_count = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long ctas = static_cast<long long>(p.max_splits) * Hkv * B;
  // more splits than one wave holds at three CTAs per SM: the warp-specialised kernel
  if (ctas > 3LL * sm_count && ctas <= 0x7fffffffLL) return launch_ws<D, G>(p, ctas, sm_count, stream);
  constexpr int kSpreadSmem = 120 * 1024;
  static_assert(TcSmem<D>::kBytes <= kSpreadSmem && 2 * kSpreadSmem > 228 * 1024,
                "one CTA per SM at the spread reservation");
  const int smem = ctas <= sm_count ? kSpreadSmem : TcSmem<D>::kBytes;
  e = cudaFuncSetAttribute(sparse_tc_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.max_splits, Hkv, B);
  cfg.blockDim = dim3(kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, sparse_tc_kernel<D, G>, p);
}

template <int D, int G>
cudaError_t launch_dg(const SParams& p, int B, int Hkv, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  constexpr int smem = static_cast<int>(sizeof(SSmem<D, G>));
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(sparse_decode_kernel<D, G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.max_splits, Hkv, B);
  cfg.blockDim = dim3(SCfg<G>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, sparse_decode_kernel<D, G>, p);
}

}  // namespace

SparsePlan plan_sparse(int k_max, int max_tail) {
  SparsePlan plan;
  const long long len = static_cast<long long>(k_max) + max_tail;
  long long per = kBatch;
  while ((len + per - 1) / per > kMaxSplits) per += kBatch;
  plan.split_len = static_cast<int>(per);
  long long ns = (len + per - 1) / per;
  plan.max_splits = static_cast<int>(ns < 1 ? 1 : ns);
  return plan;
}

size_t sparse_counter_bytes(const SparsePlan& plan, int B, int Hkv) {
  if (plan.max_splits <= 1) return 0;
  return (static_cast<size_t>(B) * Hkv * sizeof(unsigned) + 255) / 256 * 256;
}

size_t sparse_workspace_bytes(const SparsePlan& plan, int B, int Hkv, int G, int head_dim) {
  if (plan.max_splits <= 1) return 0;
  return sparse_counter_bytes(plan, B, Hkv) +
         static_cast<size_t>(B) * Hkv * plan.max_splits * ((2 * G + 3) / 4 * 4 + G * head_dim) *
             sizeof(float);
}

cudaError_t launch_sparse(const SparseArgs& sa, cudaStream_t stream) {
  if (sa.B == 0) return cudaSuccess;
  const SparsePlan plan = plan_sparse(sa.k_max, sa.max_tail);
  SParams p;
  p.q = static_cast<const uint16_t*>(sa.q);
  p.k_cache = static_cast<const uint16_t*>(sa.k_cache);
  p.v_cache = static_cast<const uint16_t*>(sa.v_cache);
  p.block_table = sa.block_table;
  p.idx = sa.idx;
  p.n_sel = sa.n_sel;
  p.tail_start = sa.tail_start;
  p.seq_len = sa.seq_len;
  p.out = static_cast<uint16_t*>(sa.out);
  p.ws = sa.ws;
  p.counters = sa.counters;
  p.status = sa.status;
  p.Hq = sa.Hq;
  p.Hkv = sa.Hkv;
  p.max_blocks = sa.max_blocks;
  p.num_blocks = sa.num_blocks;
  p.k_max = sa.k_max;
  p.split_len = plan.split_len;
  p.max_splits = plan.max_splits;
  p.scale_log2 = sa.scale * kLog2e;
  // splits of one 128-position batch run on the tensor cores; longer splits (lists
  // beyond 1024 batches) on the CUDA-core kernel, which loops over batches
  const bool tc = plan.split_len == kBatch;
#define VSD_SPARSE_CASE(DD, GG)                                                   \
  if (sa.d == DD && sa.G == GG)                                                   \
    return tc ? launch_tc<DD, GG>(p, sa.B, sa.Hkv, stream)                        \
              : launch_dg<DD, GG>(p, sa.B, sa.Hkv, stream);
  VSD_SPARSE_CASE(128, 1)
  VSD_SPARSE_CASE(128, 2)
  VSD_SPARSE_CASE(128, 4)
  VSD_SPARSE_CASE(128, 8)
  VSD_SPARSE_CASE(128, 16)
  VSD_SPARSE_CASE(64, 1)
  VSD_SPARSE_CASE(64, 2)
  VSD_SPARSE_CASE(64, 4)
  VSD_SPARSE_CASE(64, 8)
  VSD_SPARSE_CASE(64, 16)
#undef VSD_SPARSE_CASE
  return cudaErrorInvalidValue;
}

}  // namespace vsd
