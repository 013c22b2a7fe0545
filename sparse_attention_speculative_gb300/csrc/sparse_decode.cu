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
// otherwise each split (or run of splits) writes (m, l, o) to the workspace and the
// pair's last arrival (a per-pair counter in the workspace, reset to zero by that
// arrival) combines them, every load of a round in flight at once, in a fixed order.
// Results are bit-reproducible; the only atomics are the counters.
//
// Two options serve a decode loop.  (1) The step's input token: its K/V rows (k_new,
// v_new) are stored at position seq_len - 1, the last of the dense tail, and attended
// from k_new / v_new directly (no other position of the call reads that cache row).
// (2) The selection's cache rows: the first draft step after a selection writes the
// resolved cache row of every selected position (rows_mode 1) and the later steps read
// them (rows_mode 2), one dependent load (index -> block table) fewer per position.
// Three kernels:
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
  const uint16_t* k_new;  // [B][Hkv][D]: K of the step's input token, or null
  const uint16_t* v_new;
  uint16_t* k_store;      // the caches, written at the input token's position
  uint16_t* v_store;
  const int32_t* block_table;
  const int32_t* idx;
  const int32_t* n_sel;
  const int32_t* tail_start;
  const int32_t* seq_len;
  int32_t* sel_rows;  // [B][k_max]: cache row base of each selected position, or null
  int rows_mode;      // 0: sel_rows unused, 1: resolved and written, 2: read
  int early;          // gather the list before waiting for the preceding kernel
  uint16_t* out;
  float* ws;
  unsigned* counters;  // per pair: splits whose partials are complete
  unsigned* status;
  int Hq, Hkv, max_blocks, num_blocks, k_max;
  int split_len;   // positions per split (a multiple of kBatch)
  int max_splits;  // workspace slots per pair
  float scale_log2;
  // fused sparse verification: R verify rows per sequence, log2 of the group size
  int vrows = 0, gshift = 0;
  // warp-specialised step: the runs' partials are merged by a second kernel (pairs
  // spread over many CTAs) instead of by each pair's last arrival
  int ws_merge_kernel = 0;
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

// Where list position `pos` of pair (b, g) reads its K / V row: `row` is the cache row
// ((block * Hkv + g) * 16 + offset) or -1 (absent: zero-filled and masked); `fresh`
// marks the step's input token, gathered from k_new / v_new and stored at `row`.
struct SRow {
  int row;
  bool fresh;
};

constexpr int kEntryBadIndex = -2147483647 - 1;  // a selected index outside its sequence

// Resolution of a position is split in two so that a persistent kernel can keep the
// block-table load of its next item in flight: position_entry issues the one global
// load a position needs (its block-table entry; with rows_mode 2 the row base an earlier
// step recorded, which `spec` already is), position_row checks and completes it.
// `spec` is the value loaded ahead for a selected position: idx[b][pos], or with
// rows_mode 2 the recorded row base.
__device__ __forceinline__ int position_entry(const SParams& a, const SList& L, int b, int pos,
                                              int t1, int spec) {
  int j;
  if (pos < L.ns) {
    if (a.rows_mode == 2) return spec;
    if (spec < 0 || spec >= t1) return kEntryBadIndex;
    j = spec;
  } else {
    j = L.t0 + (pos - L.ns);
  }
  return __ldcg(a.block_table + static_cast<size_t>(b) * a.max_blocks + j / kPageS);
}

// Checks flag what is wrong (VSD_DEV_BAD_INDEX, VSD_DEV_BAD_BLOCK); with rows_mode 1
// the pairs of KV head 0 record the row base of every selected position (-1 if none).
__device__ __forceinline__ SRow position_row(const SParams& a, const SList& L, int b, int g,
                                             int pos, int spec, int entry) {
  SRow r{-1, false};
  int base = -1;
  if (pos < L.ns && a.rows_mode == 2) {
    const long long lim = static_cast<long long>(a.num_blocks) * a.Hkv * kPageS;
    if (entry >= 0 && entry < lim && (entry / kPageS) % a.Hkv == 0)
      base = entry;
    else
      flag_status(a.status, VSD_DEV_BAD_INDEX);
  } else {
    if (entry == kEntryBadIndex) {
      flag_status(a.status, VSD_DEV_BAD_INDEX);
    } else if (entry < 0 || entry >= a.num_blocks) {
      flag_status(a.status, VSD_DEV_BAD_BLOCK);
    } else {
      const int j = pos < L.ns ? spec : L.t0 + (pos - L.ns);
      base = entry * a.Hkv * kPageS + (j % kPageS);
    }
    if (pos < L.ns && a.rows_mode == 1 && g == 0)
      a.sel_rows[static_cast<size_t>(b) * a.k_max + pos] = base;
    if (pos >= L.ns) r.fresh = a.k_new != nullptr && pos == L.total - 1;
  }
  if (base >= 0)
    r.row = base + g * kPageS;
  else
    r.fresh = false;
  return r;
}

__device__ __forceinline__ SRow resolve_position(const SParams& a, const SList& L, int b, int g,
                                                 int pos, int t1, int spec) {
  return position_row(a, L, b, g, pos, spec, position_entry(a, L, b, pos, t1, spec));
}

// The value a selected position's resolution starts from (see position_entry).
__device__ __forceinline__ const int32_t* spec_source(const SParams& a) {
  return a.rows_mode == 2 ? a.sel_rows : a.idx;
}

// Store the step's input token, already gathered into row r of a 128-byte-swizzled K / V
// tile pair in shared memory (kHalf bytes per 64-column half), into cache row `row`:
// D / 8 16-byte chunks of K and V by one thread, no global load on its path.
template <int D, int kHalf>
__device__ __forceinline__ void store_fresh_from_tile(const SParams& a, const uint8_t* k_s,
                                                      const uint8_t* v_s, int r, int row) {
  uint4* kd = reinterpret_cast<uint4*>(a.k_store + static_cast<size_t>(row) * D);
  uint4* vd = reinterpret_cast<uint4*>(a.v_store + static_cast<size_t>(row) * D);
#pragma unroll
  for (int ch = 0; ch < D / 8; ++ch) {
    const int off = (ch >> 3) * kHalf + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
    kd[ch] = *reinterpret_cast<const uint4*>(k_s + off);
    vd[ch] = *reinterpret_cast<const uint4*>(v_s + off);
  }
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

// Combine the n partials (m, l, o) of one pair and write its G output rows: partial k
// (k < n) is in workspace slot slot_of(k), or absent when that is negative.  Thread t
// of the kSThreads that run it (`sync` is their barrier) = (float4 group of (head,
// dims), part); part p takes partials p, p + kParts, ... with all loads of a round in
// flight; the parts then combine in shared memory.
// kRound: partials per load round when a thread holds one output group.
// `out_row(hh)` is where output row hh goes (null: a padding row, not written).
template <int D, int G, int kSThreads, int kRound, typename Sync, typename SlotOf,
          typename OutRow>
__device__ __forceinline__ void merge_splits_rows(const SParams& a, float* scratch, int pair,
                                                  int n, const int t, Sync sync, SlotOf slot_of,
                                                  OutRow out_row) {
  constexpr int kQ = D / 4;
  constexpr int NG = G * kQ;                              // float4 groups of the output
  constexpr int kGPT = NG > kSThreads ? NG / kSThreads : 1;  // groups per thread
  constexpr int kParts = NG >= kSThreads ? 1 : kSThreads / NG;
  constexpr int kU = kGPT == 1 ? kRound : (kRound / kGPT > 1 ? kRound / kGPT : 1);  // per round
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
        const int sk = k < n ? slot_of(k) : -1;
        if (sk >= 0) {
          const float* sl = base + static_cast<size_t>(sk) * stride;
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
    uint16_t* row = out_row(hh);
    if (row != nullptr) *reinterpret_cast<uint2*>(row + q4 * 4) = pk;
  }
}

// The draft step's merge: output row hh of pair (b, g) is query head g * G + hh.
template <int D, int G, int kSThreads, int kRound, typename Sync, typename SlotOf>
__device__ __forceinline__ void merge_splits_by(const SParams& a, float* scratch, int pair, int b,
                                                int g, int n, const int t, Sync sync,
                                                SlotOf slot_of) {
  merge_splits_rows<D, G, kSThreads, kRound>(
      a, scratch, pair, n, t, sync, slot_of, [&a, b, g](int hh) {
        return a.out + (static_cast<size_t>(b) * a.Hq + g * G + hh) * D;
      });
}

template <int D, int G, int kSThreads, int kRound = 16>
__device__ __forceinline__ void merge_splits(const SParams& a, float* scratch, int pair, int b,
                                             int g, int n) {
  merge_splits_by<D, G, kSThreads, kRound>(a, scratch, pair, b, g, n,
                                           static_cast<int>(threadIdx.x),
                                           [] { __syncthreads(); }, [](int k) { return k; });
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

  ptx::pdl_wait_primary();       // idx / n_sel come from the preceding kernel
  ptx::pdl_launch_dependents();  // after the wait: see kv_append.cu

  // First round of loads, independent of one another: the list lengths, the first
  // batch's indices or row bases (speculatively: used only for positions that turn out
  // to be selected ones) and the queries.
  const int lo = split * a.split_len;
  const int wbase0 = lo + warp * kKeysPerWarp;
  const int32_t* spec_src = spec_source(a);
  int j_spec[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int pos = wbase0 + u * KPI + sub;
    j_spec[u] = (spec_src != nullptr && pos < a.k_max)
                    ? __ldcg(spec_src + static_cast<size_t>(b) * a.k_max + pos)
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
  const int ns_raw = a.n_sel != nullptr ? __ldcg(a.n_sel + b) : 0;
  const int t0_raw = __ldcg(a.tail_start + b);
  const int t1 = __ldcg(a.seq_len + b);
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
    bool fresh[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int pos = wbase + u * KPI + sub;
      row[u] = -1;
      fresh[u] = false;
      if (pos < hi) {
        const int spec = pos >= L.ns ? 0
                         : wbase == wbase0
                             ? j_spec[u]
                             : __ldcg(spec_src + static_cast<size_t>(b) * a.k_max + pos);
        const SRow r = resolve_position(a, L, b, g, pos, t1, spec);
        row[u] = r.row;
        fresh[u] = r.fresh;
      }
    }
    // ---- every K and V load of the batch in flight: 16 bytes of each row per lane (the
    // step's input token from k_new / v_new, each lane also storing its 16 bytes of it)
    uint4 kr[U], vr[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (fresh[u]) {
        const size_t src = (static_cast<size_t>(b) * a.Hkv + g) * D + lr * 8;
        kr[u] = *reinterpret_cast<const uint4*>(a.k_new + src);
        vr[u] = *reinterpret_cast<const uint4*>(a.v_new + src);
        const size_t dst = static_cast<size_t>(row[u]) * D + lr * 8;
        *reinterpret_cast<uint4*>(a.k_store + dst) = kr[u];
        *reinterpret_cast<uint4*>(a.v_store + dst) = vr[u];
      } else if (row[u] >= 0) {
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

// Reduce v[0 .. G) (G a power of two up to 16) over the warp's 32 lanes with `op`, every
// column at once: butterfly steps on the low lane bits that halve the columns a lane
// keeps (G - 1 shuffles), then plain steps on the other bits (5 - log2 G shuffles), all
// shuffles of a step independent.  Afterwards lane L holds column L % G.  (One shuffle
// chain per column with a shared-memory store after each, 5 G dependent shuffles, took
// 0.55 us of a 128-key tile's softmax at G = 4 and 1.2 us at G = 8.)
template <int G, typename Op>
__device__ __forceinline__ float warp_reduce_heads(float (&v)[G], Op op) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int m = G / 2; m >= 1; m >>= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < m; ++i) {
      const float send = upper ? v[i] : v[i + m];
      const float keep = upper ? v[i + m] : v[i];
      v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, m));
    }
  }
  float r = v[0];
#pragma unroll
  for (int m = 16; m >= G; m >>= 1) r = op(r, __shfl_xor_sync(0xffffffffu, r, m));
  return r;
}

// Softmax of one 128-key tile for the G heads of a group (log2 units): the thread of
// key t (warp `qw` of the tile's four) holds its logits sv[] (G columns of S^T), `valid`
// false for an absent key; `red` is [2][4][kTcNQ] floats of the 128 threads, `sync`
// their barrier.  Returns the heads' maxima in m[] and key t's probabilities in p[];
// with kSums each warp's per-head sums are stored in red[1][qw][.] (added up by the
// caller after its next barrier).
template <int G, bool kSums = true, typename Sync>
__device__ __forceinline__ void tile_softmax(const float (&sv)[G], bool valid, float scale_log2,
                                             float* red, int qw, Sync sync, float (&m)[G],
                                             float (&p)[G]) {
  const int lane = threadIdx.x & 31;
  float v[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    p[h] = valid ? sv[h] * scale_log2 : -INFINITY;
    v[h] = p[h];
  }
  const float wmax = warp_reduce_heads<G>(v, [](float x, float y) { return fmaxf(x, y); });
  if (lane < G) red[qw * kTcNQ + lane] = wmax;
  sync();
#pragma unroll
  for (int h = 0; h < G; ++h)
    m[h] = fmaxf(fmaxf(red[h], red[kTcNQ + h]), fmaxf(red[2 * kTcNQ + h], red[3 * kTcNQ + h]));
#pragma unroll
  for (int h = 0; h < G; ++h) {
    p[h] = (p[h] == -INFINITY) ? 0.f : exp2f(p[h] - m[h]);
    v[h] = p[h];
  }
  if constexpr (kSums) {
    const float wsum = warp_reduce_heads<G>(v, [](float x, float y) { return x + y; });
    if (lane < G) red[4 * kTcNQ + qw * kTcNQ + lane] = wsum;
  }
}

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
  uint64_t* bar_fin = bar_s + 2;  // every product of this CTA complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_s + 3);
  __shared__ int s_last;

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  if (t == 0) {
    ptx::mbar_init(bar_s, 1);
    ptx::mbar_init(bar_o, 1);
    ptx::mbar_init(bar_fin, 1);
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
  // In the early mode the list is resolved and gathered before the wait for the
  // preceding kernel, unless this split holds the step's input token (read from k_new);
  // the queries, the workspace and the outputs always come after it.
  bool waited = a.early == 0;
  if (waited) {
    ptx::pdl_wait_primary();  // idx / n_sel come from the preceding kernel
    ptx::pdl_launch_dependents();
  }

  // this thread's index (or row base) is loaded together with the list lengths (every
  // position below k_max is valid memory; it is used only if the position is a
  // selected one)
  const int lo = split * a.split_len;
  const int32_t* spec_src = spec_source(a);
  const int j_spec = (spec_src != nullptr && lo + t < a.k_max)
                         ? __ldcg(spec_src + static_cast<size_t>(b) * a.k_max + lo + t)
                         : 0;
  const int ns_raw = a.n_sel != nullptr ? __ldcg(a.n_sel + b) : 0;
  const int t0_raw = __ldcg(a.tail_start + b);
  const int t1 = __ldcg(a.seq_len + b);
  const SList L = attended_list(ns_raw, t0_raw, t1, a, split == 0 && g == 0 && t == 0);
  const bool work = lo < L.total || (split == 0 && L.total == 0);
  const int n_splits = (L.total + a.split_len - 1) / a.split_len;
  const bool direct = n_splits <= 1;
  const int pair = b * a.Hkv + g;
  bool timed_out = false;
  bool drain_s = false, drain_o = false;  // an MMA whose completion wait gave up
  const bool holds_fresh = a.k_new != nullptr && L.total > L.ns && L.total - 1 >= lo &&
                           L.total - 1 < lo + kBatch;
  if (!waited && (holds_fresh || !work)) {
    ptx::pdl_wait_primary();
    ptx::pdl_launch_dependents();
    waited = true;
  }

  if (work) {
    // ---- this thread's position -> cache row (-1: absent, zero-filled)
    const int pos = lo + t;
    SRow rr{-1, false};
    if (pos < L.total && pos < lo + kBatch) rr = resolve_position(a, L, b, g, pos, t1, j_spec);
    const int crow = rr.row;
    // ---- gather: warp w copies rows 32 w .. 32 w + 31, RPI whole rows per instruction
    // (the step's input token from k_new / v_new)
    const int ch = lane % LPR;
    const unsigned fresh_bits = __ballot_sync(0xffffffffu, rr.fresh);
    const size_t fresh_off = (static_cast<size_t>(b) * a.Hkv + g) * D;
    const uint16_t* k_fresh = a.k_new != nullptr ? a.k_new + fresh_off : a.k_cache;
    const uint16_t* v_fresh = a.v_new != nullptr ? a.v_new + fresh_off : a.v_cache;
#pragma unroll
    for (int u = 0; u < 32 / RPI; ++u) {
      const int rl = u * RPI + lane / LPR;  // row within the warp
      const int r = warp * 32 + rl;
      const int cr = __shfl_sync(0xffffffffu, crow, rl);
      const bool fr = (fresh_bits >> rl) & 1u;
      const size_t src = cr >= 0 ? static_cast<size_t>(cr) * D + ch * 8 : 0;
      const uint16_t* ks = fr ? k_fresh + ch * 8 : a.k_cache + src;
      const uint16_t* vs = fr ? v_fresh + ch * 8 : a.v_cache + src;
      const int off = (ch >> 3) * Sm::kHalf + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
      ptx::cp_async16(k_s + off, ks, cr >= 0 ? 16u : 0u);
      ptx::cp_async16(v_s + off, vs, cr >= 0 ? 16u : 0u);
    }
    ptx::cp_async_commit();
    if (!waited) {
      ptx::pdl_wait_primary();
      ptx::pdl_launch_dependents();
      waited = true;
    }
    uint4 qv[QPT];
#pragma unroll
    for (int u = 0; u < QPT; ++u) {
      const int i = t + u * kTcThreads, r = i / LPR, c = i % LPR;
      qv[u] = make_uint4(0, 0, 0, 0);
      if (r < G)
        qv[u] = *reinterpret_cast<const uint4*>(
            a.q + (static_cast<size_t>(b) * a.Hq + g * G + r) * D + c * 8);
    }
    // ---- the group's query rows (loaded after the wait), padded with zeros to 16
#pragma unroll
    for (int u = 0; u < QPT; ++u) {
      const int i = t + u * kTcThreads, r = i / LPR, c = i % LPR;
      *reinterpret_cast<uint4*>(q_s + (c >> 3) * (kTcNQ * 128) + r * 128 +
                                (((c & 7) ^ (r & 7)) << 4)) = qv[u];
    }
    ptx::cp_async_wait_all();
    ptx::fence_proxy_async_smem();  // make the copies and stores visible to the tensor cores
    __syncthreads();
    // the step's input token joins the cache from its gathered row (P^T overwrites the
    // K tile only after the QK product below has read it)
    if (rr.fresh) store_fresh_from_tile<D, Sm::kHalf>(a, k_s, v_s, t, crow);

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
    // (a test build waits on the end-of-kernel barrier here, which nothing completes yet)
    if (!ptx::mbar_wait(VSD_STALL(true) ? bar_fin : bar_s, 0)) {
      timed_out = true;
      drain_s = true;
    }
    ptx::tc_fence_after();
    float sv[G];  // the G real query columns (the rest are zero padding)
    ptx::tmem_ld<G>(tmem + (static_cast<uint32_t>(warp * 32) << 16), reinterpret_cast<uint32_t*>(sv));
    ptx::tmem_wait_ld();
    // ---- softmax over the CTA's keys, per head (log2 units)
    float m[G], z[G], psum[G];
    tile_softmax<G>(sv, crow >= 0, a.scale_log2, red, warp, [] { __syncthreads(); }, m, z);
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

    // ---- O^T = V^T P^T (not issued by a thread whose QK wait gave up: the QK product
    // may still be running, and the output is flagged anyway)
    bool issued_o = false;
    if (t == 0 && !drain_s) {
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
      issued_o = true;
    }
    // the heads' sums while the product runs
#pragma unroll
    for (int h = 0; h < G; ++h)
      psum[h] = red[4 * kTcNQ + h] + red[5 * kTcNQ + h] + red[6 * kTcNQ + h] + red[7 * kTcNQ + h];
    // every thread learns whether the PV product was issued (one CTA-wide vote)
    issued_o = __syncthreads_or(issued_o);
    if (issued_o && !ptx::mbar_wait(bar_o, 0)) {
      timed_out = true;
      drain_o = true;
    }
    ptx::tc_fence_after();
    if (warp < D / 32) {  // TMEM lanes 0 .. D-1 hold the output dimensions
      float o[G];
      ptx::tmem_ld<G>(tmem + (static_cast<uint32_t>(warp * 32) << 16) + 16,
                      reinterpret_cast<uint32_t*>(o));
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
  // never free TMEM under a running MMA: one more commit by the issuing thread arrives
  // once every product it issued is done (waited for with the drain limit)
  if (t == 0 && (drain_s || drain_o || work)) {
    ptx::umma_commit(bar_fin);
    ptx::mbar_wait_drain(bar_fin, 0);
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

// ---------------------------------------------------------------- fused sparse verification
// Dustin's sparse verification (summary, "Verification workflow", steps 3-4) without
// materialising the compressed cache: the tensor-core step above with the R * G verify
// rows of a KV group on the MMA's N side (row r = t * G + h, padded to NQ = 16 or 32)
// over the list idx[b, 0 .. n_sel) followed by the verify block P_b .. P_b + R - 1.
// The block is masked causally: verify row t attends block position u only for u <= t.
// One split of up to 128 list positions per CTA; a pair of more than one split writes
// the splits' (m, l, o) to the workspace and a merge kernel (one block per output row)
// combines them: one CTA merging all 32 rows of 17-65 splits took 9-35 us.
template <int D, int NQ>
struct TcvSmem {
  static constexpr int kHalf = kBatch * 128;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kBatch * D * 2;
  static constexpr int kQBytes = NQ * D * 2 < 2048 ? 2048 : NQ * D * 2;
  static constexpr int kOffQ = kOffV + kBatch * D * 2;
  static constexpr int kOffRed = kOffQ + kQBytes;         // [2][4][NQ] floats
  static constexpr int kOffBar = kOffRed + 2 * 4 * NQ * 4;
  static constexpr int kOffValid = kOffBar + 64;  // [kBatch] bytes: the key's row is present
  static constexpr int kOffP = kOffK;  // P^T in the K tile (after its QK product)
  static constexpr int kUsed =
      kOffValid + kBatch > kOffV + 2 * kHalf ? kOffValid + kBatch : kOffV + 2 * kHalf;
  static constexpr int kBytes = kUsed + 1024;
  static_assert(kOffQ % 1024 == 0 && kQBytes % 1024 == 0, "swizzle atoms need 1 KB alignment");
  static_assert(NQ * 2 <= 128, "a P^T row holds the NQ probabilities of one key");
};

// Reduce v[0 .. NQ) (NQ = 8, 16 or 32 columns) over the warp's 32 lanes with `op`,
// every column at once: full exchanges at the lane distances of NQ and above, then
// butterfly steps that halve the columns a lane keeps (lanes with the step's bit set
// keep the upper half), all of a step independent.  Afterwards lane L holds column
// L % NQ.
template <int NQ, typename Op>
__device__ __forceinline__ float warp_reduce_columns(float (&v)[NQ], Op op) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 16; off >= NQ; off >>= 1) {
#pragma unroll
    for (int i = 0; i < NQ; ++i) v[i] = op(v[i], __shfl_xor_sync(0xffffffffu, v[i], off));
  }
#pragma unroll
  for (int m = NQ / 2; m >= 1; m >>= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < m; ++i) {
      const float send = upper ? v[i] : v[i + m];
      const float keep = upper ? v[i + m] : v[i];
      v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, m));
    }
  }
  return v[0];
}

// N consecutive TMEM columns of this warp's lane quarter (N = 8, 16 or 32).
template <int N>
__device__ __forceinline__ void tmem_ld_f32(uint32_t taddr, float (&v)[N]) {
  if constexpr (N == 32) {
    ptx::tmem_ld<16>(taddr, reinterpret_cast<uint32_t*>(v));
    ptx::tmem_ld<16>(taddr + 16, reinterpret_cast<uint32_t*>(v) + 16);
  } else {
    ptx::tmem_ld<N>(taddr, reinterpret_cast<uint32_t*>(v));
  }
  ptx::tmem_wait_ld();
}

// kParts warps per TMEM lane quarter: warp w holds the keys (and, for O^T, the
// dimensions) of quarter w % 4 and the column part w / 4 of the NQ verify rows.  Only
// the lower 128 threads resolve positions and gather rows (one per key, as in the draft
// step); the others learn which keys are present through shared memory.  Two parts when
// the launch is one wave at one CTA per SM (the softmax of a 32K call 2.3 -> 1.1 us,
// the call 8.56 -> 8.22 us); one where several CTAs share an SM and hide one another's
// softmax (the 128K call took 17.6 us with one part, 18.4 with two).
template <int D, int NQ, int kParts>
__global__ void __launch_bounds__(kParts * kTcThreads) sparse_verify_tc_kernel(const SParams a) {
  using Sm = TcvSmem<D, NQ>;
  constexpr int kSvThreads = kParts * kTcThreads;
  constexpr int LPR = D / 8;                  // 16-byte chunks per row
  constexpr int RPI = 32 / LPR;               // rows per warp instruction
  constexpr int NH = NQ / kParts;             // verify columns per thread
  static_assert(NH % 8 == 0, "P^T chunks of 8 columns");
  extern __shared__ uint8_t tcv_smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(tcv_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* k_s = base + Sm::kOffK;
  uint8_t* v_s = base + Sm::kOffV;
  uint8_t* q_s = base + Sm::kOffQ;
  uint8_t* p_s = base + Sm::kOffP;
  float* red = reinterpret_cast<float*>(base + Sm::kOffRed);
  uint64_t* bar_s = reinterpret_cast<uint64_t*>(base + Sm::kOffBar);
  uint64_t* bar_o = bar_s + 1;
  uint64_t* bar_fin = bar_s + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_s + 3);
  uint8_t* valid_s = base + Sm::kOffValid;

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  // (one part: compile-time constants, every thread a gatherer)
  const int quarter = warp & 3;
  const int col0 = kParts == 1 ? 0 : (warp >> 2) * NH;
  const int key = kParts == 1 ? t : quarter * 32 + lane;  // TMEM lane: key (S^T) / dim (O^T)
  const bool gatherer = kParts == 1 || t < kBatch;        // key == t for these
  const int G = 1 << a.gshift;
  const int NR = a.vrows << a.gshift;  // real verify rows of the group (<= NQ)
  if (t == 0) {
    ptx::mbar_init(bar_s, 1);
    ptx::mbar_init(bar_o, 1);
    ptx::mbar_init(bar_fin, 1);
    ptx::fence_mbarrier_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(tmem_slot, 2 * NQ);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;  // S^T: columns [0, NQ); O^T: [NQ, 2 NQ)
  const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
  // idx / n_sel / the prefix lengths may come from the preceding kernel; in the early
  // mode they do not (nor the selected positions' cache rows): those rows are resolved
  // and gathered before the wait, the verify block's rows and the queries after it
  if (!a.early) {
    ptx::pdl_wait_primary();
    ptx::pdl_launch_dependents();
  }

  const int lo = split * a.split_len;
  const int j_spec = (gatherer && a.idx != nullptr && lo + t < a.k_max)
                         ? __ldcg(a.idx + static_cast<size_t>(b) * a.k_max + lo + t)
                         : 0;
  const int ns_raw = a.n_sel != nullptr ? __ldcg(a.n_sel + b) : 0;
  const int P = __ldcg(a.tail_start + b);  // the prefix length: the verify block starts there
  const SList L = attended_list(ns_raw, P, P + a.vrows, a, split == 0 && g == 0 && t == 0);
  const bool work = lo < L.total || (split == 0 && L.total == 0);
  const int n_splits = (L.total + a.split_len - 1) / a.split_len;
  const bool direct = n_splits <= 1;
  const int pair = b * a.Hkv + g;
  bool timed_out = false, drain_s = false, drain_o = false;
  // output row r of the pair: verify row r >> gshift, query head g * G + (r & (G - 1))
  const auto out_row = [&](int r) -> uint16_t* {
    if (r >= NR) return nullptr;
    return a.out + ((static_cast<size_t>(b) * a.vrows + (r >> a.gshift)) * a.Hq + g * G +
                    (r & (G - 1))) * D;
  };

  if (work) {
    // ---- the gatherer's position -> cache row (-1: absent, zero-filled and masked)
    const int pos = lo + key;
    SRow rr{-1, false};
    if (gatherer && pos < L.total && pos < lo + kBatch)
      rr = resolve_position(a, L, b, g, pos, P + a.vrows, j_spec);
    const int crow = rr.row;
    const bool in_block = pos >= L.ns && pos < L.total;  // a verify-block row
    const int ch = lane % LPR;
    // the selected (and absent) rows, or the verify block's rows (gatherer warps)
    const auto gather = [&](bool block_rows) {
#pragma unroll
      for (int u = 0; u < 32 / RPI; ++u) {
        const int rl = u * RPI + lane / LPR;
        const int r = warp * 32 + rl;
        const int cr = __shfl_sync(0xffffffffu, crow, rl);
        const bool blk = __shfl_sync(0xffffffffu, in_block, rl);
        const size_t src = cr >= 0 ? static_cast<size_t>(cr) * D + ch * 8 : 0;
        const int off = (ch >> 3) * Sm::kHalf + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
        if (blk == block_rows) {
          ptx::cp_async16(k_s + off, a.k_cache + src, cr >= 0 ? 16u : 0u);
          ptx::cp_async16(v_s + off, a.v_cache + src, cr >= 0 ? 16u : 0u);
        }
      }
    };
    if (gatherer) gather(false);
    if (a.early) {
      ptx::pdl_wait_primary();
      ptx::pdl_launch_dependents();
    }
    if (gatherer) {
      gather(true);
      ptx::cp_async_commit();
      if (kParts > 1) valid_s[t] = crow >= 0 ? 1 : 0;
    }
    // ---- the group's verify rows, padded with zeros to NQ, K-major and swizzled (all
    // of a thread's loads in flight at once)
    constexpr int QPT = (NQ * LPR + kSvThreads - 1) / kSvThreads;  // chunks per thread
#pragma unroll
    for (int u = 0; u < QPT; ++u) {
      const int i = t + u * kSvThreads;
      if (NQ * LPR % kSvThreads != 0 && i >= NQ * LPR) break;
      const int r = i / LPR, c = i % LPR;
      uint4 qv = make_uint4(0, 0, 0, 0);
      if (r < NR)
        qv = *reinterpret_cast<const uint4*>(
            a.q + ((static_cast<size_t>(b) * a.vrows + (r >> a.gshift)) * a.Hq + g * G +
                   (r & (G - 1))) * D + c * 8);
      *reinterpret_cast<uint4*>(q_s + (c >> 3) * (NQ * 128) + r * 128 +
                                (((c & 7) ^ (r & 7)) << 4)) = qv;
    }
    if (gatherer) ptx::cp_async_wait_all();
    ptx::fence_proxy_async_smem();
    __syncthreads();

    // ---- S^T = K Q^T  (M = 128 keys, N = NQ rows, K = head_dim)
    if (t == 0) {
      ptx::tc_fence_after();
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(128, NQ, 0, 0);
      const uint32_t ka = ptx::smem_u32(k_s), qa = ptx::smem_u32(q_s);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int hh = kk >> 2, w = kk & 3;
        const uint64_t ad = ptx::sdesc_sw128(ka + hh * Sm::kHalf + w * 32, 16, 1024);
        const uint64_t bd = ptx::sdesc_sw128(qa + hh * NQ * 128 + w * 32, 16, 1024);
        ptx::umma_bf16(tmem, ad, bd, idesc, kk > 0 ? 1u : 0u);
      }
      ptx::umma_commit(bar_s);
    }
    if (!ptx::mbar_wait(bar_s, 0)) {
      timed_out = true;
      drain_s = true;
    }
    ptx::tc_fence_after();
    float z[NH];  // this key's logits for the thread's NH rows
    tmem_ld_f32<NH>(tmem + lane_addr + col0, z);
    // ---- softmax per row over the CTA's keys (log2 units), the verify block masked
    // causally: a block key at u = pos - n_sel is seen by the rows of verify row >= u
    const bool valid = kParts == 1 ? crow >= 0 : valid_s[key] != 0;
    const int u_blk = pos - L.ns;  // < 0: a selected position, seen by every row
#pragma unroll
    for (int c = 0; c < NH; ++c) {
      const int cc = col0 + c;
      const bool seen = valid && cc < NR && (u_blk < 0 || u_blk <= (cc >> a.gshift));
      z[c] = seen ? z[c] * a.scale_log2 : -INFINITY;
    }
    // per-row maxima: one column-wise reduction over the warp's keys, the quarters meet
    // in shared memory, lane c of every warp then holds row col0 + c's maximum
    {
      float v[NH];
#pragma unroll
      for (int c = 0; c < NH; ++c) v[c] = z[c];
      const float wm = warp_reduce_columns<NH>(v, [](float x, float y) { return fmaxf(x, y); });
      if (lane < NH) red[quarter * NQ + col0 + lane] = wm;
    }
    __syncthreads();
    const int cl = col0 + lane % NH;
    const float m_lane =
        fmaxf(fmaxf(red[cl], red[NQ + cl]), fmaxf(red[2 * NQ + cl], red[3 * NQ + cl]));
    {
      float v[NH];
#pragma unroll
      for (int c = 0; c < NH; ++c) {
        const float m = __shfl_sync(0xffffffffu, m_lane, c);
        const float p = (z[c] == -INFINITY) ? 0.f : exp2f(z[c] - m);
        z[c] = p;
        v[c] = p;
      }
      const float ws = warp_reduce_columns<NH>(v, [](float x, float y) { return x + y; });
      if (lane < NH) red[4 * NQ + quarter * NQ + col0 + lane] = ws;
    }
    // row `key` of P^T: this thread's NH bf16 in NH / 8 swizzled 16-byte chunks
#pragma unroll
    for (int k = 0; k < NH / 8; ++k) {
      uint4 pk;
      pk.x = pack_bf16x2(z[k * 8 + 0], z[k * 8 + 1]);
      pk.y = pack_bf16x2(z[k * 8 + 2], z[k * 8 + 3]);
      pk.z = pack_bf16x2(z[k * 8 + 4], z[k * 8 + 5]);
      pk.w = pack_bf16x2(z[k * 8 + 6], z[k * 8 + 7]);
      const int chunk = col0 / 8 + k;
      *reinterpret_cast<uint4*>(p_s + key * 128 + ((chunk ^ (key & 7)) << 4)) = pk;
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();

    // ---- O^T = V^T P^T  (M = 128, N = NQ, K = 128 keys); not issued after a QK wait
    // that gave up (that product may still be running)
    bool issued_o = false;
    if (t == 0 && !drain_s) {
      ptx::tc_fence_after();
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(128, NQ, 1, 1);
      const uint32_t va = ptx::smem_u32(v_s), pa = ptx::smem_u32(p_s);
#pragma unroll
      for (int kk = 0; kk < kBatch / 16; ++kk) {
        const uint64_t ad = ptx::sdesc_sw128(va + kk * 2048, Sm::kHalf, 1024);
        const uint64_t bd = ptx::sdesc_sw128(pa + kk * 2048, Sm::kHalf, 1024);
        ptx::umma_bf16(tmem + NQ, ad, bd, idesc, kk > 0 ? 1u : 0u);
      }
      ptx::umma_commit(bar_o);
      issued_o = true;
    }
    issued_o = __syncthreads_or(issued_o);
    if (issued_o && !ptx::mbar_wait(bar_o, 0)) {
      timed_out = true;
      drain_o = true;
    }
    ptx::tc_fence_after();
    if (quarter < D / 32) {  // TMEM lanes 0 .. D-1 hold the output dimensions
      float o[NH];
      tmem_ld_f32<NH>(tmem + lane_addr + NQ + col0, o);
      const int dim = key;
      if (direct) {
#pragma unroll
        for (int c = 0; c < NH; ++c) {
          const int r = col0 + c;
          uint16_t* row = out_row(r);
          if (row == nullptr) continue;
          const float l = red[4 * NQ + r] + red[5 * NQ + r] + red[6 * NQ + r] + red[7 * NQ + r];
          const __nv_bfloat16 bv = __float2bfloat16_rn(l > 0.f ? o[c] / l : 0.f);
          row[dim] = *reinterpret_cast<const uint16_t*>(&bv);
        }
      } else {
        float* wsl = a.ws + (static_cast<size_t>(pair) * a.max_splits + split) * SSlot<D, NQ>::kFloats;
#pragma unroll
        for (int c = 0; c < NH; ++c) wsl[SSlot<D, NQ>::kO + (col0 + c) * D + dim] = o[c];
        if (col0 == 0 && dim < NQ) {  // m and l of row `dim`
          wsl[dim] = fmaxf(fmaxf(red[dim], red[NQ + dim]), fmaxf(red[2 * NQ + dim], red[3 * NQ + dim]));
          wsl[NQ + dim] = red[4 * NQ + dim] + red[5 * NQ + dim] + red[6 * NQ + dim] + red[7 * NQ + dim];
        }
      }
    }
    if (timed_out) flag_status(a.status, VSD_DEV_TIMEOUT);
  }
  // never free TMEM under a running MMA: one more commit arrives once every product this
  // CTA issued is done (waited for with the drain limit)
  if (t == 0 && (drain_s || drain_o || work)) {
    ptx::umma_commit(bar_fin);
    ptx::mbar_wait_drain(bar_fin, 0);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 2 * NQ);
  }
}

// The splits' partials of one output row of one pair: block (row, KV head, sequence)
// of kSvParts * D threads, thread (part, dimension); part p combines splits p,
// p + kSvParts, ... (every load of a round in flight), then the parts combine in shared
// memory in part order.  One part for up to 32 splits, four beyond (a 32K row's 17
// splits: 8.8 us per call with one part, 10.1 us with four; 128K's 65 splits: 19.5 us
// with one, 18.4 us with four).  A programmatic dependent of the kernel above (waits
// for all its partials).
template <int D, int NQ, int kSvParts>
__global__ void __launch_bounds__(kSvParts * D) sparse_verify_merge_kernel(const SParams a) {
  __shared__ float pm[kSvParts][D], pl[kSvParts][D], po[kSvParts][D];
  const int r = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int dim = threadIdx.x % D, part = threadIdx.x / D;
  ptx::pdl_wait_primary();
  ptx::pdl_launch_dependents();
  const int ns_raw = a.n_sel != nullptr ? __ldcg(a.n_sel + b) : 0;
  const int P = __ldcg(a.tail_start + b);
  const SList L = attended_list(ns_raw, P, P + a.vrows, a, false);
  const int n = (L.total + a.split_len - 1) / a.split_len;
  if (n <= 1) return;  // one split wrote its rows itself
  constexpr int kU = kSvParts == 1 ? 32 : 16;
  const size_t stride = SSlot<D, NQ>::kFloats;
  const float* base = a.ws + static_cast<size_t>(b * a.Hkv + g) * a.max_splits * stride;
  float M = -INFINITY, Ls = 0.f, O = 0.f;
  for (int k0 = part; k0 < n; k0 += kU * kSvParts) {
    float mk[kU], lk[kU], ok[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int k = k0 + u * kSvParts;
      if (k < n) {
        const float* sl = base + static_cast<size_t>(k) * stride;
        mk[u] = __ldcg(sl + r);
        lk[u] = __ldcg(sl + NQ + r);
        ok[u] = __ldcg(sl + SSlot<D, NQ>::kO + r * D + dim);
      } else {
        mk[u] = -INFINITY;
        lk[u] = 0.f;
        ok[u] = 0.f;
      }
    }
    float mn = M;
#pragma unroll
    for (int u = 0; u < kU; ++u) mn = fmaxf(mn, mk[u]);
    const float sc = (M == -INFINITY) ? 0.f : exp2f(M - mn);
    Ls *= sc;
    O *= sc;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const float w = (mk[u] == -INFINITY) ? 0.f : exp2f(mk[u] - mn);
      Ls += w * lk[u];
      O += w * ok[u];
    }
    M = mn;
  }
  if constexpr (kSvParts > 1) {
    pm[part][dim] = M;
    pl[part][dim] = Ls;
    po[part][dim] = O;
    __syncthreads();
  }
  if (part != 0) return;
  float Lt = Ls, Ot = O;
  if constexpr (kSvParts > 1) {
    float mn = -INFINITY;
#pragma unroll
    for (int q = 0; q < kSvParts; ++q) mn = fmaxf(mn, pm[q][dim]);
    Lt = 0.f;
    Ot = 0.f;
#pragma unroll
    for (int q = 0; q < kSvParts; ++q) {
      const float w = (pm[q][dim] == -INFINITY) ? 0.f : exp2f(pm[q][dim] - mn);
      Lt += w * pl[q][dim];
      Ot += w * po[q][dim];
    }
  }
  const int G = 1 << a.gshift;
  const __nv_bfloat16 bv = __float2bfloat16_rn(Lt > 0.f ? Ot / Lt : 0.f);
  a.out[((static_cast<size_t>(b) * a.vrows + (r >> a.gshift)) * a.Hq + g * G + (r & (G - 1))) * D +
        dim] = *reinterpret_cast<const uint16_t*>(&bv);
}

// ---------------------------------------------------------------- warp-specialised step
// An item's position in the launch and its pair's attended list (CTA-uniform).
struct TcItem {
  int pair, b, g, split, lo;
  SList L;
};

// For launches with more splits than one wave of the one-split kernel holds: persistent
// CTAs (one per SM) over contiguous runs of the (pair, split) items, numbered pair-major
// as that kernel's grid.  A producer warpgroup resolves each item's positions one item
// ahead of its gather (the indices or row bases two items ahead) and gathers its K / V
// rows into a ring of three stages; its copies and the item's metadata (which rows are
// present, the list length) complete the stage's `full` barrier.  Two consumer
// warpgroups take alternate items through the one-split kernel's tensor-core steps,
// each with its own TMEM columns, barriers, query block and merge scratch, and hand the
// stage back through its `empty` barrier when the PV product has read it.  A consumer
// folds its items of one pair into one running (m, l, o) in registers and writes a
// single partial per run (to the slot of the run's first split); the pair's last
// arrival merges the runs' partials, whose slots follow from the launch geometry
// (ws_slot), in a fixed order -- or, where a pair spans more than eight CTAs (a 128K
// list: ~17 CTAs, 34 partials), a second kernel does (one block per pair, a
// programmatic dependent): there the last arrival's merge outlasts a kernel boundary
// (128K step 13.4 -> 12.6 us), where a pair spans few CTAs it does not (the 36-layer
// loop 17.9 -> 20.5 us, the 72B batch 14.0 -> 15.3 us with the second kernel).
constexpr int kWsStages = 3;
constexpr int kWsThreads = 3 * kTcThreads;
constexpr float kDraftTau = 8.0f;  // slack of a run's reference maximum, log2 units

template <int D>
struct WsSmem {
  static constexpr int kHalf = kBatch * 128;
  static constexpr int kTile = kBatch * D * 2;  // one K or V tile; stage s: K at 2 s kTile
  static constexpr int kQBytes = kTcNQ * D * 2 < 2048 ? 2048 : kTcNQ * D * 2;
  static constexpr int kOffQ = 2 * kWsStages * kTile;              // [2] query blocks
  static constexpr int kOffRed = kOffQ + 2 * kQBytes;              // [2][2][4][16] floats
  static constexpr int kOffScratch = kOffRed + 2 * 2 * 4 * kTcNQ * 4;  // [2][128 * 6] floats
  static constexpr int kOffMeta = kOffScratch + 2 * kTcThreads * 6 * 4;  // [S][16] words
  static constexpr int kOffCtl = kOffMeta + kWsStages * 16 * 4;  // abort flag
  static constexpr int kCtlBytes = 64;
  static constexpr int kOffBar = kOffCtl + kCtlBytes;
  // full, empty, s[2], o[2], fin[2], TMEM slot
  static constexpr int kBarBytes = (2 * kWsStages + 6) * 8 + 16;
  // with D = 64 the PV MMA reads 16 KB past a V tile (rows never read back)
  static constexpr int kUsedA = kOffBar + kBarBytes;
  static constexpr int kUsedB = (2 * kWsStages - 1) * kTile + 2 * kHalf;
  static constexpr int kBytes = (kUsedA > kUsedB ? kUsedA : kUsedB) + 1024;
  static_assert(kTile % 1024 == 0 && kOffQ % 1024 == 0 && kQBytes % 1024 == 0,
                "swizzle atoms need 1 KB alignment");
  static_assert(kBatch * 128 <= kTile, "P^T fits in the K tile");
  static_assert(kOffScratch % 16 == 0 && kOffBar % 8 == 0, "layout");
};

// Workspace slot of partial k (k < ws_partials) of a pair whose items are
// [i0, i0 + n), c0 = i0 / ipc: partial k belongs to consumer k & 1 of CTA c0 + k / 2,
// which writes it at the split of its first item in the pair; -1 when that consumer has
// no item of the pair.  32-bit arithmetic (a launch holds fewer than 2^31 items), the
// division done once per merge: with a 64-bit division per partial the merge that
// finishes a 36-layer loop's draft step cost 0.3 us more per step.
__device__ __forceinline__ int ws_slot(int k, int i0, int n, int c0, int ipc) {
  const int i1 = i0 + n;
  const int cs = (c0 + (k >> 1)) * ipc;
  int lo = cs > i0 ? cs : i0;
  if (((lo - cs) & 1) != (k & 1)) ++lo;
  const int hi = cs + ipc < i1 ? cs + ipc : i1;
  return lo < hi ? lo - i0 : -1;
}

__device__ __forceinline__ int ws_partials(int i0, int n, int ipc) {
  return 2 * ((i0 + n - 1) / ipc - i0 / ipc + 1);
}

// OR of `pred` over the `nthreads` threads of named barrier `id` (a barrier too).
__device__ __forceinline__ bool named_vote_or(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// The list lengths of one sequence as every thread of the kernel reads them.
struct SLen {
  int ns, t0, t1;
};

__device__ __forceinline__ SLen load_len(const SParams& a, int b) {
  SLen l;
  l.ns = a.n_sel != nullptr ? __ldcg(a.n_sel + b) : 0;
  l.t0 = __ldcg(a.tail_start + b);
  l.t1 = __ldcg(a.seq_len + b);
  return l;
}

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
  // per stage: [0..3] present rows (one word per producer warp), [4] list length,
  // [8..11] per warp the lane holding the step's input token (or -1), [12..15] its row
  uint32_t* meta = reinterpret_cast<uint32_t*>(base + Sm::kOffMeta);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + Sm::kOffCtl);
  uint64_t* full = reinterpret_cast<uint64_t*>(base + Sm::kOffBar);
  uint64_t* empty = full + kWsStages;
  uint64_t* bar_s = empty + kWsStages;  // [2]
  uint64_t* bar_o = bar_s + 2;          // [2]
  uint64_t* bar_fin = bar_o + 2;        // [2] every product of a consumer complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_fin + 2);
  __shared__ int s_last[2];
  __shared__ int s_raised[2];  // per consumer: the item whose logits raised the maximum

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
      ptx::mbar_init(&bar_fin[c], 1);
    }
    *abort_flag = 0;
    s_raised[0] = s_raised[1] = -1;
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
  // A wait that gave up raises the CTA's abort flag (and the status bit once): from
  // then on no copy or MMA is issued, and the products already issued are waited for
  // again before the TMEM columns are freed.  No named barrier depends on the flag or
  // on anything a failed wait leaves unfinished, so every warpgroup runs to its end.
  const auto set_abort = [&]() {
    if (!*abort_flag) {
      *abort_flag = 1;
      flag_status(a.status, VSD_DEV_TIMEOUT);
    }
  };

  if (wg == 0) {
    // ---------------------------------------------------------------- producer
    // Position tid of each item is resolved in three stages, one item apart, so that no
    // load is waited for on the way to an item's copies: the index (or recorded row
    // base) and the list lengths two items ahead, the block-table entry one item ahead,
    // the checks and the row for the item being gathered.  In the early mode the first
    // stages' items (those without the step's input token) are resolved and gathered
    // before the wait for the preceding kernel.
    struct Pre {
      int spec;
      SLen len;
    };
    struct Mid {
      int spec, entry;
    };
    const int32_t* spec_src = spec_source(a);
    const auto pre_load = [&](const TcItem& w) {
      Pre l;
      l.spec = (spec_src != nullptr && w.lo + tid < a.k_max)
                   ? __ldcg(spec_src + static_cast<size_t>(w.b) * a.k_max + w.lo + tid)
                   : 0;
      l.len = load_len(a, w.b);
      return l;
    };
    const auto pos_in = [&](const TcItem& w) {
      const int pos = w.lo + tid;
      return pos < w.L.total && pos < w.lo + kBatch;
    };
    // sets w.L and issues the entry load (not waited for here)
    const auto mid_of = [&](TcItem& w, const Pre& l) {
      w.L = attended_list(l.len.ns, l.len.t0, l.len.t1, a, w.split == 0 && w.g == 0 && tid == 0);
      Mid m{l.spec, 0};
      if (pos_in(w)) m.entry = position_entry(a, w.L, w.b, w.lo + tid, l.len.t1, l.spec);
      return m;
    };
    // the item holds the step's input token (read from k_new, which the preceding kernel
    // may write)
    const auto holds_fresh = [&](const TcItem& w) {
      return a.k_new != nullptr && w.L.total > w.L.ns && w.L.total - 1 >= w.lo &&
             w.L.total - 1 < w.lo + kBatch;
    };
    bool waited = a.early == 0;
    if (waited) {
      ptx::pdl_wait_primary();  // idx / n_sel come from the preceding kernel
      ptx::pdl_launch_dependents();
    }
    TcItem cur = item_of(first), nxt = item_of(first + 1);
    Mid mcur{0, 0};
    Pre pnxt{0, {0, 0, 0}};
    if (n > 0) {
      const Pre p0 = pre_load(cur);
      if (n > 1) pnxt = pre_load(nxt);
      mcur = mid_of(cur, p0);
    }
    for (int j = 0; j < n; ++j) {
      // a stage is reused only after the consumers (which wait for the preceding kernel)
      // hand it back, and k_new is read only after the wait
      if (!waited && (j >= kWsStages || holds_fresh(cur))) {
        ptx::pdl_wait_primary();
        ptx::pdl_launch_dependents();
        waited = true;
      }
      // this item's row (its entry load was issued one item ago), then the next item's
      // entry load and the loads of the item after it, all before this item's stage wait
      const SRow rcur = pos_in(cur) ? position_row(a, cur.L, cur.b, cur.g, cur.lo + tid,
                                                   mcur.spec, mcur.entry)
                                    : SRow{-1, false};
      Mid mnxt{0, 0};
      if (j + 1 < n) {
        const Pre pl = pnxt;
        if (j + 2 < n) pnxt = pre_load(item_of(first + j + 2));
        mnxt = mid_of(nxt, pl);
      }
      const int s = j % kWsStages;
      const uint32_t use = static_cast<uint32_t>(j / kWsStages);
      if (use > 0 && !ptx::mbar_wait(&empty[s], (use - 1) & 1u, abort_flag)) set_abort();
      const int crow = rcur.row;
      const unsigned fresh_bits = __ballot_sync(0xffffffffu, rcur.fresh);
      if (has_work(cur) && !*abort_flag) {
        // warp w copies rows 32 w .. 32 w + 31, RPI whole rows per instruction (the
        // step's input token from k_new / v_new)
        uint8_t* k_s = base + s * 2 * Sm::kTile;
        uint8_t* v_s = k_s + Sm::kTile;
        const int ch = lane % LPR;
        const size_t fresh_off = (static_cast<size_t>(cur.b) * a.Hkv + cur.g) * D + ch * 8;
#pragma unroll
        for (int u = 0; u < 32 / RPI; ++u) {
          const int rl = u * RPI + lane / LPR;
          const int r = warp * 32 + rl;
          const int cr = __shfl_sync(0xffffffffu, crow, rl);
          const bool fr = (fresh_bits >> rl) & 1u;
          const size_t src = cr >= 0 ? static_cast<size_t>(cr) * D + ch * 8 : 0;
          const uint16_t* ks = fr ? a.k_new + fresh_off : a.k_cache + src;
          const uint16_t* vs = fr ? a.v_new + fresh_off : a.v_cache + src;
          const int off = (ch >> 3) * Sm::kHalf + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
          ptx::cp_async16(k_s + off, ks, cr >= 0 ? 16u : 0u);
          ptx::cp_async16(v_s + off, vs, cr >= 0 ? 16u : 0u);
        }
      }
      ptx::cp_async_mbar_arrive_noinc(&full[s]);
      const unsigned rows = __ballot_sync(0xffffffffu, crow >= 0);
      if (lane == 0) {
        meta[s * 16 + warp] = rows;
        meta[s * 16 + 8 + warp] = fresh_bits ? static_cast<uint32_t>(__ffs(fresh_bits) - 1) : 0xFFFFFFFFu;
      }
      if (rcur.fresh) meta[s * 16 + 12 + warp] = static_cast<uint32_t>(crow);
      if (tid == 0) meta[s * 16 + 4] = static_cast<uint32_t>(cur.L.total);
      ptx::named_barrier_sync(3, kTcThreads);
      if (tid == 0) ptx::mbar_arrive(&full[s]);  // releases the metadata
      cur = nxt;
      nxt = item_of(first + j + 2);
      mcur = mnxt;
    }
    if (!waited) {
      ptx::pdl_wait_primary();
      ptx::pdl_launch_dependents();
    }
    ptx::cp_async_wait_all();
  } else {
    // ---------------------------------------------------------------- consumers
    ptx::pdl_wait_primary();  // the workspace, q and the outputs: after the preceding kernel
    ptx::pdl_launch_dependents();
    const int c = wg - 1;
    const int ct = tid - wg * kTcThreads;  // key of the item = TMEM lane
    const int cw = ct >> 5;                // lane quarter
    const uint32_t tm = tmem + 32 * c;     // S^T: columns [0, 16); O^T: [16, 32)
    uint8_t* q_s = base + Sm::kOffQ + c * Sm::kQBytes;
    float* red = reinterpret_cast<float*>(base + Sm::kOffRed) + c * (2 * 4 * kTcNQ);
    float* scratch = reinterpret_cast<float*>(base + Sm::kOffScratch) + c * (kTcThreads * 6);
    const uint32_t bar_id = 1 + c;
    const auto csync = [bar_id] { ptx::named_barrier_sync(bar_id, kTcThreads); };
    // the query rows of a (sequence, KV group), padded with zeros to 16 rows, and the
    // list lengths of an item's sequence: loaded one item of this consumer ahead
    const auto load_q = [&](const TcItem& w, uint4 (&qv)[QPT]) {
#pragma unroll
      for (int u = 0; u < QPT; ++u) {
        const int i = ct + u * kTcThreads, r = i / LPR, cc = i % LPR;
        qv[u] = make_uint4(0, 0, 0, 0);
        if (r < G)
          qv[u] = *reinterpret_cast<const uint4*>(
              a.q + (static_cast<size_t>(w.b) * a.Hq + w.g * G + r) * D + cc * 8);
      }
    };
    uint4 qcur[QPT], qnext[QPT];
    SLen lcur{0, 0, 0}, lnext{0, 0, 0};
    int qnext_pair = -1;
    if (c < n) {
      const TcItem w0 = item_of(first + c);
      lnext = load_len(a, w0.b);
      load_q(w0, qnext);
      qnext_pair = w0.pair;
    }
    int staged_pair = -1;
    // The running partial of this consumer's current run of one pair's splits.  The
    // run's items share one reference maximum per head, m_ref, set by the run's first
    // item: a later item's probabilities are exp2(z - m_ref) unless one of its logits
    // exceeds m_ref by more than kDraftTau, which the barrier before the PV product
    // reports (and m_ref is raised, o_run and l_part rescaled).  So a later item reduces
    // neither maxima nor sums across threads: each thread adds up the probabilities of
    // its keys in l_part, and the run's sums are reduced once, when the run is written.
    // (With per-item maxima and sums the two cross-warp reductions took a quarter of an
    // item's time.)  Pairs of a single split keep the exact per-item softmax.
    int run_pair = -1, run_first = 0, run_count = 0, run_splits = 0;
    float m_ref[G], l_part[G], o_run[G];
    uint32_t phase = 0;
    const auto flush = [&]() {
      // the run's sums over every thread's keys (the first barrier: the sums' area may
      // still be read for an earlier item)
      float v[G];
#pragma unroll
      for (int h = 0; h < G; ++h) v[h] = l_part[h];
      const float wsum = warp_reduce_heads<G>(v, [](float x, float y) { return x + y; });
      csync();
      if (lane < G) red[4 * kTcNQ + cw * kTcNQ + lane] = wsum;
      csync();
      // the run's partial at the slot of its first split; the barrier orders every
      // thread's stores before the acquire-release count, whose last arrival merges
      float* wsl = a.ws + (static_cast<size_t>(run_pair) * a.max_splits + run_first) *
                              SSlot<D, G>::kFloats;
      if (ct < D) {
#pragma unroll
        for (int h = 0; h < G; ++h) wsl[SSlot<D, G>::kO + h * D + ct] = o_run[h];
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        if (h == ct) {
          wsl[h] = m_ref[h];
          wsl[G + h] =
              red[4 * kTcNQ + h] + red[5 * kTcNQ + h] + red[6 * kTcNQ + h] + red[7 * kTcNQ + h];
        }
      }
      if (a.ws_merge_kernel) {  // merged by the next kernel
        run_count = 0;
        return;
      }
      csync();
      if (ct == 0) {
        const unsigned old =
            ptx::atom_add_acq_rel_gpu(a.counters + run_pair, static_cast<unsigned>(run_count));
        const int lst =
            old + static_cast<unsigned>(run_count) == static_cast<unsigned>(run_splits);
        if (lst) ptx::st_relaxed_gpu(a.counters + run_pair, 0u);
        s_last[c] = lst;
      }
      csync();
      if (s_last[c]) {
        const int pb = run_pair / a.Hkv;
        const int i0 = run_pair * a.max_splits;
        const int ns = run_splits, ipc = items_per_cta, c0 = i0 / ipc;
        // a pair has two partials per CTA it spans (about a dozen in a 36-layer decode
        // loop): a load round of 12 (8 for wider groups) keeps the merge's registers
        // within the consumer's
        merge_splits_by<D, G, kTcThreads, (G <= 4 ? 12 : 8)>(
            a, scratch, run_pair, pb, run_pair - pb * a.Hkv, ws_partials(i0, ns, ipc), ct, csync,
            [i0, ns, c0, ipc](int k) { return ws_slot(k, i0, ns, c0, ipc); });
      }
      run_count = 0;
    };
    for (int j = c; j < n; j += 2) {
      TcItem cur = item_of(first + j);
      lcur = lnext;
      if (cur.pair != staged_pair) {
#pragma unroll
        for (int u = 0; u < QPT; ++u) qcur[u] = qnext[u];
      }
      // the next item's lengths and (for a new pair) query rows go out now
      if (j + 2 < n) {
        const TcItem wn = item_of(first + j + 2);
        lnext = load_len(a, wn.b);
        if (wn.pair != cur.pair && wn.pair != qnext_pair) {
          load_q(wn, qnext);
          qnext_pair = wn.pair;
        }
      }
      // every thread computes the same list from the same lengths: the control flow of
      // the warpgroup never depends on what a wait left behind
      cur.L = attended_list(lcur.ns, lcur.t0, lcur.t1, a, false);
      const bool work = has_work(cur);
      const int n_splits = (cur.L.total + a.split_len - 1) / a.split_len;
      const bool direct = n_splits <= 1;
      if (run_count > 0 && (cur.pair != run_pair || !work || direct)) flush();
      const int s = j % kWsStages;
      const uint32_t use = static_cast<uint32_t>(j / kWsStages);
      // (a test build waits on the end-of-kernel barrier for the first item, which
      // nothing completes yet)
      if (!(VSD_STALL(j == c) ? ptx::mbar_wait(&bar_fin[c], 0u, abort_flag)
                              : ptx::mbar_wait(&full[s], use & 1u, abort_flag)))
        set_abort();
      const bool stop = *abort_flag != 0;
      if (!work) {
        if (ct == 0) ptx::mbar_arrive(&empty[s]);  // nothing of this stage is read
        continue;
      }
      const bool valid = (meta[s * 16 + cw] >> (ct & 31)) & 1u;
      uint8_t* k_s = base + s * 2 * Sm::kTile;
      uint8_t* v_s = k_s + Sm::kTile;
      uint8_t* p_s = k_s;
      // the step's input token joins the cache from its gathered row (P^T overwrites the
      // K tile only after the QK product below has read it)
      if (!stop && static_cast<int>(meta[s * 16 + 8 + cw]) == (ct & 31))
        store_fresh_from_tile<D, Sm::kHalf>(a, k_s, v_s, ct,
                                            static_cast<int>(meta[s * 16 + 12 + cw]));
      if (cur.pair != staged_pair) {
        // the group's query rows (this consumer's previous QK product, the block's last
        // reader, has completed)
#pragma unroll
        for (int u = 0; u < QPT; ++u) {
          const int i = ct + u * kTcThreads, r = i / LPR, cc = i % LPR;
          *reinterpret_cast<uint4*>(q_s + (cc >> 3) * (kTcNQ * 128) + r * 128 +
                                    (((cc & 7) ^ (r & 7)) << 4)) = qcur[u];
        }
        staged_pair = cur.pair;
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        csync();
      }
      // ---- S^T = K Q^T (the stage has landed: this thread waited for it)
      if (ct == 0 && !stop) {
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
      bool s_failed = false;
      if (!stop && !ptx::mbar_wait(&bar_s[c], phase, abort_flag)) {
        set_abort();
        s_failed = true;
      }
      ptx::tc_fence_after();
      float sv[G];  // the G real query columns (the rest are zero padding)
      ptx::tmem_ld<G>(tm + (static_cast<uint32_t>(cw * 32) << 16),
                      reinterpret_cast<uint32_t*>(sv));
      ptx::tmem_wait_ld();
      // ---- probabilities over the item's keys, per head (log2 units)
      const auto write_p = [&](const float (&pv)[G]) {
        // row ct of P^T: 16 bf16 (heads >= G are zero) in two swizzled 16-byte chunks
        float pr[kTcNQ];
#pragma unroll
        for (int cc = 0; cc < kTcNQ; ++cc) pr[cc] = cc < G ? pv[cc < G ? cc : 0] : 0.f;
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
      };
      float z[G], p[G], psum[G];
      bool over = false;
      if (direct) {
        float m[G];
        tile_softmax<G, true>(sv, valid, a.scale_log2, red, cw, csync, m, p);
      } else if (run_count == 0) {
        tile_softmax<G, false>(sv, valid, a.scale_log2, red, cw, csync, m_ref, p);
      } else {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          z[h] = valid ? sv[h] * a.scale_log2 : -INFINITY;
          over |= z[h] > m_ref[h] + kDraftTau;
          p[h] = (z[h] == -INFINITY) ? 0.f : exp2f(z[h] - m_ref[h]);
        }
      }
      write_p(p);
      if (over) s_raised[c] = j;
      // a barrier that also tells every thread whether some QK wait gave up (the PV
      // product is issued only when the QK product is known to be complete) or some
      // logit raised the maximum
      bool skip_pv = named_vote_or(bar_id, kTcThreads, stop || s_failed || over);
      if (skip_pv) {
        const bool raised = s_raised[c] == j;
        skip_pv = named_vote_or(bar_id, kTcThreads, stop || s_failed);
        if (raised && !skip_pv) {
          // the new maxima over the reference and this item's logits; the run so far
          // is rescaled and the probabilities written again
          float v[G];
#pragma unroll
          for (int h = 0; h < G; ++h) v[h] = z[h];
          const float wmax = warp_reduce_heads<G>(v, [](float x, float y) { return fmaxf(x, y); });
          if (lane < G) red[cw * kTcNQ + lane] = wmax;
          csync();
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float mn = fmaxf(fmaxf(m_ref[h], fmaxf(red[h], red[kTcNQ + h])),
                                   fmaxf(red[2 * kTcNQ + h], red[3 * kTcNQ + h]));
            const float f = (m_ref[h] == -INFINITY) ? 0.f : exp2f(m_ref[h] - mn);
            o_run[h] *= f;
            l_part[h] *= f;
            m_ref[h] = mn;
            p[h] = (z[h] == -INFINITY) ? 0.f : exp2f(z[h] - mn);
          }
          write_p(p);
          csync();
        }
      }
      // ---- O^T = V^T P^T; its completion also hands the stage back to the producer
      if (ct == 0) {
        if (!skip_pv) {
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
        } else {
          ptx::mbar_arrive(&empty[s]);
        }
      }
      // a single split's sums while the product runs
      if (direct) {
#pragma unroll
        for (int h = 0; h < G; ++h)
          psum[h] = red[4 * kTcNQ + h] + red[5 * kTcNQ + h] + red[6 * kTcNQ + h] + red[7 * kTcNQ + h];
      }
      if (!skip_pv && !ptx::mbar_wait(&bar_o[c], phase, abort_flag)) set_abort();
      ptx::tc_fence_after();
      // both barriers completed a phase when both products ran; after an abort the
      // phases no longer matter (no product is issued and the drain keeps its parity)
      if (!skip_pv) phase ^= 1u;
      float o[G];
#pragma unroll
      for (int h = 0; h < G; ++h) o[h] = 0.f;
      if (cw < D / 32) {  // TMEM lanes 0 .. D-1 hold the output dimensions
        ptx::tmem_ld<G>(tm + (static_cast<uint32_t>(cw * 32) << 16) + 16,
                        reinterpret_cast<uint32_t*>(o));
        ptx::tmem_wait_ld();
      }
      if (direct) {
        if (ct < D) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float val = psum[h] > 0.f ? o[h] / psum[h] : 0.f;
            const __nv_bfloat16 bv = __float2bfloat16_rn(val);
            a.out[(static_cast<size_t>(cur.b) * a.Hq + cur.g * G + h) * D + ct] =
                *reinterpret_cast<const uint16_t*>(&bv);
          }
        }
      } else if (run_count == 0) {
        run_pair = cur.pair;
        run_first = cur.split;
        run_splits = n_splits;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          l_part[h] = p[h];
          o_run[h] = o[h];
        }
        run_count = 1;
      } else {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          l_part[h] += p[h];
          o_run[h] += o[h];
        }
        ++run_count;
      }
    }
    if (run_count > 0) flush();
    // one more commit by the issuing thread arrives once every product it issued is
    // done (waited for with the drain limit) before the TMEM columns are freed
    if (ct == 0) {
      ptx::umma_commit(&bar_fin[c]);
      ptx::mbar_wait_drain(&bar_fin[c], 0);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 64);
  }
}

// The runs' partials of one pair of the warp-specialised step when the step leaves
// them to a second kernel: block = pair, thread = a float4 group of the G x D output
// (in parts where the output has fewer than 128 groups), every partial's load of a
// round in flight, the slots from the launch geometry.
template <int D, int G>
__global__ void __launch_bounds__(kTcThreads) ws_merge_kernel(const SParams a, const int items_per_cta) {
  __shared__ float scratch[kTcThreads * 6];
  ptx::pdl_wait_primary();  // every partial of the step is written
  ptx::pdl_launch_dependents();
  const int pair = blockIdx.x, b = pair / a.Hkv, g = pair - b * a.Hkv;
  const SLen len = load_len(a, b);
  const SList L = attended_list(len.ns, len.t0, len.t1, a, false);
  const int n_splits = (L.total + a.split_len - 1) / a.split_len;
  if (n_splits <= 1) return;  // one split wrote its output itself
  const int i0 = pair * a.max_splits, ipc = items_per_cta, c0 = i0 / ipc;
  merge_splits_by<D, G, kTcThreads, 16>(
      a, scratch, pair, b, g, ws_partials(i0, n_splits, ipc), static_cast<int>(threadIdx.x),
      [] { __syncthreads(); },
      [i0, n_splits, c0, ipc](int k) { return ws_slot(k, i0, n_splits, c0, ipc); });
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
  // a pair's splits spread over more than eight CTAs: the merge as a second kernel
  SParams q = p;
  q.ws_merge_kernel = p.max_splits > 1 && (p.max_splits + per_cta - 1) / per_cta + 1 > 8;
  e = cudaLaunchKernelEx(&cfg, sparse_ws_kernel<D, G>, q, per_cta, static_cast<int>(items));
  if (e != cudaSuccess || !q.ws_merge_kernel) return e;
  cfg.gridDim = dim3(static_cast<unsigned>(items / p.max_splits), 1, 1);
  cfg.blockDim = dim3(kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, ws_merge_kernel<D, G>, q, per_cta);
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

template <int D, int NQ>
cudaError_t launch_tcv(const SParams& p, int B, int Hkv, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int dev = 0, sm_count = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // as the draft step: one CTA per SM when the splits fit one wave, else as many as fit
  const long long ctas = static_cast<long long>(p.max_splits) * Hkv * B;
  constexpr int kSpreadSmem = 120 * 1024;
  static_assert(TcvSmem<D, NQ>::kBytes <= kSpreadSmem, "spread reservation");
  const bool one_wave = ctas <= sm_count;
  const int smem = one_wave ? kSpreadSmem : TcvSmem<D, NQ>::kBytes;
  const auto kern = one_wave ? sparse_verify_tc_kernel<D, NQ, 2> : sparse_verify_tc_kernel<D, NQ, 1>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.max_splits, Hkv, B);
  cfg.blockDim = dim3((one_wave ? 2 : 1) * kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess || p.max_splits <= 1) return e;
  cfg.gridDim = dim3(p.vrows << p.gshift, Hkv, B);
  cfg.dynamicSmemBytes = 0;
  if (p.max_splits <= 32) {
    cfg.blockDim = dim3(D, 1, 1);
    return cudaLaunchKernelEx(&cfg, sparse_verify_merge_kernel<D, NQ, 1>, p);
  }
  cfg.blockDim = dim3(4 * D, 1, 1);
  return cudaLaunchKernelEx(&cfg, sparse_verify_merge_kernel<D, NQ, 4>, p);
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
  p.k_new = static_cast<const uint16_t*>(sa.k_new);
  p.v_new = static_cast<const uint16_t*>(sa.v_new);
  p.k_store = static_cast<uint16_t*>(sa.k_store);
  p.v_store = static_cast<uint16_t*>(sa.v_store);
  p.sel_rows = sa.sel_rows;
  p.rows_mode = sa.sel_rows != nullptr && sa.k_max > 0 ? sa.rows_mode : 0;
  p.early = sa.early;
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

int sparse_verify_fused_nq(int R, int G, int k_max) {
  const int nr = R * G;
  if (nr < 1 || nr > 32 || (G & (G - 1)) != 0) return 0;
  if (plan_sparse(k_max, R).split_len != kBatch) return 0;  // lists beyond 1024 batches
  return nr <= 16 ? 16 : 32;
}

size_t sparse_verify_fused_bytes(int B, int Hkv, int R, int G, int k_max, int head_dim) {
  const int nq = sparse_verify_fused_nq(R, G, k_max);
  if (nq == 0) return 0;
  const SparsePlan plan = plan_sparse(k_max, R);
  return static_cast<size_t>(B) * Hkv * plan.max_splits * ((2 * nq + 3) / 4 * 4 + nq * head_dim) *
         sizeof(float);
}

cudaError_t launch_sparse_verify_fused(const SparseArgs& sa, int R, cudaStream_t stream) {
  if (sa.B == 0) return cudaSuccess;
  const int nq = sparse_verify_fused_nq(R, sa.G, sa.k_max);
  if (nq == 0) return cudaErrorInvalidValue;
  const SparsePlan plan = plan_sparse(sa.k_max, R);
  SParams p;
  p.q = static_cast<const uint16_t*>(sa.q);
  p.k_cache = static_cast<const uint16_t*>(sa.k_cache);
  p.v_cache = static_cast<const uint16_t*>(sa.v_cache);
  p.k_new = nullptr;
  p.v_new = nullptr;
  p.k_store = nullptr;
  p.v_store = nullptr;
  p.sel_rows = nullptr;
  p.rows_mode = 0;
  p.early = sa.early;
  p.block_table = sa.block_table;
  p.idx = sa.idx;
  p.n_sel = sa.n_sel;
  p.tail_start = sa.tail_start;  // the prefix lengths
  p.seq_len = nullptr;
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
  p.vrows = R;
  int gs = 0;
  while ((1 << gs) < sa.G) ++gs;
  p.gshift = gs;
  if (sa.d == 128) return nq == 16 ? launch_tcv<128, 16>(p, sa.B, sa.Hkv, stream)
                                   : launch_tcv<128, 32>(p, sa.B, sa.Hkv, stream);
  if (sa.d == 64) return nq == 16 ? launch_tcv<64, 16>(p, sa.B, sa.Hkv, stream)
                                  : launch_tcv<64, 32>(p, sa.B, sa.Hkv, stream);
  return cudaErrorInvalidValue;
}

}  // namespace vsd
