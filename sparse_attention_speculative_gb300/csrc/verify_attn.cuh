// verify_attn.cuh -- verification attention with Collect-2-Query on sm_103a
// (kernel templates; instantiated per head dimension in verify_attn_d*.cu).
//
// What it computes ("Vegas" technical summary, sec. 2 verification phase, sec. 2.B
// Collect-2-Query, sec. 3 kernel instrumentation): the gamma+1 verify rows of every
// sequence attend the whole paged KV cache (causal inside the verify block) and, in
// the same pass over K, the scaled pre-softmax logits of two chosen rows are written
// to HBM together with their per-KV-group sums (the first reduction of the
// selection score of sec. 2.A).
//
// How (GB300 design):
//   * One persistent CTA per SM.  The work is the list of (sequence, KV head) pairs
//     times 128-key tiles; CTA c streams the contiguous range [c W / C, (c+1) W / C)
//     of that list, so every SM gets the same number of tiles (split-K over the
//     context, balanced to the tile).  A pair cut by CTA boundaries leaves one
//     partial (m, l, o) per CTA; a merge kernel (one block per pair and verify row,
//     a programmatic dependent, all partial loads of a block in one round)
//     combines them.
//   * Warps 0 and 10 stream K and V pages with 4-D TMA loads (128-byte swizzle) into
//     two separate shared-memory rings (3 stages of 32 KB each for head_dim 128, 5
//     of 16 KB for 64), so a K stage is refilled as soon as its QK MMA has read it.
//     Each 128-key tile is 8 pages; a page whose block-table entry is invalid is
//     fetched at an out-of-range coordinate, which the TMA unit fills with zeros.
//   * Warp 1 issues tcgen05 MMAs with the small dimension on N ("swap AB"):
//       S^T[128 keys x NQ] = K_tile[128 x d] * Q^T        (K-major A and B)
//       O^T[d x NQ]       += V_tile^T[d x 128] * P^T      (MN-major A and B)
//     NQ = R*G rounded up to 16 covers all verify rows of one KV group.  It runs an
//     event loop: QK of a tile as soon as its K tile has landed, PV of a tile as soon
//     as its P^T is written, whichever is ready first (non-blocking polls).
//     Accumulators live in TMEM (S double-buffered, O single).  For NQ <= 32 P^T is
//     double-buffered in the two halves of each 128-byte swizzled row, so the
//     softmax of tile i+1 never waits for the PV MMA of tile i.
//   * Warps 2-9 (softmax): TMEM lane = key, and the NQ columns are split between the
//     two warps that share a lane quarter.  Each thread reads its half row of logits,
//     forms P against a running maximum shared by all keys of a column, and writes
//     its P^T chunks.  The maximum is only raised when some logit exceeds it by more
//     than 2^8 (one CTA vote per tile, bar.red.or), so the common path needs no
//     cross-thread max; each thread keeps partial row sums l, reduced once per pair.
//     Causal / length / bad-page masks are evaluated per key only where a key can be
//     hidden.  The lower half also reads the two collected rows' logits with
//     runtime-addressed TMEM loads and writes them (32 consecutive keys per warp
//     store) with their group sum.
#pragma once

#include <cfloat>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace vsd {
namespace verify_detail {

using namespace ptx;

constexpr int kTile = 128;      // keys per tile (the MMA M dimension of S^T)
constexpr int kPage = 16;       // tokens per cache page
constexpr int kPagesPerTile = kTile / kPage;
constexpr float kTau = 8.0f;    // lazy-max slack, log2 units
constexpr int kSoftmaxWarps = 8;
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
// warp 0: K producer, warp 1: MMA issuer, warps 2-9: softmax, warp 10: V producer
constexpr int kThreads = 96 + kSoftmaxThreads;
constexpr int kVWarp = 10;
constexpr int kSoftmaxBar = 1;  // named barrier of the softmax threads

// Shared-memory plan for head dimension D and NQ verify columns.  P^T is always
// double-buffered: for NQ <= 32 the two buffers are the two halves of each 128-byte
// row of one region; for wider NQ they are two regions, paid for with one V stage.
template <int D, int NQ>
struct VCfg {
  static constexpr int kStagesK = (D == 128) ? 3 : 5;  // depth of the K ring
  static constexpr bool kSplitP = NQ <= 32;             // P buffers share 128-byte rows
  static constexpr int kStagesV = kSplitP ? kStagesK : kStagesK - 1;  // depth of the V ring
  static constexpr int kKVBytes = kTile * D * 2;      // K (or V) of one tile
  static constexpr int kHalfBytes = kTile * 128;      // 64-column half of a tile
  static constexpr int kQBytesMax = 64 * D * 2;
  static constexpr int kPRegion = kTile * 128;         // one 128 keys x 128 B region
  static constexpr int kPBytes = kSplitP ? kPRegion : 2 * kPRegion;
  static constexpr int kOffV = kStagesK * kKVBytes;
  static constexpr int kOffQ = kOffV + kStagesV * kKVBytes;
  static constexpr int kOffP = kOffQ + kQBytesMax;
  static constexpr int kOffMisc = kOffP + kPBytes;
  static constexpr int kMiscBytes = 1920;
  static constexpr int kSmemBytes = kOffMisc + kMiscBytes + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kOffP % 1024 == 0 && kOffQ % 1024 == 0, "swizzle atoms need 1 KB alignment");
};

struct VParams {
  const uint16_t* q;
  const int32_t* block_table;
  const int32_t* prefix_len;
  float* logits;
  float* partial;
  uint16_t* out;
  float* ws;
  unsigned* status;
  int B, Hq, Hkv, R, NV, max_blocks, num_blocks, P_max;
  int row0, row1;
  int collect_all;  // every verify row collected; partial sums over all rows
  const uint8_t* head_mask;  // [Hq] or NULL: only heads with a non-zero byte are collected
  float* score;              // fused aggregation outputs, or NULL (see VerifyArgs)
  uint32_t* hist;
  int hist_sink, hist_recent;  // the histogram skips the first / last positions
  int early;  // the K / V producers issue their first stages before the dependency wait
  // the verify block's keys / values ([B][R][Hkv][D]) stored into the cache at P_b ..
  // P_b + R - 1 by the producers before they copy those tiles (or null)
  const uint16_t* k_new;
  const uint16_t* v_new;
  uint16_t* k_store;
  uint16_t* v_store;
  int pairs, t_max, max_chunks;
  float scale;
};

constexpr int kHistBins = 4096;  // top 12 bits of the score keys

// CTA whose range holds virtual tile v (ranges are [c W / C, (c+1) W / C)).
__device__ __forceinline__ int cta_of(long long v, long long W, int C) {
  return static_cast<int>(((v + 1) * C - 1) / W);
}

struct Seg {
  int p, b, g;
  bool bad_len;        // prefix length outside the declared bounds (no key is read)
  int t_begin, t_end;  // tiles of this CTA inside the pair, clipped to the sequence
  int P, L;            // prefix length and cache length (P + R)
  long long next_v;
};

__device__ __forceinline__ Seg segment_at(long long v, long long v1, const VParams& a) {
  Seg s;
  s.p = static_cast<int>(v / a.t_max);
  const long long pair_end = static_cast<long long>(s.p + 1) * a.t_max;
  const long long e = v1 < pair_end ? v1 : pair_end;
  s.next_v = e;
  s.b = s.p / a.Hkv;
  s.g = s.p - s.b * a.Hkv;
  const int P = __ldcg(a.prefix_len + s.b);
  const bool ok = P >= 0 && P <= a.P_max &&
                  static_cast<long long>(P) + a.R <= static_cast<long long>(a.max_blocks) * kPage;
  s.bad_len = !ok;
  s.P = ok ? P : 0;
  s.L = ok ? P + a.R : 0;
  const int T = ok ? (s.L + kTile - 1) / kTile : 0;
  s.t_begin = static_cast<int>(v - static_cast<long long>(s.p) * a.t_max);
  const int te = static_cast<int>(e - static_cast<long long>(s.p) * a.t_max);
  s.t_end = te < T ? te : T;
  if (s.t_end < s.t_begin) s.t_end = s.t_begin;
  return s;
}

__device__ __forceinline__ bool softmax_vote(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "n"(kSoftmaxBar), "n"(kSoftmaxThreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void softmax_sync() {
  named_barrier_sync(kSoftmaxBar, kSoftmaxThreads);
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <int D, int NQ, int G>
__global__ void __launch_bounds__(kThreads, 1)
    verify_attn_collect_kernel(const __grid_constant__ CUtensorMap kmap,
                               const __grid_constant__ CUtensorMap vmap, const VParams a) {
  using Cfg = VCfg<D, NQ>;
  constexpr int SK = Cfg::kStagesK;
  constexpr int SV = Cfg::kStagesV;
  constexpr int NC = NQ / 2;  // columns per softmax thread
  constexpr int PB = 2;       // P^T buffers
  static_assert(NQ % 16 == 0 && NQ <= 64, "NQ");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* k_ring = base;
  uint8_t* v_ring = base + Cfg::kOffV;
  uint8_t* q_smem = base + Cfg::kOffQ;
  uint8_t* p_smem = base + Cfg::kOffP;
  uint8_t* misc = base + Cfg::kOffMisc;
  uint64_t* k_full = reinterpret_cast<uint64_t*>(misc);
  uint64_t* k_empty = k_full + SK;
  uint64_t* v_full = k_empty + SK;
  uint64_t* v_empty = v_full + SV;
  uint64_t* s_full = v_empty + SV;    // [2]
  uint64_t* s_empty = s_full + 2;     // [2]
  uint64_t* p_full = s_empty + 2;     // [2]
  uint64_t* pv_done = p_full + 2;     // [2]
  uint64_t* q_ready = pv_done + 2;
  uint64_t* mma_fin = q_ready + 1;    // every product of the issuer complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 260);
  float* m2s = reinterpret_cast<float*>(misc + 320);              // [64] new running max
  float* red = reinterpret_cast<float*>(misc + 576);              // [4][64] reductions
  float* alphas = reinterpret_cast<float*>(misc + 1600);          // [64] rescale factors

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < SV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], kSoftmaxThreads);
      mbar_init(&p_full[i], kSoftmaxThreads);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(q_ready, kSoftmaxThreads);
    mbar_init(mma_fin, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Inputs may come from the preceding kernel on the stream: every warp waits for it
  // here, except in the early mode the two producers, which wait once they have issued
  // their first stages of tiles wholly inside the prefix (below).
  const bool producer = warp == 0 || warp == kVWarp;
  if (!(producer && a.early)) {
    pdl_wait_primary();
    pdl_launch_dependents();
  }
  if (a.hist != nullptr && !producer) {
    // the aggregation in the merge kernel adds into a zeroed histogram (zeroed by the
    // warps between the producers, after their wait)
    constexpr int kZeroThreads = kThreads - 64;
    for (int i = blockIdx.x * kZeroThreads + threadIdx.x - 32; i < a.B * kHistBins;
         i += gridDim.x * kZeroThreads)
      a.hist[i] = 0u;
  }
  const uint32_t tmem_s0 = tmem;       // S^T buffer b: columns [64 b, 64 b + NQ)
  const uint32_t tmem_o = tmem + 128;  // O^T: columns [128, 128 + NQ)

  const long long W = static_cast<long long>(a.pairs) * a.t_max;
  const int C = gridDim.x;
  const long long v0 = static_cast<long long>(blockIdx.x) * W / C;
  const long long v1 = static_cast<long long>(blockIdx.x + 1) * W / C;

  auto set_abort = [&]() {
    if (!*abort_flag) {
      *abort_flag = 1;
      flag_status(a.status, VSD_DEV_TIMEOUT);
    }
  };

  if (warp == 0 || warp == kVWarp) {
    // ------------------------------------------------------------ TMA producers
    // warp 0 streams the K tiles, warp 10 the V tiles, each through its own ring, so
    // a K stage is refilled as soon as its QK MMA has read it.
    const bool is_k = warp == 0;
    const CUtensorMap* map = is_k ? &kmap : &vmap;
    uint8_t* ring = is_k ? k_ring : v_ring;
    uint64_t* full = is_k ? k_full : v_full;
    uint64_t* empty = is_k ? k_empty : v_empty;
    const int S = is_k ? SK : SV;  // depth of this warp's ring
    const uint64_t pol = l2_policy_evict_first();
    if (lane == 0) tma_prefetch_desc(map);
    uint32_t it = 0, issued = 0;
    // In the early mode the first S tiles are issued before the dependency wait when
    // they lie wholly inside the prefix (the preceding kernel may write the verify
    // block's rows, at P and beyond; the block table, the prefix lengths and the rows
    // below P are the caller's promise)
    bool waited = a.early == 0;
    for (long long v = v0; v < v1;) {
      // Block-table entries come 4 tiles (32 pages, one per lane) per load round and
      // two rounds ahead; the first two rounds are issued together with the prefix
      // length load, so the first copies leave one memory latency after the start.
      const int p0 = static_cast<int>(v / a.t_max);
      const int b0 = p0 / a.Hkv;
      const int tb0 = static_cast<int>(v - static_cast<long long>(p0) * a.t_max);
      const int32_t* bt_row = a.block_table + static_cast<size_t>(b0) * a.max_blocks;
      auto raw_entry = [&](int tile_base) {
        const int lp = (tile_base + (lane >> 3)) * kPagesPerTile + (lane & 7);
        return lp < a.max_blocks ? __ldcg(bt_row + lp) : a.num_blocks;
      };
      int ent_cur = raw_entry(tb0);
      int ent_nxt = raw_entry(tb0 + 4);
      const Seg s = segment_at(v, v1, a);
      v = s.next_v;
      if (is_k && s.bad_len && lane == 0) flag_status(a.status, VSD_DEV_BAD_LENGTH);
      for (int tile = s.t_begin; tile < s.t_end; ++tile, ++it) {
        const int k4 = (tile - s.t_begin) & 3;
        if (k4 == 0 && tile != s.t_begin) {
          ent_cur = ent_nxt;
          ent_nxt = raw_entry(tile + 4);  // in flight during the next 4 tiles
        }
        // block id of page `lane` (lanes 0-7) of this tile; outside the sequence or
        // invalid -> an out-of-range block, which the copy fills with zeros
        const int e = __shfl_sync(0xffffffffu, ent_cur, k4 * 8 + (lane & 7));
        const int lp = tile * kPagesPerTile + (lane & 7);
        const bool inside = lane < kPagesPerTile && lp * kPage < s.L;
        const bool bad = inside && (e < 0 || e >= a.num_blocks);
        const int blk = (inside && !bad) ? e : a.num_blocks;
        if (!waited && (it >= static_cast<uint32_t>(S) || (tile + 1) * kTile > s.P)) {
          pdl_wait_primary();
          pdl_launch_dependents();
          waited = true;
        }
        const int stage = it % S;
        const uint32_t use = it / S;
        int ok = 1;
        if (lane == 0 && use > 0) ok = mbar_wait(&empty[stage], (use - 1) & 1, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok && lane == 0) set_abort();
        if (*abort_flag) continue;
        if (a.k_new != nullptr) {
          // the verify block's rows in this tile join the cache first (after the wait:
          // the preceding kernel may write them), row u from lanes u * CPR .. on, then
          // the stores are ordered before the tensor copies of this tile
          const int r_lo = (s.P > tile * kTile ? s.P : tile * kTile) - s.P;
          const int r_end = s.P + a.R < (tile + 1) * kTile ? s.P + a.R : (tile + 1) * kTile;
          const int r_hi = r_end - s.P;
          if (r_lo < r_hi) {
            constexpr int CPR = D / 8;     // 16-byte chunks per row
            constexpr int RPW = 32 / CPR;  // rows per warp pass
            const uint16_t* src = is_k ? a.k_new : a.v_new;
            uint16_t* dstc = is_k ? a.k_store : a.v_store;
            for (int u0 = r_lo; u0 < r_hi; u0 += RPW) {
              const int u = u0 + lane / CPR, c = lane % CPR;
              const int pos = s.P + (u < r_hi ? u : r_lo);
              const int eb = __shfl_sync(0xffffffffu, blk, (pos >> 4) - tile * kPagesPerTile);
              if (u < r_hi && eb < a.num_blocks) {
                const uint4 val = *reinterpret_cast<const uint4*>(
                    src + ((static_cast<size_t>(s.b) * a.R + u) * a.Hkv + s.g) * D + c * 8);
                *reinterpret_cast<uint4*>(
                    dstc + ((static_cast<size_t>(eb) * a.Hkv + s.g) * kPage + (pos & (kPage - 1))) * D +
                    c * 8) = val;
              }
            }
            fence_proxy_async_all();
            __syncwarp();
          }
        }
        const unsigned badbits = __ballot_sync(0xffffffffu, bad);
        if (lane == 0) {
          if (is_k && badbits) flag_status(a.status, VSD_DEV_BAD_BLOCK);
          mbar_arrive_expect_tx(&full[stage], Cfg::kKVBytes);
        }
        __syncwarp();
        if (lane < kPagesPerTile) {
          uint8_t* dst = ring + stage * Cfg::kKVBytes + lane * (kPage * 128);
#pragma unroll
          for (int h = 0; h < D / 64; ++h)
            tma_load_4d(dst + h * Cfg::kHalfBytes, map, &full[stage], h * 64, 0, s.g, blk, pol);
        }
        issued = it + 1;
      }
    }
    if (!waited) {
      pdl_wait_primary();
      pdl_launch_dependents();
    }
    // Never leave a copy in flight: wait (with the drain limit) for the last stages.
    if (lane == 0) {
      const uint32_t first = issued > static_cast<uint32_t>(S) ? issued - S : 0;
      for (uint32_t i = first; i < issued; ++i) mbar_wait_drain(&full[i % S], (i / S) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, NQ, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, NQ, 1, 1);
      const uint32_t q_addr = smem_u32(q_smem);
      const uint32_t p_addr = smem_u32(p_smem);
      const uint32_t k_addr0 = smem_u32(k_ring);
      const uint32_t v_addr0 = smem_u32(v_ring);
      uint32_t total = 0;
      for (long long v = v0; v < v1;) {
        const Seg s = segment_at(v, v1, a);
        v = s.next_v;
        total += static_cast<uint32_t>(s.t_end - s.t_begin);
      }
      long long qv = v0;
      Seg qs = segment_at(qv, v1, a);
      int q_tile = qs.t_begin;
      uint32_t nseg = 0;
      uint32_t first_bits = 0;  // bit (i & 31): tile i is the first tile of its segment
      uint32_t qi = 0, pi = 0;
      const uint64_t t_start = global_timer_ns();
      uint32_t spins = 0;
      while (pi < total) {
        bool progressed = false;
        // ---- PV of tile pi (accumulates unless first of its segment)
        if (pi < qi && mbar_test(&p_full[pi % PB], (pi / PB) & 1) &&
            mbar_test(&v_full[pi % SV], (pi / SV) & 1)) {
          tc_fence_after();
          const int stage_i = static_cast<int>(pi % SV);
          const bool first_i = (first_bits >> (pi & 31)) & 1u;
          const uint32_t v_addr = v_addr0 + stage_i * Cfg::kKVBytes;
          const uint32_t pb_addr =
              p_addr + (pi % PB) * (Cfg::kSplitP ? 64u : static_cast<uint32_t>(Cfg::kPRegion));
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint64_t adesc = sdesc_sw128(v_addr + kk * 2048, Cfg::kHalfBytes, 1024);
            const uint64_t bdesc = sdesc_sw128(pb_addr + kk * 2048, Cfg::kHalfBytes, 1024);
            umma_bf16(tmem_o, adesc, bdesc, idesc_pv, (kk > 0 || !first_i) ? 1u : 0u);
          }
          umma_commit(&v_empty[stage_i]);
          umma_commit(&pv_done[pi % PB]);
          ++pi;
          progressed = true;
        }
        // ---- QK of tile qi (needs its K tile, a free S buffer, and Q of its segment)
        if (qi < total && qi < pi + 2) {
          while (q_tile >= qs.t_end) {  // advance to the next non-empty segment
            qv = qs.next_v;
            qs = segment_at(qv, v1, a);
            q_tile = qs.t_begin;
          }
          const bool first = q_tile == qs.t_begin;
          const int stage = static_cast<int>(qi % SK);
          const int buf = qi & 1;
          const bool ready = (!first || mbar_test(q_ready, nseg & 1)) &&
                             mbar_test(&k_full[stage], (qi / SK) & 1) &&
                             (qi < 2 || mbar_test(&s_empty[buf], ((qi >> 1) - 1) & 1));
          if (ready) {
            tc_fence_after();
            const uint32_t k_addr = k_addr0 + stage * Cfg::kKVBytes;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const int half = kk >> 2, w = kk & 3;
              const uint64_t adesc =
                  sdesc_sw128(k_addr + half * Cfg::kHalfBytes + w * 32, 16, 1024);
              const uint64_t bdesc = sdesc_sw128(q_addr + half * NQ * 128 + w * 32, 16, 1024);
              umma_bf16(tmem_s0 + buf * 64, adesc, bdesc, idesc_qk, kk > 0 ? 1u : 0u);
            }
            umma_commit(&k_empty[stage]);
            umma_commit(&s_full[buf]);
            if (first) {
              first_bits |= 1u << (qi & 31);
              ++nseg;
            } else {
              first_bits &= ~(1u << (qi & 31));
            }
            ++q_tile;
            ++qi;
            progressed = true;
          }
        }
        if (progressed) {
          spins = 0;
        } else {
          __nanosleep(32);
          if ((++spins & 63u) == 0 &&
              (*abort_flag || global_timer_ns() - t_start > VSD_WAIT_LIMIT_NS)) {
            set_abort();
            break;
          }
        }
      }
      // Never leave an MMA in flight: one more commit arrives once every product this
      // thread issued (QK ones after the last PV included) is done; wait for it with the
      // drain limit before the TMEM columns go back.
      umma_commit(mma_fin);
      mbar_wait_drain(mma_fin, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    const int sw = warp - 2;                   // 0..7
    const int quarter = warp & 3;              // TMEM lane quarter of this warp
    const int half = sw >> 2;                  // which NC columns of the row
    const int row = quarter * 32 + lane;       // key in tile (S^T) / dim (O^T)
    const int ts = threadIdx.x - 64;           // 0..255
    const int col0 = half * NC;                // first column of this thread
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const float scale = a.scale;
    const float scale_log2 = a.scale * kLog2e;
    const bool collect_any = a.logits != nullptr || a.partial != nullptr;
    constexpr bool kAllFits = NQ * D * 2 + 2 * kTile * 4 <= Cfg::kQBytesMax;
    const bool collect_all = kAllFits && collect_any && a.collect_all != 0;
    const bool collect = collect_any && !collect_all;  // the two chosen rows
    // all rows: the upper column half's per-key sums reach the lower half through
    // [2][kTile] floats after the Q rows (NQ <= 48 leaves that much of the area free)
    float* xsum = reinterpret_cast<float*>(q_smem + NQ * D * 2);
    // two rows: where that area exists the lower half writes row0 and the upper half
    // row1 (their sums meet there too), else the lower half writes both
    const bool split_collect = kAllFits && collect;
    uint32_t it = 0;
    for (long long v = v0; v < v1;) {
      // Loads that need no prefix length go out first: the segment's Q rows and this
      // thread's first block-table entry, then the length itself.
      const int p0 = static_cast<int>(v / a.t_max);
      const int b0 = p0 / a.Hkv, g0 = p0 - (p0 / a.Hkv) * a.Hkv;
      const int tb0 = static_cast<int>(v - static_cast<long long>(p0) * a.t_max);
      constexpr int kQL = (NQ * (D / 8) + kSoftmaxThreads - 1) / kSoftmaxThreads;
      uint4 qv[kQL];
#pragma unroll
      for (int u = 0; u < kQL; ++u) {
        const int idx = ts + u * kSoftmaxThreads;
        const int r = idx / (D / 8), ch = idx % (D / 8);
        qv[u] = make_uint4(0, 0, 0, 0);
        if (idx < NQ * (D / 8) && r < a.NV) {
          const int t = r / G, hl = r % G;
          qv[u] = *reinterpret_cast<const uint4*>(
              a.q + ((static_cast<size_t>(b0) * a.R + t) * a.Hq + g0 * G + hl) * D + ch * 8);
        }
      }
      const int lp0 = (tb0 * kTile + row) / kPage;
      const int entry_first =
          lp0 < a.max_blocks ? __ldcg(a.block_table + static_cast<size_t>(b0) * a.max_blocks + lp0)
                             : 0;
      const Seg s = segment_at(v, v1, a);
      v = s.next_v;
      // heads of this group whose logits are collected (all unless a mask is given)
      constexpr uint32_t kAllHeads = (G >= 32) ? 0xFFFFFFFFu : ((1u << G) - 1u);
      uint32_t gmask = kAllHeads;
      if (a.head_mask != nullptr) {
        gmask = 0u;
#pragma unroll
        for (int hl = 0; hl < G; ++hl)
          gmask |= (__ldcg(a.head_mask + s.g * G + hl) != 0 ? 1u : 0u) << hl;
      }
      const bool all_heads = gmask == kAllHeads;
      const long long first_v = static_cast<long long>(s.p) * a.t_max;
      const int c_first = cta_of(first_v, W, C);
      const int c_last = cta_of(first_v + a.t_max - 1, W, C);
      const bool direct = c_first == c_last;
      const int slot = s.p * a.max_chunks + (static_cast<int>(blockIdx.x) - c_first);
      const bool has_tiles = s.t_begin < s.t_end;
      float lacc[NC], m2[NC];
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        lacc[c] = 0.f;
        // padded columns get +inf: their probabilities are exp2(-inf) = 0 and they
        // never trigger a rescale
        m2[c] = (col0 + c < a.NV) ? -INFINITY : INFINITY;
      }

      if (has_tiles) {
        // Q rows of this (sequence, KV group): row r = t * G + hl -> q[b, t, g*G + hl, :]
#pragma unroll
        for (int u = 0; u < kQL; ++u) {
          const int idx = ts + u * kSoftmaxThreads;
          if (idx < NQ * (D / 8)) {
            const int r = idx / (D / 8), ch = idx % (D / 8);
            const int hh = ch >> 3, w = ch & 7;
            *reinterpret_cast<uint4*>(q_smem + hh * NQ * 128 + r * 128 + ((w ^ (r & 7)) << 4)) =
                qv[u];
          }
        }
        if (ts < 64) m2s[ts] = (ts < a.NV) ? -INFINITY : INFINITY;
        fence_proxy_async_smem();
        mbar_arrive(q_ready);
      }

      // block-table entry of this thread's key page, fetched one tile ahead (a page
      // outside [0, num_blocks) was zero-filled by the producer and is masked here)
      auto page_entry = [&](int tile) {
        const int jj = tile * kTile + row;
        return (tile < s.t_end && jj < s.L)
                   ? __ldcg(a.block_table + static_cast<size_t>(s.b) * a.max_blocks + jj / kPage)
                   : 0;
      };
      int entry_next =
          (s.t_begin < s.t_end && s.t_begin * kTile + row < s.L) ? entry_first : 0;
      for (int tile = s.t_begin; tile < s.t_end; ++tile, ++it) {
        const int stage = it % SV;  // V stage of this tile (masked rows are zeroed there)
        const int buf = it & 1;
        const int pb = it % PB;
        const int entry = entry_next;
        entry_next = page_entry(tile + 1);
        // (a test build waits on the issuer's end-of-kernel barrier for the first tile,
        // which nothing completes yet)
        if (!(VSD_STALL(it == 0) ? mbar_wait(mma_fin, 0, abort_flag)
                                 : mbar_wait(&s_full[buf], (it >> 1) & 1, abort_flag)))
          set_abort();
        const int j = tile * kTile + row;
        const bool want_collect = collect && !split_collect && half == 0 && j < s.P;
        tc_fence_after();
        const uint32_t s_addr = tmem_s0 + buf * 64 + lane_addr;
        float sv[NC];
        uint32_t c0raw[G], c1raw[G];
        tmem_ld_cols<NC>(s_addr + col0, reinterpret_cast<uint32_t*>(sv));
        if (split_collect) {
          // warp-uniform: each half reads its collected row
          tmem_ld<G>(s_addr + (half == 0 ? a.row0 : a.row1) * G, c0raw);
        } else if (collect && half == 0) {
          // warp-uniform: the lower-half warps read the two collected rows
          tmem_ld<G>(s_addr + a.row0 * G, c0raw);
          tmem_ld<G>(s_addr + a.row1 * G, c1raw);
        }
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&s_empty[buf]);

        // Collect-2-Query: logits of rows row0 / row1 and their group sum, j < P_b.
        // The per-head mask test is compiled in only for segments that have a mask (a
        // uniform branch): unmasked calls keep the loop of the plain collect.
        auto collect_row = [&](auto masked, const uint32_t* raw, int c, float& acc) {
#pragma unroll
          for (int hl = 0; hl < G; ++hl) {
            if constexpr (decltype(masked)::value) {
              if (!((gmask >> hl) & 1u)) continue;
            }
            const float z = __uint_as_float(raw[hl]) * scale;
            if (a.logits)
              __stcs(a.logits + ((static_cast<size_t>(s.b) * 2 + c) * a.Hq + s.g * G + hl) *
                                    a.P_max + j, z);
            acc += z;
          }
        };
        if (want_collect) {
          float acc = 0.f;
          if (all_heads) {
            collect_row(std::false_type{}, c0raw, 0, acc);
            collect_row(std::false_type{}, c1raw, 1, acc);
          } else {
            collect_row(std::true_type{}, c0raw, 0, acc);
            collect_row(std::true_type{}, c1raw, 1, acc);
          }
          if (a.partial) a.partial[(static_cast<size_t>(s.b) * a.Hkv + s.g) * a.P_max + j] = acc;
        }
        // all rows: every column of this thread, then the two halves' sums; two rows
        // split between the halves: this half's row, then the two halves' sums
        float call = 0.f;
        if (split_collect && j < s.P) {
          if (all_heads)
            collect_row(std::false_type{}, c0raw, half, call);
          else
            collect_row(std::true_type{}, c0raw, half, call);
          if (half == 1) xsum[(it & 1) * kTile + row] = call;
        }
        if (collect_all && j < s.P) {
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            const int cc = col0 + c;
            if (cc < a.NV && (all_heads || ((gmask >> (cc % G)) & 1u))) {
              const float z = sv[c] * scale;
              if (a.logits)
                __stcs(a.logits + ((static_cast<size_t>(s.b) * a.R + cc / G) * a.Hq + s.g * G +
                                   cc % G) * a.P_max + j, z);
              call += z;
            }
          }
          if (half == 1) xsum[(it & 1) * kTile + row] = call;
        }

        // d = y - m2 in log2 units (y = scaled logit); masks only where a key can be hidden
        const bool bad = entry < 0 || entry >= a.num_blocks;
        const bool masked = j >= s.P || bad;  // per key
        int c_lo = 0;                         // first visible column of this key
        if (masked) {
          const bool valid = j < s.L && !bad;
          c_lo = !valid ? NQ : (j - s.P) * G;
        }
        float dmax = -INFINITY;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const float d = fmaf(sv[c], scale_log2, -m2[c]);
          if (!masked || col0 + c >= c_lo) dmax = fmaxf(dmax, d);
        }
        const bool raise = softmax_vote(dmax > kTau);  // also orders the xsum stores
        if ((collect_all || split_collect) && half == 0 && j < s.P && a.partial)
          a.partial[(static_cast<size_t>(s.b) * a.Hkv + s.g) * a.P_max + j] =
              call + xsum[(it & 1) * kTile + row];
        if (raise) {
          // rare: some visible logit is far above its column's running max
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            const bool vis = !masked || col0 + c >= c_lo;
            const float x = warp_max(vis ? sv[c] * scale_log2 : -INFINITY);
            if (lane == 0) red[quarter * 64 + col0 + c] = x;
          }
          softmax_sync();
          if (ts < NQ) {
            const int c = ts;
            const float mx = fmaxf(fmaxf(red[c], red[64 + c]), fmaxf(red[128 + c], red[192 + c]));
            const float mo = m2s[c];
            const float mn = fmaxf(mo, mx);
            // -inf: nothing accumulated yet; +inf: padding column, never used
            alphas[c] = (mo == -INFINITY) ? 0.f : (mo == INFINITY ? 1.f : exp2f(mo - mn));
            m2s[c] = mn;
          }
          softmax_sync();
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            lacc[c] *= alphas[col0 + c];
            m2[c] = m2s[col0 + c];
          }
          if (tile != s.t_begin) {
            // O^T holds earlier tiles: rescale this thread's columns once the last PV is done
            if (!mbar_wait(&pv_done[(it - 1) % PB], ((it - 1) / PB) & 1, abort_flag)) set_abort();
            tc_fence_after();
            uint32_t r[NC];
            tmem_ld_cols<NC>(tmem_o + lane_addr + col0, r);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < NC; ++c)
              r[c] = __float_as_uint(__uint_as_float(r[c]) * alphas[col0 + c]);
            tmem_st_cols<NC>(tmem_o + lane_addr + col0, r);
            tmem_wait_st();
          }
        }
        // probabilities relative to the shared running max
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const bool vis = !masked || col0 + c >= c_lo;
          const float pc = vis ? exp2f(fmaf(sv[c], scale_log2, -m2[c])) : 0.f;
          lacc[c] += pc;
          sv[c] = pc;
        }
        // P^T buffer pb: the PV that last read it must be done
        if (it >= static_cast<uint32_t>(PB) &&
            !mbar_wait(&pv_done[pb], ((it - PB) / PB) & 1, abort_flag))
          set_abort();
        if (j >= s.L) {
          // rows past the sequence end hold whatever the cache holds: zero V there once
          // the tile has landed (each half of the pair zeroes one 64-column half)
          if (!mbar_wait(&v_full[stage], (it / SV) & 1, abort_flag)) set_abort();
          if (half < D / 64) {
            uint8_t* vrow = v_ring + stage * Cfg::kKVBytes + half * Cfg::kHalfBytes + row * 128;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
              *reinterpret_cast<uint4*>(vrow + ch * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        uint8_t* prow = p_smem + (Cfg::kSplitP ? 0 : pb * Cfg::kPRegion) + row * 128;
#pragma unroll
        for (int k = 0; k < NC / 8; ++k) {
          // split rows: buffer 1 starts 32 elements in; else each buffer has its region
          const int ch = (Cfg::kSplitP ? pb * 4 : 0) + col0 / 8 + k;
          uint4 pk;
          pk.x = pack_bf16x2(sv[k * 8 + 0], sv[k * 8 + 1]);
          pk.y = pack_bf16x2(sv[k * 8 + 2], sv[k * 8 + 3]);
          pk.z = pack_bf16x2(sv[k * 8 + 4], sv[k * 8 + 5]);
          pk.w = pack_bf16x2(sv[k * 8 + 6], sv[k * 8 + 7]);
          *reinterpret_cast<uint4*>(prow + ((ch ^ (row & 7)) << 4)) = pk;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&p_full[pb]);
      }

      // ---------------------------------------------------------- pair epilogue
      const size_t slot_base = static_cast<size_t>(slot) * NQ * (D + 2);
      if (has_tiles) {
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const float x = warp_sum(lacc[c]);
          if (lane == 0) red[quarter * 64 + col0 + c] = x;
        }
        softmax_sync();
        if (!mbar_wait(&pv_done[(it - 1) % PB], ((it - 1) / PB) & 1, abort_flag)) set_abort();
        tc_fence_after();
        float o[NC];
        tmem_ld_cols<NC>(tmem_o + lane_addr + col0, reinterpret_cast<uint32_t*>(o));
        tmem_wait_ld();
        tc_fence_before();
        if (row < D) {
          const int dim = row;
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            const int cc = col0 + c;
            if (cc < a.NV) {
              if (direct) {
                const float l = red[cc] + red[64 + cc] + red[128 + cc] + red[192 + cc];
                const int t = cc / G, hl = cc % G;
                const float val = l > 0.f ? o[c] / l : 0.f;
                const __nv_bfloat16 bv = __float2bfloat16_rn(val);
                a.out[((static_cast<size_t>(s.b) * a.R + t) * a.Hq + s.g * G + hl) * D + dim] =
                    *reinterpret_cast<const uint16_t*>(&bv);
              } else {
                a.ws[slot_base + 2 * NQ + static_cast<size_t>(cc) * D + dim] = o[c];
              }
            }
          }
        }
        if (!direct && quarter == 0 && lane == 0) {
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            const int cc = col0 + c;
            a.ws[slot_base + cc] = m2[c];
            a.ws[slot_base + NQ + cc] = red[cc] + red[64 + cc] + red[128 + cc] + red[192 + cc];
          }
        }
        softmax_sync();
      } else {
        // no key of this pair in this CTA: an empty partial (or zeros when alone)
        if (direct) {
          for (int idx = ts; idx < a.NV * D; idx += kSoftmaxThreads) {
            const int c = idx / D, dim = idx % D;
            const int t = c / G, hl = c % G;
            a.out[((static_cast<size_t>(s.b) * a.R + t) * a.Hq + s.g * G + hl) * D + dim] = 0;
          }
        } else {
          if (ts < NQ) {
            a.ws[slot_base + ts] = -INFINITY;
            a.ws[slot_base + NQ + ts] = 0.f;
          }
          for (int idx = ts; idx < NQ * D; idx += kSoftmaxThreads) a.ws[slot_base + 2 * NQ + idx] = 0.f;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// Fused aggregation (blocks past the merge blocks): 4 * D consecutive positions of one
// sequence per block, 4 per thread.  The score of position j is the sum of its
// per-group partials in group order (fp32, starting from zero: the same sum, in the
// same order, as the selection kernel forms); the block counts the top 12 bits of the
// scores' order-preserving keys in shared memory and adds its non-zero bins to the
// sequence's histogram.
template <int D>
__device__ __forceinline__ void aggregate_scores(const VParams& a, int blk) {
  constexpr int kPos = 4 * D;
  __shared__ uint32_t h[kHistBins];
  const int per_seq = (a.P_max + kPos - 1) / kPos;
  const int b = blk / per_seq;
  const int j0 = (blk - b * per_seq) * kPos + static_cast<int>(threadIdx.x) * 4;
  for (int i = threadIdx.x; i < kHistBins; i += D) h[i] = 0u;
  // the partials are loaded before the prefix length arrives (every position below
  // P_max is valid memory); positions at or past P_b are masked afterwards
  float s[4] = {0.f, 0.f, 0.f, 0.f};
  if (j0 < a.P_max) {
    const float* base = a.partial + static_cast<size_t>(b) * a.Hkv * a.P_max + j0;
    if ((a.P_max & 3) == 0) {
      int g = 0;
      for (; g + 8 <= a.Hkv; g += 8) {
        float4 x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          x[u] = __ldcg(reinterpret_cast<const float4*>(base + static_cast<size_t>(g + u) * a.P_max));
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          s[0] += x[u].x;
          s[1] += x[u].y;
          s[2] += x[u].z;
          s[3] += x[u].w;
        }
      }
      for (; g < a.Hkv; ++g) {
        const float4 x = __ldcg(reinterpret_cast<const float4*>(base + static_cast<size_t>(g) * a.P_max));
        s[0] += x.x;
        s[1] += x.y;
        s[2] += x.z;
        s[3] += x.w;
      }
    } else {
      for (int g = 0; g < a.Hkv; ++g)
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (j0 + u < a.P_max) s[u] += __ldcg(base + static_cast<size_t>(g) * a.P_max + u);
    }
  }
  const int P = __ldcg(a.prefix_len + b);
  const bool ok = P >= 0 && P <= a.P_max;  // else flagged by the verification kernel
  __syncthreads();
  if (ok) {
    // the histogram counts the selection's candidates only: the sinks and the recent
    // window (as the selection clamps them) are left out
    const int c_lo = a.hist_sink < P ? a.hist_sink : P;
    const int c_hi = P - a.hist_recent > c_lo ? P - a.hist_recent : c_lo;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = j0 + u;
      if (j < P) {
        a.score[static_cast<size_t>(b) * a.P_max + j] = s[u];
        const uint32_t bits = __float_as_uint(s[u]);
        const uint32_t key = (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
        if (j >= c_lo && j < c_hi) atomicAdd(&h[key >> 20], 1u);
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kHistBins; i += D)
    if (h[i] != 0u) atomicAdd(a.hist + static_cast<size_t>(b) * kHistBins + i, h[i]);
}

// Combine the partial (m, l, o) of the CTAs that shared a pair: block (pair, verify
// row c), thread = dim.  Each block issues the loads of up to kU partials at once and
// combines them in chunk order: kU = 32 where a pair is spread over many CTAs (one
// sequence: ~C / Hkv), kU = 8 where it meets at most 8 (a batch of sequences), which
// keeps the kernel's registers low enough for ten blocks per SM instead of four (the
// 36-layer decode loop's 1280 merge and aggregation blocks took 2.1 waves).
// One flat grid: blocks [0, merge_pairs * NV) merge (pair, verify row); with kAgg the
// rest are the fused-aggregation blocks (only that variant carries their 16 KB of
// shared memory).
template <int D, int NQ, int G, bool kAgg, int kU>
__global__ void __launch_bounds__(D) verify_merge_kernel(const VParams a, int ctas,
                                                         int merge_pairs) {
  const int x = blockIdx.x;
  const int dim = threadIdx.x;
  pdl_wait_primary();  // partials of the verification kernel are complete
  pdl_launch_dependents();
  if (x >= merge_pairs * a.NV) {
    if constexpr (kAgg) aggregate_scores<D>(a, x - merge_pairs * a.NV);
    return;
  }
  const int p = x / a.NV;
  const int c = x - p * a.NV;
  const long long W = static_cast<long long>(a.pairs) * a.t_max;
  const long long first_v = static_cast<long long>(p) * a.t_max;
  const int c_first = cta_of(first_v, W, ctas);
  const int c_last = cta_of(first_v + a.t_max - 1, W, ctas);
  if (c_first == c_last) return;
  const int n = c_last - c_first + 1;
  const size_t stride = static_cast<size_t>(NQ) * (D + 2);
  const float* base = a.ws + static_cast<size_t>(p) * a.max_chunks * stride;
  float M = -INFINITY, L = 0.f, O = 0.f;
  for (int k0 = 0; k0 < n; k0 += kU) {
    float mk[kU], lk[kU], ok[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (k0 + u < n) {
        const float* sl = base + (k0 + u) * stride;
        mk[u] = __ldcg(sl + c);
        lk[u] = __ldcg(sl + NQ + c);
        ok[u] = __ldcg(sl + 2 * NQ + static_cast<size_t>(c) * D + dim);
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
    L *= sc;
    O *= sc;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const float w = (mk[u] == -INFINITY) ? 0.f : exp2f(mk[u] - mn);
      L += w * lk[u];
      O += w * ok[u];
    }
    M = mn;
  }
  const int b = p / a.Hkv, g = p - (p / a.Hkv) * a.Hkv;
  const int t = c / G, hl = c % G;
  const __nv_bfloat16 bv = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
  a.out[((static_cast<size_t>(b) * a.R + t) * a.Hq + g * G + hl) * D + dim] =
      *reinterpret_cast<const uint16_t*>(&bv);
}

template <int D, int NQ, int G>
cudaError_t launch_dng(const VerifyArgs& va, const VerifyPlan& plan, const VParams& p,
                       cudaStream_t stream) {
  auto kern = verify_attn_collect_kernel<D, NQ, G>;
  constexpr int smem = VCfg<D, NQ>::kSmemBytes;
  // set on every call: the attribute is per device and the call costs no GPU work
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // Both kernels are programmatic dependents of their predecessor on the stream:
  // their launch and prologue overlap it, and they wait for its results before
  // reading any input.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.ctas, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, va.kmap, va.vmap, p);
  // merge blocks for pairs cut by CTA boundaries, then the fused-aggregation blocks
  const int merge_pairs = plan.max_chunks > 1 ? plan.pairs : 0;
  const int agg = p.score != nullptr ? p.B * ((p.P_max + 4 * D - 1) / (4 * D)) : 0;
  if (e != cudaSuccess || merge_pairs + agg == 0) return e;
  cfg.gridDim = dim3(merge_pairs * p.NV + agg, 1, 1);
  cfg.blockDim = dim3(D, 1, 1);
  cfg.dynamicSmemBytes = 0;
  const bool few = plan.max_chunks <= 8;  // partials per pair: one round of 8 loads
  if (agg > 0)
    return few ? cudaLaunchKernelEx(&cfg, verify_merge_kernel<D, NQ, G, true, 8>, p, plan.ctas,
                                    merge_pairs)
               : cudaLaunchKernelEx(&cfg, verify_merge_kernel<D, NQ, G, true, 32>, p, plan.ctas,
                                    merge_pairs);
  return few ? cudaLaunchKernelEx(&cfg, verify_merge_kernel<D, NQ, G, false, 8>, p, plan.ctas,
                                  merge_pairs)
             : cudaLaunchKernelEx(&cfg, verify_merge_kernel<D, NQ, G, false, 32>, p, plan.ctas,
                                  merge_pairs);
}

inline VParams make_params(const VerifyArgs& va, const VerifyPlan& plan) {
  VParams p;
  p.q = static_cast<const uint16_t*>(va.q);
  p.block_table = va.block_table;
  p.prefix_len = va.prefix_len;
  p.logits = va.logits;
  p.partial = va.partial;
  p.out = static_cast<uint16_t*>(va.out);
  p.ws = va.ws;
  p.status = va.status;
  p.B = va.B;
  p.Hq = va.Hq;
  p.Hkv = va.Hkv;
  p.R = va.R;
  p.NV = va.R * va.G;
  p.max_blocks = va.max_blocks;
  p.num_blocks = va.num_blocks;
  p.P_max = va.P_max;
  p.row0 = va.row0;
  p.row1 = va.row1;
  p.collect_all = va.collect_all;
  p.head_mask = va.head_mask;
  p.score = va.score;
  p.hist = va.hist;
  p.hist_sink = va.hist_sink;
  p.early = va.early;
  p.k_new = static_cast<const uint16_t*>(va.k_new);
  p.v_new = static_cast<const uint16_t*>(va.v_new);
  p.k_store = static_cast<uint16_t*>(va.k_store);
  p.v_store = static_cast<uint16_t*>(va.v_store);
  p.hist_recent = va.hist_recent;
  p.pairs = plan.pairs;
  p.t_max = plan.t_max;
  p.max_chunks = plan.max_chunks;
  p.scale = va.scale;
  return p;
}

// Dispatch over (G, NQ) for one head dimension.
template <int D>
cudaError_t launch_verify_d(const VerifyArgs& va, const VerifyPlan& plan, cudaStream_t stream) {
  const VParams p = make_params(va, plan);
#define VSD_VERIFY_CASE(GG, NN) \
  if (va.G == GG && plan.nq == NN) return launch_dng<D, NN, GG>(va, plan, p, stream);
  VSD_VERIFY_CASE(1, 16)
  VSD_VERIFY_CASE(2, 16)
  VSD_VERIFY_CASE(2, 32)
  VSD_VERIFY_CASE(4, 16)
  VSD_VERIFY_CASE(4, 32)
  VSD_VERIFY_CASE(4, 48)
  VSD_VERIFY_CASE(4, 64)
  VSD_VERIFY_CASE(8, 16)
  VSD_VERIFY_CASE(8, 32)
  VSD_VERIFY_CASE(8, 48)
  VSD_VERIFY_CASE(8, 64)
  VSD_VERIFY_CASE(16, 16)
  VSD_VERIFY_CASE(16, 32)
  VSD_VERIFY_CASE(16, 48)
  VSD_VERIFY_CASE(16, 64)
#undef VSD_VERIFY_CASE
  return cudaErrorInvalidValue;
}

}  // namespace verify_detail
}  // namespace vsd
