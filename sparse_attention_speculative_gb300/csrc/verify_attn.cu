// verify_attn.cu -- verification attention with Collect-2-Query on sm_103a.
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
//     of that list, so every SM gets the same number of tiles ("split-K" over the
//     context, balanced to the tile).  A pair cut by CTA boundaries leaves one
//     partial (m, l, o) per CTA, combined by a small merge kernel.
//   * Warp 0 streams K and V pages with 4-D TMA loads (128-byte swizzle) into a
//     3-stage shared-memory ring (5 stages for head_dim 64).  Each 128-key tile is
//     8 pages; a page whose block-table entry is invalid is fetched at an
//     out-of-range coordinate, which the TMA unit fills with zeros.
//   * Warp 1 issues tcgen05 MMAs with the small dimension moved to N ("swap AB"):
//       S^T[128 keys x NQ] = K_tile[128 x d] * Q^T        (K-major A and B)
//       O^T[d x NQ]       += V_tile^T[d x 128] * P^T      (MN-major A and B)
//     where NQ = R*G rounded up to 16 covers all verify rows of one KV group, so the
//     tensor cores do no padding work beyond that rounding.  Accumulators live in
//     TMEM (S double-buffered, O single).
//   * Warps 2-5 own one key each (TMEM lane = key): they read the key's NQ logits,
//     store the collected rows' logits and the group sum with coalesced stores
//     (32 consecutive keys per warp), and form P for the online softmax.  The
//     running maximum is shared by all keys of a column; it is only raised when
//     some logit exceeds it by more than 2^8 (one vote per tile), which keeps
//     exp2 arguments bounded while the common path needs no cross-thread max.
//     Each thread keeps its own partial row sums l; they are reduced once per pair.
#include <cfloat>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace vsd {
namespace {

using namespace ptx;

constexpr int kTile = 128;          // keys per tile (the MMA M dimension of S^T)
constexpr int kPage = 16;           // tokens per cache page
constexpr int kPagesPerTile = kTile / kPage;
constexpr float kTau = 8.0f;        // lazy-max slack, log2 units
constexpr int kThreads = 192;       // producer warp, MMA warp, 4 softmax warps
constexpr int kSoftmaxBar = 1;      // named barrier of the 128 softmax threads

template <int D>
struct VCfg {
  static constexpr int kStages = (D == 128) ? 3 : 5;
  static constexpr int kKVBytes = kTile * D * 2;           // one of K or V of a tile
  static constexpr int kStageBytes = 2 * kKVBytes;
  static constexpr int kHalfBytes = kTile * 128;           // 64-column half of a tile
  static constexpr int kQBytesMax = 64 * D * 2;
  static constexpr int kPBytes = kTile * 128;
  static constexpr int kOffQ = kStages * kStageBytes;
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
  int B, Hq, Hkv, G, lgG, R, NV, max_blocks, num_blocks, P_max;
  int row0, row1;
  int pairs, t_max, max_chunks;
  float scale;
};

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
  const int P = __ldg(a.prefix_len + s.b);
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

__device__ __forceinline__ bool bar_red_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "n"(kSoftmaxBar)
      : "memory");
  return r != 0;
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

template <int D, int NQ>
__global__ void __launch_bounds__(kThreads, 1)
    verify_attn_collect_kernel(const __grid_constant__ CUtensorMap kmap,
                               const __grid_constant__ CUtensorMap vmap, const VParams a) {
  using Cfg = VCfg<D>;
  constexpr int S = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* q_smem = base + Cfg::kOffQ;
  uint8_t* p_smem = base + Cfg::kOffP;
  uint8_t* misc = base + Cfg::kOffMisc;
  uint64_t* kv_full = reinterpret_cast<uint64_t*>(misc);
  uint64_t* kv_empty = kv_full + S;
  uint64_t* s_full = kv_empty + S;    // [2]
  uint64_t* s_empty = s_full + 2;     // [2]
  uint64_t* p_full = s_empty + 2;
  uint64_t* pv_done = p_full + 1;
  uint64_t* q_ready = pv_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 260);
  uint32_t* badmask = reinterpret_cast<uint32_t*>(misc + 272);  // [S]
  float* m2s = reinterpret_cast<float*>(misc + 320);              // [64] running max (log2)
  float* red = reinterpret_cast<float*>(misc + 576);              // [4][64] reductions
  float* alphas = reinterpret_cast<float*>(misc + 1600);          // [64] rescale factors

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 128);
    }
    mbar_init(p_full, 128);
    mbar_init(pv_done, 1);
    mbar_init(q_ready, 128);
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
  const uint32_t tmem_s0 = tmem;         // S^T buffer 0: columns [0, NQ)
  const uint32_t tmem_o = tmem + 128;    // O^T: columns [128, 128 + NQ)

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

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    const uint64_t pol = l2_policy_evict_first();
    if (lane == 0) {
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
    }
    uint32_t it = 0, issued = 0;
    for (long long v = v0; v < v1;) {
      const Seg s = segment_at(v, v1, a);
      v = s.next_v;
      if (s.bad_len && lane == 0) flag_status(a.status, VSD_DEV_BAD_LENGTH);
      for (int tile = s.t_begin; tile < s.t_end; ++tile, ++it) {
        const int stage = it % S;
        const uint32_t use = it / S;
        int ok = 1;
        if (lane == 0 && use > 0) ok = mbar_wait(&kv_empty[stage], (use - 1) & 1, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok && lane == 0) set_abort();
        if (*abort_flag) continue;
        int blk = a.num_blocks;  // out of range: the TMA unit fills zeros
        bool bad = false;
        if (lane < kPagesPerTile) {
          const int lp = tile * kPagesPerTile + lane;
          if (lp * kPage < s.L) {
            const int e = __ldg(a.block_table + static_cast<size_t>(s.b) * a.max_blocks + lp);
            if (e < 0 || e >= a.num_blocks) bad = true;
            else blk = e;
          }
        }
        const unsigned badbits = __ballot_sync(0xffffffffu, bad);
        if (lane == 0) {
          if (badbits) flag_status(a.status, VSD_DEV_BAD_BLOCK);
          badmask[stage] = badbits;
          mbar_arrive_expect_tx(&kv_full[stage], Cfg::kStageBytes);
        }
        __syncwarp();
        if (lane < kPagesPerTile) {
          uint8_t* kdst = base + stage * Cfg::kStageBytes + lane * (kPage * 128);
          uint8_t* vdst = kdst + Cfg::kKVBytes;
#pragma unroll
          for (int h = 0; h < D / 64; ++h) {
            tma_load_4d(kdst + h * Cfg::kHalfBytes, &kmap, &kv_full[stage], h * 64, 0, s.g, blk,
                        pol);
            tma_load_4d(vdst + h * Cfg::kHalfBytes, &vmap, &kv_full[stage], h * 64, 0, s.g, blk,
                        pol);
          }
        }
        issued = it + 1;
      }
    }
    // Never leave a copy in flight: wait (bounded) for the last stages issued.
    if (lane == 0) {
      const uint32_t first = issued > static_cast<uint32_t>(S) ? issued - S : 0;
      for (uint32_t i = first; i < issued; ++i) mbar_wait(&kv_full[i % S], (i / S) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, NQ, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, NQ, 1, 1);
      const uint32_t q_addr = smem_u32(q_smem);
      const uint32_t p_addr = smem_u32(p_smem);
      const uint32_t ring = smem_u32(base);
      uint32_t it = 0, nseg = 0, pv_issued = 0;
      bool have_prev = false, prev_first = false;
      int prev_stage = 0;
      auto issue_pv = [&](uint32_t i, int stage_i, bool first_i) {
        if (!mbar_wait(p_full, i & 1, abort_flag)) set_abort();
        if (*abort_flag) return;
        tc_fence_after();
        const uint32_t v_addr = ring + stage_i * Cfg::kStageBytes + Cfg::kKVBytes;
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint64_t adesc = sdesc_sw128(v_addr + kk * 2048, Cfg::kHalfBytes, 1024);
          const uint64_t bdesc = sdesc_sw128(p_addr + kk * 2048, Cfg::kHalfBytes, 1024);
          umma_bf16(tmem_o, adesc, bdesc, idesc_pv, (kk > 0 || !first_i) ? 1u : 0u);
        }
        umma_commit(&kv_empty[stage_i]);
        umma_commit(pv_done);
        pv_issued = i + 1;
      };
      for (long long v = v0; v < v1;) {
        const Seg s = segment_at(v, v1, a);
        v = s.next_v;
        if (s.t_begin >= s.t_end) continue;
        for (int tile = s.t_begin; tile < s.t_end; ++tile, ++it) {
          const bool first = tile == s.t_begin;
          const int stage = it % S;
          const int buf = it & 1;
          if (first && have_prev) {
            issue_pv(it - 1, prev_stage, prev_first);
            have_prev = false;
          }
          bool ok = true;
          if (first) ok = mbar_wait(q_ready, nseg & 1, abort_flag);
          ok = ok && mbar_wait(&kv_full[stage], (it / S) & 1, abort_flag);
          if (it >= 2) ok = ok && mbar_wait(&s_empty[buf], ((it >> 1) - 1) & 1, abort_flag);
          if (!ok) set_abort();
          if (!*abort_flag) {
            tc_fence_after();
            const uint32_t k_addr = ring + stage * Cfg::kStageBytes;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const int half = kk >> 2, w = kk & 3;
              const uint64_t adesc =
                  sdesc_sw128(k_addr + half * Cfg::kHalfBytes + w * 32, 16, 1024);
              const uint64_t bdesc = sdesc_sw128(q_addr + half * NQ * 128 + w * 32, 16, 1024);
              umma_bf16(tmem_s0 + buf * 64, adesc, bdesc, idesc_qk, kk > 0 ? 1u : 0u);
            }
            umma_commit(&s_full[buf]);
          }
          if (have_prev) issue_pv(it - 1, prev_stage, prev_first);
          have_prev = true;
          prev_stage = stage;
          prev_first = first;
        }
        ++nseg;
      }
      if (have_prev) issue_pv(it - 1, prev_stage, prev_first);
      // Never leave an MMA in flight: wait (bounded) for the last PV issued.
      if (pv_issued > 0) mbar_wait(pv_done, (pv_issued - 1) & 1);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    const int quarter = warp & 3;                 // TMEM lane quarter of this warp
    const int row = quarter * 32 + lane;          // key in tile (S^T) / dim (O^T)
    const int sw = warp - 2;                      // 0..3
    const int ts = threadIdx.x - 64;              // 0..127
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const float scale = a.scale;
    const float scale_log2 = a.scale * kLog2e;
    const bool collect = a.logits != nullptr || a.partial != nullptr;
    uint32_t it = 0, nseg = 0;
    for (long long v = v0; v < v1;) {
      const Seg s = segment_at(v, v1, a);
      v = s.next_v;
      const long long first_v = static_cast<long long>(s.p) * a.t_max;
      const int c_first = cta_of(first_v, W, C);
      const int c_last = cta_of(first_v + a.t_max - 1, W, C);
      const bool direct = c_first == c_last;
      const int slot = s.p * a.max_chunks + (static_cast<int>(blockIdx.x) - c_first);
      const bool has_tiles = s.t_begin < s.t_end;
      float lacc[NQ];
#pragma unroll
      for (int c = 0; c < NQ; ++c) lacc[c] = 0.f;

      if (has_tiles) {
        // Q rows of this (sequence, KV group): row c = t * G + hl -> q[b, t, g*G + hl, :]
        for (int idx = ts; idx < NQ * (D / 8); idx += 128) {
          const int r = idx / (D / 8), ch = idx % (D / 8);
          uint4 val = make_uint4(0, 0, 0, 0);
          if (r < a.NV) {
            const int t = r >> a.lgG, hl = r & (a.G - 1);
            val = *reinterpret_cast<const uint4*>(
                a.q + ((static_cast<size_t>(s.b) * a.R + t) * a.Hq + s.g * a.G + hl) * D + ch * 8);
          }
          const int half = ch >> 3, w = ch & 7;
          *reinterpret_cast<uint4*>(q_smem + half * NQ * 128 + r * 128 + ((w ^ (r & 7)) << 4)) =
              val;
        }
        fence_proxy_async_smem();
        mbar_arrive(q_ready);
        if (ts < 64) m2s[ts] = -INFINITY;
        named_barrier_sync(kSoftmaxBar, 128);
        ++nseg;
      }

      for (int tile = s.t_begin; tile < s.t_end; ++tile, ++it) {
        const int stage = it % S;
        const int buf = it & 1;
        bool ok = mbar_wait(&kv_full[stage], (it / S) & 1, abort_flag);
        ok = ok && mbar_wait(&s_full[buf], (it >> 1) & 1, abort_flag);
        if (!ok) set_abort();
        const uint32_t badbits = badmask[stage];
        tc_fence_after();
        float sv[NQ];
#pragma unroll
        for (int c0 = 0; c0 < NQ; c0 += 16) {
          uint32_t r[16];
          tmem_ld16(tmem_s0 + buf * 64 + lane_addr + c0, r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) sv[c0 + i] = __uint_as_float(r[i]);
        }
        tc_fence_before();
        mbar_arrive(&s_empty[buf]);

        const int j = tile * kTile + row;
        const bool bad = (badbits >> (row / kPage)) & 1u;
        const bool valid = j < s.L && !bad;
        // scaled logits
#pragma unroll
        for (int c = 0; c < NQ; ++c) sv[c] *= scale;
        // Collect-2-Query: logits of rows row0 / row1 and their group sum, j < P_b
        if (collect && j < s.P) {
          float acc = 0.f;
#pragma unroll
          for (int c = 0; c < NQ; ++c) {
            if (c < a.NV) {
              const int t = c >> a.lgG, hl = c & (a.G - 1);
              const size_t hrow = static_cast<size_t>(s.g) * a.G + hl;
              if (t == a.row0) {
                if (a.logits)
                  __stcs(a.logits + ((static_cast<size_t>(s.b) * 2 + 0) * a.Hq + hrow) * a.P_max + j,
                         sv[c]);
                acc += sv[c];
              }
              if (t == a.row1) {
                if (a.logits)
                  __stcs(a.logits + ((static_cast<size_t>(s.b) * 2 + 1) * a.Hq + hrow) * a.P_max + j,
                         sv[c]);
                acc += sv[c];
              }
            }
          }
          if (a.partial) a.partial[(static_cast<size_t>(s.b) * a.Hkv + s.g) * a.P_max + j] = acc;
        }
        // softmax in log2 units; column c is verify row t = c / G (causal: j <= P + t)
        // visible(c) <=> c < NV and t(c) >= j - P  <=> c >= (j - P) * G for j >= P
        const int c_lo = valid ? (j < s.P ? 0 : (j - s.P) << a.lgG) : NQ;
        bool need = false;
#pragma unroll
        for (int c = 0; c < NQ; ++c) {
          sv[c] *= kLog2e;
          const bool vis = c >= c_lo && c < a.NV;
          if (vis && sv[c] > m2s[c] + kTau) need = true;
        }
        if (bar_red_or(need)) {
#pragma unroll
          for (int c = 0; c < NQ; ++c) {
            const bool vis = c >= c_lo && c < a.NV;
            const float x = warp_max(vis ? sv[c] : -INFINITY);
            if (lane == 0) red[sw * 64 + c] = x;
          }
          named_barrier_sync(kSoftmaxBar, 128);
          if (ts < NQ) {
            const float mo = m2s[ts];
            const float mx = fmaxf(fmaxf(red[ts], red[64 + ts]), fmaxf(red[128 + ts], red[192 + ts]));
            const float mn = fmaxf(mo, mx);
            alphas[ts] = (mo == -INFINITY) ? 0.f : exp2f(mo - mn);
            m2s[ts] = mn;
          }
          named_barrier_sync(kSoftmaxBar, 128);
#pragma unroll
          for (int c = 0; c < NQ; ++c) lacc[c] *= alphas[c];
          if (tile != s.t_begin) {
            // O^T holds earlier tiles: rescale its columns once the last PV is done
            if (!mbar_wait(pv_done, (it - 1) & 1, abort_flag)) set_abort();
            tc_fence_after();
#pragma unroll
            for (int c0 = 0; c0 < NQ; c0 += 16) {
              uint32_t r[16];
              tmem_ld16(tmem_o + lane_addr + c0, r);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i)
                r[i] = __float_as_uint(__uint_as_float(r[i]) * alphas[c0 + i]);
              tmem_st16(tmem_o + lane_addr + c0, r);
            }
            tmem_wait_st();
          }
        }
        // probabilities relative to the shared running max
#pragma unroll
        for (int c = 0; c < NQ; ++c) {
          const bool vis = c >= c_lo && c < a.NV;
          const float pc = vis ? exp2f(sv[c] - m2s[c]) : 0.f;
          lacc[c] += pc;
          sv[c] = pc;
        }
        // P^T is single-buffered: the previous PV must have finished reading it
        if (it > 0 && !mbar_wait(pv_done, (it - 1) & 1, abort_flag)) set_abort();
        if (j >= s.L) {
          // rows past the sequence end hold whatever the cache holds: zero V there
          uint8_t* vrow = base + stage * Cfg::kStageBytes + Cfg::kKVBytes + row * 128;
#pragma unroll
          for (int h = 0; h < D / 64; ++h)
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
              *reinterpret_cast<uint4*>(vrow + h * Cfg::kHalfBytes + ch * 16) =
                  make_uint4(0, 0, 0, 0);
        }
        uint8_t* prow = p_smem + row * 128;
#pragma unroll
        for (int ch = 0; ch < NQ / 8; ++ch) {
          uint4 pk;
          pk.x = pack_bf16x2(sv[ch * 8 + 0], sv[ch * 8 + 1]);
          pk.y = pack_bf16x2(sv[ch * 8 + 2], sv[ch * 8 + 3]);
          pk.z = pack_bf16x2(sv[ch * 8 + 4], sv[ch * 8 + 5]);
          pk.w = pack_bf16x2(sv[ch * 8 + 6], sv[ch * 8 + 7]);
          *reinterpret_cast<uint4*>(prow + ((ch ^ (row & 7)) << 4)) = pk;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(p_full);
      }

      // ---------------------------------------------------------- pair epilogue
      const size_t slot_base = static_cast<size_t>(slot) * NQ * (D + 2);
      if (has_tiles) {
#pragma unroll
        for (int c = 0; c < NQ; ++c) {
          const float x = warp_sum(lacc[c]);
          if (lane == 0) red[sw * 64 + c] = x;
        }
        named_barrier_sync(kSoftmaxBar, 128);
        if (!mbar_wait(pv_done, (it - 1) & 1, abort_flag)) set_abort();
        tc_fence_after();
        float o[NQ];
#pragma unroll
        for (int c0 = 0; c0 < NQ; c0 += 16) {
          uint32_t r[16];
          tmem_ld16(tmem_o + lane_addr + c0, r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) o[c0 + i] = __uint_as_float(r[i]);
        }
        tc_fence_before();
        if (row < D) {
          const int dim = row;
#pragma unroll
          for (int c = 0; c < NQ; ++c) {
            if (c < a.NV) {
              if (direct) {
                const float l = red[c] + red[64 + c] + red[128 + c] + red[192 + c];
                const int t = c >> a.lgG, hl = c & (a.G - 1);
                const float val = l > 0.f ? o[c] / l : 0.f;
                const __nv_bfloat16 bv = __float2bfloat16_rn(val);
                a.out[((static_cast<size_t>(s.b) * a.R + t) * a.Hq + s.g * a.G + hl) * D + dim] =
                    *reinterpret_cast<const uint16_t*>(&bv);
              } else {
                a.ws[slot_base + 2 * NQ + static_cast<size_t>(c) * D + dim] = o[c];
              }
            }
          }
        }
        if (!direct && ts < NQ) {
          a.ws[slot_base + ts] = m2s[ts];
          a.ws[slot_base + NQ + ts] = red[ts] + red[64 + ts] + red[128 + ts] + red[192 + ts];
        }
        named_barrier_sync(kSoftmaxBar, 128);
      } else {
        // no key of this pair in this CTA: an empty partial (or zeros when alone)
        if (direct) {
          for (int idx = ts; idx < a.NV * D; idx += 128) {
            const int c = idx / D, dim = idx % D;
            const int t = c >> a.lgG, hl = c & (a.G - 1);
            a.out[((static_cast<size_t>(s.b) * a.R + t) * a.Hq + s.g * a.G + hl) * D + dim] = 0;
          }
        } else {
          if (ts < NQ) {
            a.ws[slot_base + ts] = -INFINITY;
            a.ws[slot_base + NQ + ts] = 0.f;
          }
          for (int idx = ts; idx < NQ * D; idx += 128) a.ws[slot_base + 2 * NQ + idx] = 0.f;
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

// Combine the partial (m, l, o) of the CTAs that shared a pair.
template <int D, int NQ>
__global__ void __launch_bounds__(128) verify_merge_kernel(const VParams a, int ctas) {
  const int p = blockIdx.x;
  const long long W = static_cast<long long>(a.pairs) * a.t_max;
  const long long first_v = static_cast<long long>(p) * a.t_max;
  const int c_first = cta_of(first_v, W, ctas);
  const int c_last = cta_of(first_v + a.t_max - 1, W, ctas);
  if (c_first == c_last) return;
  const int n = c_last - c_first + 1;
  const int b = p / a.Hkv, g = p - (p / a.Hkv) * a.Hkv;
  const float* ws = a.ws + static_cast<size_t>(p) * a.max_chunks * NQ * (D + 2);
  const size_t slot_stride = static_cast<size_t>(NQ) * (D + 2);
  for (int idx = threadIdx.x; idx < a.NV * D; idx += blockDim.x) {
    const int c = idx / D, dim = idx % D;
    float M = -INFINITY;
    for (int k = 0; k < n; ++k) M = fmaxf(M, ws[k * slot_stride + c]);
    float L = 0.f, acc = 0.f;
    if (M != -INFINITY) {
      for (int k = 0; k < n; ++k) {
        const float mk = ws[k * slot_stride + c];
        if (mk == -INFINITY) continue;
        const float w = exp2f(mk - M);
        L += w * ws[k * slot_stride + NQ + c];
        acc += w * ws[k * slot_stride + 2 * NQ + static_cast<size_t>(c) * D + dim];
      }
    }
    const float val = L > 0.f ? acc / L : 0.f;
    const int t = c >> a.lgG, hl = c & (a.G - 1);
    const __nv_bfloat16 bv = __float2bfloat16_rn(val);
    a.out[((static_cast<size_t>(b) * a.R + t) * a.Hq + g * a.G + hl) * D + dim] =
        *reinterpret_cast<const uint16_t*>(&bv);
  }
}

template <int D, int NQ>
cudaError_t launch_dn(const VerifyArgs& va, const VerifyPlan& plan, const VParams& p,
                      cudaStream_t stream) {
  auto kern = verify_attn_collect_kernel<D, NQ>;
  constexpr int smem = VCfg<D>::kSmemBytes;
  // set on every call: the attribute is per device and the call costs no GPU work
  cudaError_t e0 = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e0 != cudaSuccess) return e0;
  kern<<<plan.ctas, kThreads, smem, stream>>>(va.kmap, va.vmap, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (plan.max_chunks > 1) {
    verify_merge_kernel<D, NQ><<<plan.pairs, 128, 0, stream>>>(p, plan.ctas);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace

VerifyPlan plan_verify(int B, int Hkv, int R, int G, int P_max, int num_sms) {
  VerifyPlan plan;
  plan.pairs = B * Hkv;
  plan.t_max = (P_max + R + kTile - 1) / kTile;
  const long long W = static_cast<long long>(plan.pairs) * plan.t_max;
  plan.ctas = static_cast<int>(W < num_sms ? W : num_sms);
  if (plan.ctas < 1) plan.ctas = 1;
  plan.nq = ((R * G + 15) / 16) * 16;
  int mc = 1;
  if (W > 0) {
    for (int p = 0; p < plan.pairs; ++p) {
      const long long f = static_cast<long long>(p) * plan.t_max;
      const long long l = f + plan.t_max - 1;
      const int cf = static_cast<int>(((f + 1) * plan.ctas - 1) / W);
      const int cl = static_cast<int>(((l + 1) * plan.ctas - 1) / W);
      if (cl - cf + 1 > mc) mc = cl - cf + 1;
    }
  }
  plan.max_chunks = mc;
  return plan;
}

size_t verify_workspace_bytes(const VerifyPlan& plan, int head_dim) {
  if (plan.max_chunks <= 1) return 0;
  return static_cast<size_t>(plan.pairs) * plan.max_chunks * plan.nq * (head_dim + 2) *
         sizeof(float);
}

cudaError_t launch_verify(const VerifyArgs& va, const VerifyPlan& plan, cudaStream_t stream) {
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
  p.G = va.G;
  int lg = 0;
  while ((1 << lg) < va.G) ++lg;
  p.lgG = lg;
  p.R = va.R;
  p.NV = va.R * va.G;
  p.max_blocks = va.max_blocks;
  p.num_blocks = va.num_blocks;
  p.P_max = va.P_max;
  p.row0 = va.row0;
  p.row1 = va.row1;
  p.pairs = plan.pairs;
  p.t_max = plan.t_max;
  p.max_chunks = plan.max_chunks;
  p.scale = va.scale;
  if (plan.pairs == 0) return cudaSuccess;
  const int nq = plan.nq;
  if (va.d == 128) {
    switch (nq) {
      case 16: return launch_dn<128, 16>(va, plan, p, stream);
      case 32: return launch_dn<128, 32>(va, plan, p, stream);
      case 48: return launch_dn<128, 48>(va, plan, p, stream);
      case 64: return launch_dn<128, 64>(va, plan, p, stream);
    }
  } else if (va.d == 64) {
    switch (nq) {
      case 16: return launch_dn<64, 16>(va, plan, p, stream);
      case 32: return launch_dn<64, 32>(va, plan, p, stream);
      case 48: return launch_dn<64, 48>(va, plan, p, stream);
      case 64: return launch_dn<64, 64>(va, plan, p, stream);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace vsd
