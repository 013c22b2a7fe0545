// block_topk.cu -- per-query block-sparse top-k on sm_103a.
//
// What it computes (the sparse-verification summary, "Sparse Verification Engine",
// attention sparsity): every query keeps only its top-k key/value blocks, chosen by a
// cheap relevance score.  The blocks are the 16-token pages of the prefix; the score of
// page beta for query (b, t, h) is
//   r[b,t,h,beta] = scale * < q[b,t,h,:], kbar[b,h/G,beta,:] >,
//   kbar[b,g,beta,:] = mean of K[b,j,g,:] over the page's rows j < P_b,
// and (b, t, h) keeps the kb pages with the highest r, ties to the lower page, listed
// in ascending page order.  Unlike the aggregated selection of the verification pass,
// the set differs between heads and verify rows.
//
// How (GB300 design), three kernels:
//  * page_mean_kernel: one warp per (sequence, KV group, page).  The page's 16 rows are
//    16 * d * 2 contiguous bytes; every lane issues all of its 16-byte loads before it
//    adds, then lanes holding the same columns combine with shuffles.  An optional
//    per-sequence first page lets a decode loop refresh only the pages that changed:
//    the means are a resident summary of the cache, like the cache itself.
//  * block_score_tc_kernel: persistent CTAs, each over a contiguous run of (sequence,
//    KV group, 128 pages) tiles on the tensor cores: TMA loads the fp32 means into
//    swizzled tiles (the next tile's copy under the current tile's epilogue),
//    tcgen05.mma kind::tf32 forms S^T = kbar Q^T in TMEM, and each thread writes one
//    page's scores.
//  * block_select_kernel: one CTA per query row.  The row's scores become
//    order-preserving 32-bit keys held in registers (each thread a contiguous run of
//    pages).  A first histogram buckets the values linearly between the row's minimum
//    and maximum (256 buckets, one per thread of the first 256; a monotone map, so it ranks exactly up
//    to the bucket) and finds the bucket holding the k-th value; its candidates, few
//    for any spread of scores, are gathered and each ranked against the others
//    (ties to the lower page).  Only when more than 256 pages share that bucket does
//    an exact radix select over the keys' 8-bit digits (from the highest bit where the
//    bucket's keys differ; increments aggregated over the lanes of a warp that hit the
//    same bin) finish the job.  One exclusive scan of the per-thread kept counts then
//    writes the kept pages in ascending order.
#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace vsd {
namespace {

constexpr int kPageB = 16;
constexpr int kMeanWarps = 8;         // pages per page-mean CTA
constexpr int kSelThreads = 512;

// ---------------------------------------------------------------- page means
template <int D>
__global__ void __launch_bounds__(kMeanWarps * 32) page_mean_kernel(const BlockTopkArgs a) {
  constexpr int CPR = D / 8;          // 16-byte chunks per row
  constexpr int RPL = 32 / CPR;       // rows covered by one warp-wide load
  constexpr int NL = kPageB / RPL;    // loads per lane
  const int b = blockIdx.z, g = blockIdx.y;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int beta = blockIdx.x * kMeanWarps + w;
  ptx::pdl_wait_primary();  // the cache and the lengths may come from the preceding kernel
  ptx::pdl_launch_dependents();
  const int P = __ldcg(a.prefix_len + b);
  const int nblk = (P + kPageB - 1) / kPageB;
  if (P < 0 || static_cast<long long>(P) > static_cast<long long>(a.max_blocks) * kPageB ||
      nblk > a.nblk_max) {
    if (threadIdx.x == 0 && g == 0 && blockIdx.x == 0) flag_status(a.status, VSD_DEV_BAD_LENGTH);
    return;
  }
  int first = a.page_begin != nullptr ? __ldcg(a.page_begin + b) : 0;
  if (first < 0) {
    if (threadIdx.x == 0 && g == 0 && blockIdx.x == 0) flag_status(a.status, VSD_DEV_BAD_LENGTH);
    return;
  }
  if (beta < first || beta >= nblk) return;
  const int n_rows = min(kPageB, P - beta * kPageB);
  const int blk = __ldcg(a.block_table + static_cast<size_t>(b) * a.max_blocks + beta);
  float* dst = a.kbar + ((static_cast<size_t>(b) * a.Hkv + g) * a.nblk_max + beta) * D;
  const int col = lane % CPR, row0 = lane / CPR;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  if (blk < 0 || blk >= a.num_blocks) {
    if (lane == 0) flag_status(a.status, VSD_DEV_BAD_BLOCK);
  } else {
    const uint16_t* src = static_cast<const uint16_t*>(a.k_cache) +
                          (static_cast<size_t>(blk) * a.Hkv + g) * kPageB * D;
    uint4 v[NL];
#pragma unroll
    for (int i = 0; i < NL; ++i) {
      const int r = RPL * i + row0;
      v[i] = r < n_rows ? ldg_stream16(src + r * D + col * 8) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < NL; ++i) {
      const uint32_t u[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc[2 * e] += bf16_lo(u[e]);
        acc[2 * e + 1] += bf16_hi(u[e]);
      }
    }
  }
#pragma unroll
  for (int off = CPR; off < 32; off <<= 1) {
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], off);
  }
  if (lane < CPR) {
    const float inv = 1.f / static_cast<float>(n_rows);
    float4* o = reinterpret_cast<float4*>(dst + col * 8);
    o[0] = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
    o[1] = make_float4(acc[4] * inv, acc[5] * inv, acc[6] * inv, acc[7] * inv);
  }
}

// ---------------------------------------------------------------- page scores
// Persistent CTAs of four warps on the tensor cores.  The (sequence, KV group,
// 128-page tile) triples are numbered in that order and each CTA takes a contiguous run
// of them, so a group's query block is staged once per run rather than once per tile:
// S^T[128 pages x NQ] = kbar[128 x d] . Q^T[d x NQ] (NQ = R * G rounded up to 16).
// TMA brings the fp32 page means straight into 128-byte-swizzled K-major tiles (32 fp32
// per row, d / 32 boxes); the group's bf16 query rows are staged as fp32 in the same
// layout; tcgen05.mma kind::tf32 accumulates in TMEM (bf16 queries are exact in tf32,
// the means lose their low 13 mantissa bits: ~1e-4 on a score).  Once a tile's product
// is complete its buffer takes the next tile's copy, which then runs under this tile's
// epilogue: thread t reads page t's NQ scores and writes them, each column a coalesced
// run of pages.
constexpr int kTcPages = 128;
constexpr int kTcScoreThreads = 128;

template <int D, int NQ>
struct TcScoreSmem {
  static constexpr int kBox = kTcPages * 128;           // one 32-column box of the means
  static constexpr int kOffA = 0;
  static constexpr int kOffQ = kOffA + (D / 32) * kBox;
  static constexpr int kOffBar = kOffQ + (D / 32) * NQ * 128;
  static constexpr int kBytes = kOffBar + 64 + 1024;    // + alignment slack
  static_assert(kOffQ % 1024 == 0 && kOffBar % 8 == 0, "layout");
};

template <int D, int NQ>
__global__ void __launch_bounds__(kTcScoreThreads) block_score_tc_kernel(
    const __grid_constant__ CUtensorMap kbar_map, const BlockTopkArgs a, const int tiles_per_cta) {
  using Sm = TcScoreSmem<D, NQ>;
  extern __shared__ uint8_t sc_smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(sc_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* a_s = base + Sm::kOffA;
  uint8_t* q_s = base + Sm::kOffQ;
  uint64_t* bar_a = reinterpret_cast<uint64_t*>(base + Sm::kOffBar);
  uint64_t* bar_s = bar_a + 1;
  uint64_t* bar_fin = bar_a + 2;  // every product of this CTA complete (before TMEM goes back)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_a + 3);
  const int t = threadIdx.x, warp = t >> 5;
  const int G = a.G, RG = a.R * a.G;
  const int ntile = (a.nblk_max + kTcPages - 1) / kTcPages;
  const int first = blockIdx.x * tiles_per_cta;
  const int last = min(a.B * a.Hkv * ntile, first + tiles_per_cta);
  if (t == 0) {
    ptx::mbar_init(bar_a, 1);
    ptx::mbar_init(bar_s, 1);
    ptx::mbar_init(bar_fin, 1);
    ptx::fence_mbarrier_init();
    ptx::tma_prefetch_desc(&kbar_map);
  }
  if (warp == 0) {
    ptx::tmem_alloc(tmem_slot, NQ <= 32 ? 32 : 64);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  ptx::pdl_wait_primary();  // the page means come from the preceding kernel
  ptx::pdl_launch_dependents();

  // tile id -> its (sequence, KV group) pair bg = b * Hkv + g and first page; a tile has
  // work when its sequence's length is valid and reaches the tile
  const auto pages_of = [&](int P) { return (P + kPageB - 1) / kPageB; };
  const auto has_work = [&](int id, int P) {
    return P >= 0 && pages_of(P) <= a.nblk_max && (id % ntile) * kTcPages < pages_of(P);
  };
  const auto fetch = [&](int id) {  // thread 0: the tile's means into the buffer
    ptx::mbar_arrive_expect_tx(bar_a, (D / 32) * Sm::kBox);
    const int row0 = (id / ntile) * a.nblk_max + (id % ntile) * kTcPages;
#pragma unroll
    for (int c = 0; c < D / 32; ++c)
      ptx::tma_load_2d(a_s + c * Sm::kBox, &kbar_map, bar_a, c * 32, row0);
  };

  constexpr int QL = NQ * (D / 8) / kTcScoreThreads;
  static_assert(NQ * (D / 8) % kTcScoreThreads == 0, "query staging");
  const uint16_t* qb = static_cast<const uint16_t*>(a.q);
  uint32_t a_phase = 0, s_phase = 0;
  bool in_flight = false;  // thread 0: a copy into the buffer has not been waited for
  bool timed_out = false;
  int staged_bg = -1;
  int P_next = first < last ? __ldcg(a.prefix_len + first / ntile / a.Hkv) : 0;
  for (int id = first; id < last; ++id) {
    const int x = id % ntile, bg = id / ntile, g = bg % a.Hkv, b = bg / a.Hkv;
    const int P = P_next;
    if (id + 1 < last) P_next = __ldcg(a.prefix_len + (id + 1) / ntile / a.Hkv);
    if ((P < 0 || pages_of(P) > a.nblk_max) && t == 0 && g == 0 && x == 0)
      flag_status(a.status, VSD_DEV_BAD_LENGTH);
    if (!has_work(id, P)) continue;  // CTA-uniform; nothing was fetched for it
    if (t == 0 && !in_flight) {
      fetch(id);
      in_flight = true;
    }
    if (bg != staged_bg) {
      // the group's query rows r = tr * G + hl as fp32, zero past R * G (the previous
      // tile's product, the last reader of this block, is complete)
      uint4 qv[QL];
#pragma unroll
      for (int u = 0; u < QL; ++u) {
        const int i = t + u * kTcScoreThreads, r = i / (D / 8), c8 = i % (D / 8);
        qv[u] = make_uint4(0, 0, 0, 0);
        if (r < RG)
          qv[u] = __ldcg(reinterpret_cast<const uint4*>(
              qb + ((static_cast<size_t>(b) * a.R + r / G) * a.Hq + g * G + r % G) * D + c8 * 8));
      }
#pragma unroll
      for (int u = 0; u < QL; ++u) {
        const int i = t + u * kTcScoreThreads, r = i / (D / 8), c8 = i % (D / 8);
        const int c = c8 >> 2;            // 32-dim box
        const int u0 = (c8 & 3) * 2;      // first 16-byte unit of the 128-byte row
        uint8_t* row = q_s + c * NQ * 128 + r * 128;
        const uint4 v = qv[u];
        *reinterpret_cast<float4*>(row + ((u0 ^ (r & 7)) << 4)) =
            make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y));
        *reinterpret_cast<float4*>(row + (((u0 + 1) ^ (r & 7)) << 4)) =
            make_float4(bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w));
      }
      ptx::fence_proxy_async_smem();
      staged_bg = bg;
    }
    ptx::tc_fence_before();
    // the query block is staged and the previous tile's TMEM reads are done
    if (__syncthreads_or(timed_out)) break;
    if (t == 0) {
      if (ptx::mbar_wait(bar_a, a_phase)) {
        a_phase ^= 1;
        in_flight = false;
      } else {
        timed_out = true;
      }
    }
    // no product on a tile whose copy has not landed (the loop ends at the next vote)
    if (__syncthreads_or(timed_out)) break;
    if (t == 0) {
      ptx::tc_fence_after();
      constexpr uint32_t idesc = ptx::idesc_tf32_f32(128, NQ, 0, 0);
      const uint32_t aa = ptx::smem_u32(a_s), qa = ptx::smem_u32(q_s);
#pragma unroll
      for (int kk = 0; kk < D / 8; ++kk) {
        const int c = kk >> 2, w = kk & 3;
        const uint64_t ad = ptx::sdesc_sw128(aa + c * Sm::kBox + w * 32, 16, 1024);
        const uint64_t bd = ptx::sdesc_sw128(qa + c * NQ * 128 + w * 32, 16, 1024);
        ptx::umma_tf32(tmem, ad, bd, idesc, kk > 0 ? 1u : 0u);
      }
      ptx::umma_commit(bar_s);
    }
    if (!ptx::mbar_wait(bar_s, s_phase)) timed_out = true;
    s_phase ^= 1;
    ptx::tc_fence_after();
    // the product has read the buffer: it takes the next tile's copy now
    if (t == 0 && !timed_out && id + 1 < last && has_work(id + 1, P_next)) {
      fetch(id + 1);
      in_flight = true;
    }
    float sv[NQ];
    ptx::tmem_ld_cols<NQ>(tmem + (static_cast<uint32_t>(warp * 32) << 16),
                          reinterpret_cast<uint32_t*>(sv));
    ptx::tmem_wait_ld();
    const int beta = x * kTcPages + t;  // TMEM lane t = page beta
    if (beta < pages_of(P)) {
      // column c = tr * G + hl is query row (b, tr, g * G + hl): consecutive columns step
      // one head, and past the group's last head to the next draft position's first
      const size_t step_h = static_cast<size_t>(a.nblk_max);
      const size_t step_r = static_cast<size_t>(a.Hq - G + 1) * a.nblk_max;
      float* dst = a.scores + (static_cast<size_t>(b) * a.R * a.Hq + g * G) * a.nblk_max + beta;
      int hl = 0;
#pragma unroll
      for (int c = 0; c < NQ; ++c) {
        if (c < RG) {
          *dst = sv[c] * a.scale + 0.f;  // + 0 turns -0 into +0: equal scores compare equal as keys
          if (++hl == G) {
            hl = 0;
            dst += step_r;
          } else {
            dst += step_h;
          }
        }
      }
    }
  }
  // a copy still in flight lands and every product issued completes before the CTA
  // leaves and frees its TMEM (waits with the drain limit)
  if (t == 0) {
    if (in_flight && !ptx::mbar_wait_drain(bar_a, a_phase)) timed_out = true;
    ptx::umma_commit(bar_fin);  // arrives once every earlier product of this thread is done
    if (!ptx::mbar_wait_drain(bar_fin, 0)) timed_out = true;
  }
  if (timed_out) flag_status(a.status, VSD_DEV_TIMEOUT);
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, NQ <= 32 ? 32 : 64);
  }
}

// ---------------------------------------------------------------- per-query selection
__device__ __forceinline__ uint32_t order_key(float s) {
  const uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Inclusive prefix sum over the CTA (NT threads); `wsum` holds the warp totals.
template <int NT>
__device__ __forceinline__ int cta_inclusive_scan(int x, int* wsum) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[w] = x;
  __syncthreads();
  int add = 0;
#pragma unroll
  for (int i = 0; i < NT / 32; ++i)
    if (i < w) add += wsum[i];
  return x + add;
}

// Histogram increment aggregated over the lanes of a warp that hit the same bin (the
// keys of one row share many leading bits, so a plain shared-memory atomic per key
// would serialise on a few hot bins).  Every lane of the warp calls it.
__device__ __forceinline__ void hist_add(int* H, uint32_t bin, bool active) {
  const unsigned act = __ballot_sync(0xffffffffu, active);
  if (active) {
    const unsigned peers = __match_any_sync(act, bin);
    if (__ffs(peers) - 1 == static_cast<int>(threadIdx.x & 31)) atomicAdd(&H[bin], __popc(peers));
  }
}

// 8-bit digit of `key` whose lowest bit is `shift` (shift < 0: the digit runs past bit 0
// and its low bits are zero).
__device__ __forceinline__ uint32_t digit_of(uint32_t key, int shift) {
  return (shift >= 0 ? key >> shift : key << -shift) & 0xFFu;
}
__device__ __forceinline__ uint32_t digit_mask(int shift) {
  return shift >= 0 ? 0xFFu << shift : 0xFFu >> -shift;
}

__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// NT threads per row; the boundary bucket's candidates are ranked directly up to NT
constexpr int kBins = 256;

// The 256-thread form runs when rows are plentiful: capped at 40 registers so that six
// CTAs (six rows) are resident per SM instead of five.
template <int ITEMS, int NT>
__global__ void __launch_bounds__(NT, NT == 256 ? 6 : 1) block_select_kernel(const BlockTopkArgs a) {
  constexpr int kSelThreads = NT, kMaxCand = NT;
  static_assert(kSelThreads >= kBins && ITEMS <= 32, "one bin per thread; keep mask in 32 bits");
  __shared__ int hist[2][kBins];
  __shared__ int wsum[kSelThreads / 32];
  __shared__ uint32_t s_min[kSelThreads / 32], s_max[kSelThreads / 32];
  __shared__ uint32_t keep_bits[16384 / 32];
  __shared__ uint32_t cand_key[kMaxCand];
  __shared__ int cand_j[kMaxCand];
  __shared__ int s_digit, s_need, s_all, s_cnt;
  const int row = blockIdx.x;  // (b, t, h) flattened
  const int b = row / (a.R * a.Hq);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  int32_t* out = a.blocks + static_cast<size_t>(row) * a.kb;
  ptx::pdl_wait_primary();  // the scores come from the preceding kernel
  ptx::pdl_launch_dependents();
  const int P = __ldcg(a.prefix_len + b);
  int nblk = (P + kPageB - 1) / kPageB;
  if (P < 0 || nblk > a.nblk_max) nblk = 0;  // flagged by the score kernel
  if (nblk <= a.kb) {  // every page is kept
    for (int i = tid; i < a.kb; i += kSelThreads) out[i] = i < nblk ? i : -1;
    return;
  }
  const float* sc = a.scores + static_cast<size_t>(row) * a.nblk_max;
  const int j0 = tid * ITEMS;
  const int n_mine = max(0, min(ITEMS, nblk - j0));  // this thread's pages j0 .. j0+n_mine
  uint32_t key[ITEMS];
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll
  for (int m = 0; m < ITEMS; ++m) {
    key[m] = m < n_mine ? order_key(__ldcg(sc + j0 + m)) : 0u;
    if (m < n_mine) {
      kmin = min(kmin, key[m]);
      kmax = max(kmax, key[m]);
    }
  }
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if (lane == 0) {
    s_min[w] = kmin;
    s_max[w] = kmax;
  }
  if (tid < kBins) hist[0][tid] = 0;
  for (int i = tid; i < (nblk + 31) / 32; i += kSelThreads) keep_bits[i] = 0u;
  if (tid == 0) s_cnt = 0;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kSelThreads / 32; ++i) {
    kmin = min(kmin, s_min[i]);
    kmax = max(kmax, s_max[i]);
  }

  // Pass 0: 256 buckets linear in the value between the row's min and max (monotone,
  // so every page of a higher bucket outranks every page of a lower one).
  const float fmin = key_value(kmin), range = key_value(kmax) - fmin;
  float inv = 256.f / range;
  const bool linear = kmax != kmin && range < 3.0e38f && inv > 0.f && inv < 3.0e38f;
  int bk[ITEMS];
#pragma unroll
  for (int m = 0; m < ITEMS; ++m)
    bk[m] = linear ? min(kBins - 1, static_cast<int>((key_value(key[m]) - fmin) * inv)) : 0;
  int bstar = 0;            // boundary bucket
  int need = a.kb;          // pages still to take from the boundary class
  bool whole = false;       // the whole boundary class is taken
  uint32_t prefix = 0u, mask = 0u;  // exact-key class inside the boundary bucket (radix)
  bool radix = false;
  if (kmax == kmin) {
    radix = true;  // every key equal: the class is the whole row, lowest pages first
    mask = 0xFFFFFFFFu;
    prefix = kmin;
  } else {
#pragma unroll
    for (int m = 0; m < ITEMS; ++m)
      if (m < n_mine) atomicAdd(&hist[0][bk[m]], 1);
    if (tid < kBins) hist[1][tid] = 0;
    __syncthreads();
    // counts from the highest bucket down: thread tid < 256 owns bucket 255 - tid
    const int c = tid < kBins ? hist[0][kBins - 1 - tid] : 0;
    const int incl = cta_inclusive_scan<NT>(c, wsum);
    const int excl = incl - c;
    if (c > 0 && excl < need && need <= incl) {
      s_digit = kBins - 1 - tid;
      s_need = need - excl;
      s_all = c == need - excl ? 1 : (c <= kMaxCand ? 0 : -1);
    }
    __syncthreads();
    bstar = s_digit;
    need = s_need;
    whole = s_all == 1;
    if (s_all == 0) {
      // few candidates: gather them and rank each against the others
#pragma unroll
      for (int m = 0; m < ITEMS; ++m) {
        if (m < n_mine && bk[m] == bstar) {
          const int slot = atomicAdd(&s_cnt, 1);
          cand_key[slot] = key[m];
          cand_j[slot] = j0 + m;
        }
      }
      __syncthreads();
      const int cnt = s_cnt;
      if (tid < cnt) {
        const uint32_t kx = cand_key[tid];
        const int jx = cand_j[tid];
        int rank = 0;
#pragma unroll 4
        for (int y = 0; y < cnt; ++y) {
          const uint32_t ky = cand_key[y];
          rank += ky > kx || (ky == kx && cand_j[y] < jx);
        }
        if (rank < need) atomicOr(&keep_bits[jx >> 5], 1u << (jx & 31));
      }
      __syncthreads();
    } else if (s_all == -1) {
      // many candidates: exact-key radix over the boundary bucket, 8-bit digits from
      // the highest bit where its keys differ
      radix = true;
      uint32_t kor = 0u, kand = 0xFFFFFFFFu;
#pragma unroll
      for (int m = 0; m < ITEMS; ++m) {
        if (m < n_mine && bk[m] == bstar) {
          kor |= key[m];
          kand &= key[m];
        }
      }
      kor = __reduce_or_sync(0xffffffffu, kor);
      kand = __reduce_and_sync(0xffffffffu, kand);
      if (lane == 0) {
        s_min[w] = kor;
        s_max[w] = kand;
      }
      __syncthreads();
#pragma unroll
      for (int i = 0; i < kSelThreads / 32; ++i) {
        kor |= s_min[i];
        kand &= s_max[i];
      }
      const uint32_t diff = kor ^ kand;
      const int hb = diff ? 31 - __clz(diff) : -1;
      mask = hb >= 31 ? 0u : (0xFFFFFFFFu << (hb + 1));
      prefix = kand & mask;
#pragma unroll 1
      for (int shift = hb - 7, pass = 1; shift > -8; shift -= 8, ++pass) {
        int* Hp = hist[pass & 1];
#pragma unroll
        for (int m = 0; m < ITEMS; ++m)
          hist_add(Hp, digit_of(key[m], shift),
                   m < n_mine && bk[m] == bstar && (key[m] & mask) == prefix);
        if (tid < kBins) hist[(pass + 1) & 1][tid] = 0;  // its readers finished last pass
        __syncthreads();
        const int cd = tid < kBins ? Hp[kBins - 1 - tid] : 0;
        const int incd = cta_inclusive_scan<NT>(cd, wsum);
        const int exd = incd - cd;
        if (cd > 0 && exd < need && need <= incd) {
          s_digit = kBins - 1 - tid;
          s_need = need - exd;
          s_all = cd == need - exd;
        }
        __syncthreads();
        need = s_need;
        const uint32_t dg = static_cast<uint32_t>(s_digit);
        prefix |= shift >= 0 ? dg << shift : dg >> -shift;
        mask |= digit_mask(shift);
        if (s_all) {
          whole = true;
          break;
        }
      }
    }
  }
  // Decide every page once: above the boundary bucket; in it and ranked in (or the
  // whole bucket taken); on the radix path, above the exact-key class, or in it and
  // among its first `need` pages.  Then write the kept pages in ascending order.
  uint32_t keep = 0u, in_class = 0u;
#pragma unroll
  for (int m = 0; m < ITEMS; ++m) {
    if (m < n_mine) {
      const int j = j0 + m;
      bool k = bk[m] > bstar;
      if (bk[m] == bstar) {
        if (!radix) {
          k = whole || ((keep_bits[j >> 5] >> (j & 31)) & 1u);
        } else {
          const uint32_t mk = key[m] & mask;
          k = mk > prefix;
          if (mk == prefix) in_class |= 1u << m;
        }
      }
      if (k) keep |= 1u << m;
    }
  }
  const int packed = __popc(keep) | (__popc(in_class) << 16);  // both < 2^16
  const int excl = cta_inclusive_scan<NT>(packed, wsum) - packed;
  int eq_before = excl >> 16;
  const int eq_take = whole ? (1 << 30) : need;
  int pos = (excl & 0xFFFF) + min(eq_before, eq_take);
#pragma unroll
  for (int m = 0; m < ITEMS; ++m) {
    bool k = (keep >> m) & 1u;
    if ((in_class >> m) & 1u) {
      k = eq_before < eq_take;
      ++eq_before;
    }
    if (k) out[pos++] = j0 + m;
  }
}

template <typename K>
cudaError_t launch_pdl(K kernel, dim3 grid, int threads, int smem, cudaStream_t stream,
                       const BlockTopkArgs& a) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

template <int D, int NQ>
cudaError_t launch_scores_dn(const CUtensorMap& map, const BlockTopkArgs& a, cudaStream_t stream) {
  auto kern = block_score_tc_kernel<D, NQ>;
  constexpr int smem = TcScoreSmem<D, NQ>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  // persistent CTAs: as many as fit at once, each with a contiguous run of tiles
  static int per_sm = 0;
  if (per_sm == 0) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kTcScoreThreads, smem);
    if (e != cudaSuccess) return e;
    per_sm = per_sm > 0 ? per_sm : 1;
  }
  int dev = 0, sm_count = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long tiles =
      static_cast<long long>(a.B) * a.Hkv * ((a.nblk_max + kTcPages - 1) / kTcPages);
  const long long slots = static_cast<long long>(per_sm) * sm_count;
  const int per_cta = static_cast<int>((tiles + slots - 1) / slots);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((tiles + per_cta - 1) / per_cta), 1, 1);
  cfg.blockDim = dim3(kTcScoreThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, map, a, per_cta);
}

template <int D>
cudaError_t launch_scores_d(const CUtensorMap& map, const BlockTopkArgs& a, cudaStream_t stream) {
  const int nq = (a.R * a.G + 15) / 16 * 16;
  if (nq <= 16) return launch_scores_dn<D, 16>(map, a, stream);
  if (nq <= 32) return launch_scores_dn<D, 32>(map, a, stream);
  if (nq <= 48) return launch_scores_dn<D, 48>(map, a, stream);
  return launch_scores_dn<D, 64>(map, a, stream);
}

}  // namespace

int block_select_items(int nblk_max) {
  int items = 1;
  while (items * kSelThreads < nblk_max) items <<= 1;
  return items <= 32 ? items : -1;
}

cudaError_t launch_page_means(const BlockTopkArgs& a, cudaStream_t stream) {
  if (a.B == 0 || a.nblk_max == 0) return cudaSuccess;
  dim3 grid((a.nblk_max + kMeanWarps - 1) / kMeanWarps, a.Hkv, a.B);
  if (a.d == 128) return launch_pdl(page_mean_kernel<128>, grid, kMeanWarps * 32, 0, stream, a);
  if (a.d == 64) return launch_pdl(page_mean_kernel<64>, grid, kMeanWarps * 32, 0, stream, a);
  return cudaErrorInvalidValue;
}

cudaError_t launch_block_topk(const CUtensorMap& kbar_map, const BlockTopkArgs& a,
                              cudaStream_t stream) {
  if (a.B == 0) return cudaSuccess;
  if (a.nblk_max > 0) {
    cudaError_t e = a.d == 128   ? launch_scores_d<128>(kbar_map, a, stream)
                    : a.d == 64 ? launch_scores_d<64>(kbar_map, a, stream)
                                : cudaErrorInvalidValue;
    if (e != cudaSuccess) return e;
  }
  const int rows = a.B * a.R * a.Hq;
  const dim3 grid(rows);
  // many rows: 256-thread CTAs (twice as many resident per SM); few rows: 512 threads,
  // half the work per thread on each row's dependent chain
  int sm_count = 152;
  {
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess)
      cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev);
  }
  if (rows > 2 * sm_count && a.nblk_max <= 256 * 32) {
    int items = 1;
    while (items * 256 < a.nblk_max) items <<= 1;
    switch (items) {
      case 1: return launch_pdl(block_select_kernel<1, 256>, grid, 256, 0, stream, a);
      case 2: return launch_pdl(block_select_kernel<2, 256>, grid, 256, 0, stream, a);
      case 4: return launch_pdl(block_select_kernel<4, 256>, grid, 256, 0, stream, a);
      case 8: return launch_pdl(block_select_kernel<8, 256>, grid, 256, 0, stream, a);
      case 16: return launch_pdl(block_select_kernel<16, 256>, grid, 256, 0, stream, a);
      case 32: return launch_pdl(block_select_kernel<32, 256>, grid, 256, 0, stream, a);
    }
    return cudaErrorInvalidValue;
  }
  switch (block_select_items(a.nblk_max)) {
    case 1: return launch_pdl(block_select_kernel<1, kSelThreads>, grid, kSelThreads, 0, stream, a);
    case 2: return launch_pdl(block_select_kernel<2, kSelThreads>, grid, kSelThreads, 0, stream, a);
    case 4: return launch_pdl(block_select_kernel<4, kSelThreads>, grid, kSelThreads, 0, stream, a);
    case 8: return launch_pdl(block_select_kernel<8, kSelThreads>, grid, kSelThreads, 0, stream, a);
    case 16: return launch_pdl(block_select_kernel<16, kSelThreads>, grid, kSelThreads, 0, stream, a);
    case 32: return launch_pdl(block_select_kernel<32, kSelThreads>, grid, kSelThreads, 0, stream, a);
  }
  return cudaErrorInvalidValue;
}

}  // namespace vsd
