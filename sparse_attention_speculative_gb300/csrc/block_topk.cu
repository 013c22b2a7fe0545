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
// How (GB300 design), three kernels, each an HBM or latency problem, none a tensor-core
// contraction worth the name (R*G <= 64 query rows per KV group):
//  * page_mean_kernel: one warp per (sequence, KV group, page).  The page's 16 rows are
//    16 * d * 2 contiguous bytes; every lane issues all of its 16-byte loads before it
//    adds, then lanes holding the same columns combine with shuffles.  An optional
//    per-sequence first page lets a decode loop refresh only the pages that changed:
//    the means are a resident summary of the cache, like the cache itself.
//  * block_score_kernel: one CTA per (64 pages, KV group, sequence).  The 64 x d tile
//    of means and the group's R*G query rows sit in shared memory (the means with a
//    row stride of d + 4 floats, so the float4 reads of 8 consecutive pages hit
//    distinct banks; the query reads are warp-wide broadcasts); a thread owns one page
//    and every fourth query row.
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
constexpr int kScorePages = 64;       // pages per score CTA
constexpr int kScoreThreads = 256;
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
  ptx::pdl_launch_dependents();
  ptx::pdl_wait_primary();  // the cache and the lengths may come from the preceding kernel
  const int P = __ldg(a.prefix_len + b);
  const int nblk = (P + kPageB - 1) / kPageB;
  if (P < 0 || static_cast<long long>(P) > static_cast<long long>(a.max_blocks) * kPageB ||
      nblk > a.nblk_max) {
    if (threadIdx.x == 0 && g == 0 && blockIdx.x == 0) flag_status(a.status, VSD_DEV_BAD_LENGTH);
    return;
  }
  int first = a.page_begin != nullptr ? __ldg(a.page_begin + b) : 0;
  if (first < 0) {
    if (threadIdx.x == 0 && g == 0 && blockIdx.x == 0) flag_status(a.status, VSD_DEV_BAD_LENGTH);
    return;
  }
  if (beta < first || beta >= nblk) return;
  const int n_rows = min(kPageB, P - beta * kPageB);
  const int blk = __ldg(a.block_table + static_cast<size_t>(b) * a.max_blocks + beta);
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
template <int D>
struct ScoreSmem {
  float kbar[kScorePages][D + 4];
  float q[64][D];
};

// NR: query rows per thread (every fourth row from the thread's start), at least
// ceil(R * G / 4); slots past R * G are predicated off.
template <int D, int NR>
__global__ void __launch_bounds__(kScoreThreads, 2) block_score_kernel(const BlockTopkArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  ScoreSmem<D>& sm = *reinterpret_cast<ScoreSmem<D>*>(smem_raw);
  const int b = blockIdx.z, g = blockIdx.y;
  const int beta0 = blockIdx.x * kScorePages;
  const int t = threadIdx.x;
  const int G = a.G, RG = a.R * a.G;
  ptx::pdl_launch_dependents();
  ptx::pdl_wait_primary();  // the page means come from the preceding kernel
  const int P = __ldg(a.prefix_len + b);
  const int nblk = (P + kPageB - 1) / kPageB;
  if (P < 0 || nblk > a.nblk_max) {
    if (t == 0 && g == 0 && blockIdx.x == 0) flag_status(a.status, VSD_DEV_BAD_LENGTH);
    return;
  }
  if (beta0 >= nblk) return;
  const int n_pages = min(kScorePages, nblk - beta0);
  // stage the means and the query rows (bf16 -> fp32): every load of a thread is
  // issued before the first shared-memory store
  constexpr int C4 = D / 4, C8 = D / 8;
  constexpr int KL = kScorePages * C4 / kScoreThreads;  // float4 of means per thread
  constexpr int QL = 64 * C8 / kScoreThreads;           // 16-byte query chunks per thread
  const float* src = a.kbar + ((static_cast<size_t>(b) * a.Hkv + g) * a.nblk_max + beta0) * D;
  const uint16_t* qb = static_cast<const uint16_t*>(a.q);
  float4 kv_r[KL];
  uint4 q_r[QL];
#pragma unroll
  for (int u = 0; u < KL; ++u) {
    const int i = t + u * kScoreThreads, p = i / C4, c = (i % C4) * 4;
    kv_r[u] = p < n_pages ? __ldg(reinterpret_cast<const float4*>(src + static_cast<size_t>(p) * D + c))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int u = 0; u < QL; ++u) {
    const int i = t + u * kScoreThreads, r = i / C8, c = (i % C8) * 8;
    q_r[u] = make_uint4(0, 0, 0, 0);
    if (r < RG)
      q_r[u] = __ldg(reinterpret_cast<const uint4*>(
          qb + ((static_cast<size_t>(b) * a.R + r / G) * a.Hq + g * G + r % G) * D + c));
  }
#pragma unroll
  for (int u = 0; u < KL; ++u) {
    const int i = t + u * kScoreThreads, p = i / C4, c = (i % C4) * 4;
    *reinterpret_cast<float4*>(&sm.kbar[p][c]) = kv_r[u];
  }
#pragma unroll
  for (int u = 0; u < QL; ++u) {
    const int i = t + u * kScoreThreads, r = i / C8, c = (i % C8) * 8;
    if (r < RG) {
      float4* o = reinterpret_cast<float4*>(&sm.q[r][c]);
      o[0] = make_float4(bf16_lo(q_r[u].x), bf16_hi(q_r[u].x), bf16_lo(q_r[u].y), bf16_hi(q_r[u].y));
      o[1] = make_float4(bf16_lo(q_r[u].z), bf16_hi(q_r[u].z), bf16_lo(q_r[u].w), bf16_hi(q_r[u].w));
    }
  }
  __syncthreads();
  const int p = t & (kScorePages - 1);
  const int rs = t / kScorePages;  // 0..3, uniform within a warp
  if (p >= n_pages) return;
  float acc[NR];
#pragma unroll
  for (int i = 0; i < NR; ++i) acc[i] = 0.f;
#pragma unroll 4
  for (int c = 0; c < D; c += 4) {
    const float4 kv = *reinterpret_cast<const float4*>(&sm.kbar[p][c]);
#pragma unroll
    for (int i = 0; i < NR; ++i) {
      const int r = rs + 4 * i;
      if (i < NR - 1 || r < RG) {
        const float4 qv = *reinterpret_cast<const float4*>(&sm.q[r][c]);
        acc[i] = fmaf(qv.x, kv.x, acc[i]);
        acc[i] = fmaf(qv.y, kv.y, acc[i]);
        acc[i] = fmaf(qv.z, kv.z, acc[i]);
        acc[i] = fmaf(qv.w, kv.w, acc[i]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    const int r = rs + 4 * i;
    if (r < RG) {
      const int tr = r / G, h = g * G + r % G;
      a.scores[((static_cast<size_t>(b) * a.R + tr) * a.Hq + h) * a.nblk_max + beta0 + p] =
          acc[i] * a.scale + 0.f;  // + 0 turns -0 into +0: equal scores compare equal as keys
    }
  }
}

// ---------------------------------------------------------------- per-query selection
__device__ __forceinline__ uint32_t order_key(float s) {
  const uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Inclusive prefix sum over the CTA (kSelThreads threads); `wsum` holds the warp totals.
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
  for (int i = 0; i < kSelThreads / 32; ++i)
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

constexpr int kMaxCand = kSelThreads;  // boundary-bucket candidates ranked directly
constexpr int kBins = 256;

template <int ITEMS>
__global__ void __launch_bounds__(kSelThreads) block_select_kernel(const BlockTopkArgs a) {
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
  ptx::pdl_launch_dependents();
  ptx::pdl_wait_primary();  // the scores come from the preceding kernel
  const int P = __ldg(a.prefix_len + b);
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
    key[m] = m < n_mine ? order_key(__ldg(sc + j0 + m)) : 0u;
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
    const int incl = cta_inclusive_scan(c, wsum);
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
        const int incd = cta_inclusive_scan(cd, wsum);
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
  const int excl = cta_inclusive_scan(packed, wsum) - packed;
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

template <int D, int NR>
cudaError_t launch_scores_dn(const BlockTopkArgs& a, cudaStream_t stream) {
  dim3 grid((a.nblk_max + kScorePages - 1) / kScorePages, a.Hkv, a.B);
  return launch_pdl(block_score_kernel<D, NR>, grid, kScoreThreads,
                    static_cast<int>(sizeof(ScoreSmem<D>)), stream, a);
}

// rows per thread rounded up to one of a few instantiations
template <int D>
cudaError_t launch_scores_d(const BlockTopkArgs& a, cudaStream_t stream) {
  const int nr = (a.R * a.G + 3) / 4;
  if (nr <= 2) return launch_scores_dn<D, 2>(a, stream);
  if (nr <= 4) return launch_scores_dn<D, 4>(a, stream);
  if (nr <= 6) return launch_scores_dn<D, 6>(a, stream);
  if (nr <= 8) return launch_scores_dn<D, 8>(a, stream);
  if (nr <= 12) return launch_scores_dn<D, 12>(a, stream);
  return launch_scores_dn<D, 16>(a, stream);
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

cudaError_t launch_block_topk(const BlockTopkArgs& a, cudaStream_t stream) {
  if (a.B == 0) return cudaSuccess;
  if (a.nblk_max > 0) {
    cudaError_t e = a.d == 128   ? launch_scores_d<128>(a, stream)
                    : a.d == 64 ? launch_scores_d<64>(a, stream)
                                : cudaErrorInvalidValue;
    if (e != cudaSuccess) return e;
  }
  const dim3 grid(a.B * a.R * a.Hq);
  switch (block_select_items(a.nblk_max)) {
    case 1: return launch_pdl(block_select_kernel<1>, grid, kSelThreads, 0, stream, a);
    case 2: return launch_pdl(block_select_kernel<2>, grid, kSelThreads, 0, stream, a);
    case 4: return launch_pdl(block_select_kernel<4>, grid, kSelThreads, 0, stream, a);
    case 8: return launch_pdl(block_select_kernel<8>, grid, kSelThreads, 0, stream, a);
    case 16: return launch_pdl(block_select_kernel<16>, grid, kSelThreads, 0, stream, a);
    case 32: return launch_pdl(block_select_kernel<32>, grid, kSelThreads, 0, stream, a);
  }
  return cudaErrorInvalidValue;
}

}  // namespace vsd
