// sparse_decode.cu -- sparse draft-step attention on sm_103a.
//
// What it computes ("Vegas" technical summary, sec. 2 drafting phase and sec. 3
// sparse execution): one query row per head attends only the selected positions
// (paged attention with page size 1 whose page indices are the selected token
// indices) plus the tokens appended after the selection (dense tail).
//
// How (GB300 design).  The step moves a few MB of randomly placed 256-byte rows, so it
// is bound by the latency of its dependent loads (index -> block table -> K and V
// rows), not by bandwidth.  The design therefore issues every load of a CTA at once
// and spreads the list over as many SMs as there are batches of 64 positions:
//   * The attended list of one (sequence, KV head) pair, idx[0 .. n_sel) followed by
//     [tail_start, seq_len), is cut into splits of 64 positions (more per split only
//     when the list is very long); one CTA of four warps takes one split, each warp
//     16 positions.
//   * Two lanes own one key: each gathers half of the key's K row with 16-byte
//     loads (adjacent lanes read adjacent 16 bytes), and the warp also issues the V
//     loads of its 16 rows (lane = 4 or 2 dims of every row, coalesced per row).
//   * Logits of the G query heads of the group are fp32 dot products (q in shared
//     memory), the pair of lanes combining its halves with one shuffle; the warp
//     softmax over its 16 keys and the P.V product follow in registers.
//   * The four warps merge in shared memory in a fixed order.  A pair with a single
//     split writes its output directly; otherwise each split writes (m, l, o) to the
//     workspace and a merge kernel (one block per pair and head, launched as a
//     programmatic dependent so it is resident before the splits finish) combines
//     them in split order.  Results are bit-reproducible; no atomics.
#include <cfloat>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace vsd {
namespace {

constexpr int kSWarps = 4;
constexpr int kSThreads = kSWarps * 32;
constexpr int kKeysPerWarp = 16;
constexpr int kBatch = kSWarps * kKeysPerWarp;  // positions per CTA per batch
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
  unsigned* status;
  int Hq, Hkv, max_blocks, num_blocks, k_max;
  int split_len;   // positions per split (a multiple of kBatch)
  int max_splits;  // workspace slots per pair
  float scale_log2;
};

template <int D, int G>
struct SSmem {
  float q[G][D];
  float p[kSWarps][kKeysPerWarp][G];
  float wm[kSWarps][G];
  float wl[kSWarps][G];
  float wo[kSWarps][G][D];
};

__device__ __forceinline__ float wmax_pairs(float x) {
  // max over the 16 keys of a warp (lanes 2k and 2k+1 hold the same value)
#pragma unroll
  for (int o = 2; o < 32; o <<= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float wsum_pairs(float x) {
#pragma unroll
  for (int o = 2; o < 32; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// The attended list of sequence b and its validity (false: bad lengths, nothing read).
struct SList {
  int ns, t0, total;
};

__device__ __forceinline__ SList attended_list(const SParams& a, int b, bool flag) {
  SList L;
  int ns = a.n_sel != nullptr ? __ldg(a.n_sel + b) : 0;
  const int t0 = __ldg(a.tail_start + b);
  const int t1 = __ldg(a.seq_len + b);
  const bool ok = ns >= 0 && ns <= a.k_max && t0 >= 0 && t0 <= t1 &&
                  static_cast<long long>(t1) <= static_cast<long long>(a.max_blocks) * kPageS;
  if (!ok && flag) flag_status(a.status, VSD_DEV_BAD_LENGTH);
  L.ns = ok ? ns : 0;
  L.t0 = t0;
  L.total = ok ? ns + (t1 - t0) : 0;
  return L;
}

template <int D, int G>
__global__ void __launch_bounds__(kSThreads) sparse_decode_kernel(const SParams a) {
  constexpr int DPL = D / 32;       // dims per lane for V and the output
  constexpr int KH = D / 2;         // K dims per lane (half a row)
  constexpr int KV16 = KH / 8;      // 16-byte K loads per lane
  __shared__ __align__(16) SSmem<D, G> sm;
  const int split = blockIdx.x;
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = lane & 1;

  ptx::pdl_launch_dependents();  // the merge kernel may become resident now
  ptx::pdl_wait_primary();       // idx / n_sel come from the preceding kernel

  const int t1 = __ldg(a.seq_len + b);
  const SList L = attended_list(a, b, split == 0 && g == 0 && threadIdx.x == 0);
  const int lo = split * a.split_len;
  if (lo >= L.total && !(split == 0 && L.total == 0)) return;  // no work in this split
  const int hi = min(lo + a.split_len, L.total);
  const int n_splits = (L.total + a.split_len - 1) / a.split_len;

  for (int i = threadIdx.x; i < G * D / 8; i += kSThreads) {
    const int hh = i / (D / 8), c8 = i % (D / 8);
    const uint4 raw = *reinterpret_cast<const uint4*>(
        a.q + (static_cast<size_t>(b) * a.Hq + g * G + hh) * D + c8 * 8);
    float* dst = &sm.q[hh][c8 * 8];
    dst[0] = bf16_lo(raw.x);
    dst[1] = bf16_hi(raw.x);
    dst[2] = bf16_lo(raw.y);
    dst[3] = bf16_hi(raw.y);
    dst[4] = bf16_lo(raw.z);
    dst[5] = bf16_hi(raw.z);
    dst[6] = bf16_lo(raw.w);
    dst[7] = bf16_hi(raw.w);
  }
  __syncthreads();

  float m[G], lsum[G], acc[G][DPL];
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    m[hh] = -INFINITY;
    lsum[hh] = 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[hh][e] = 0.f;
  }

  for (int base = lo + warp * kKeysPerWarp; base < hi; base += kBatch) {
    // ---- this lane pair's key: list position -> token -> cache row
    const int pos = base + (lane >> 1);
    int row = -1;
    if (pos < hi) {
      const int j = pos < L.ns ? __ldg(a.idx + static_cast<size_t>(b) * a.k_max + pos)
                               : L.t0 + (pos - L.ns);
      if (j < 0 || j >= t1) {
        if (half == 0) flag_status(a.status, VSD_DEV_BAD_INDEX);
      } else {
        const int blk = __ldg(a.block_table + static_cast<size_t>(b) * a.max_blocks + j / kPageS);
        if (blk < 0 || blk >= a.num_blocks) {
          if (half == 0) flag_status(a.status, VSD_DEV_BAD_BLOCK);
        } else {
          row = (blk * a.Hkv + g) * kPageS + (j % kPageS);
        }
      }
    }
    // ---- all loads of the batch in flight: half a K row per lane, V slices
    uint4 kr[KV16];
    if (row >= 0) {
      const uint16_t* src = a.k_cache + static_cast<size_t>(row) * D + half * KH;
#pragma unroll
      for (int i = 0; i < KV16; ++i) kr[i] = ldg_stream16(src + i * 8);
    } else {
#pragma unroll
      for (int i = 0; i < KV16; ++i) kr[i] = make_uint4(0, 0, 0, 0);
    }
    uint32_t vr[kKeysPerWarp][DPL / 2];
#pragma unroll
    for (int kk = 0; kk < kKeysPerWarp; ++kk) {
      const int r = __shfl_sync(0xffffffffu, row, 2 * kk);
      if (r >= 0) {
        const uint16_t* src = a.v_cache + static_cast<size_t>(r) * D + lane * DPL;
        if constexpr (DPL == 4) {
          const uint2 v2 = ldg_stream8(src);
          vr[kk][0] = v2.x;
          vr[kk][1] = v2.y;
        } else {
          vr[kk][0] = ldg_stream4(src);
        }
      } else {
#pragma unroll
        for (int e = 0; e < DPL / 2; ++e) vr[kk][e] = 0u;
      }
    }
    // ---- logits: half-row dot products, combined across the lane pair
    float z[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) z[hh] = 0.f;
#pragma unroll
    for (int i = 0; i < KV16; ++i) {
      float kf[8];
      kf[0] = bf16_lo(kr[i].x); kf[1] = bf16_hi(kr[i].x);
      kf[2] = bf16_lo(kr[i].y); kf[3] = bf16_hi(kr[i].y);
      kf[4] = bf16_lo(kr[i].z); kf[5] = bf16_hi(kr[i].z);
      kf[6] = bf16_lo(kr[i].w); kf[7] = bf16_hi(kr[i].w);
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        const float4 qa = *reinterpret_cast<const float4*>(&sm.q[hh][half * KH + i * 8]);
        const float4 qb = *reinterpret_cast<const float4*>(&sm.q[hh][half * KH + i * 8 + 4]);
        float s = z[hh];
        s = fmaf(qa.x, kf[0], s); s = fmaf(qa.y, kf[1], s);
        s = fmaf(qa.z, kf[2], s); s = fmaf(qa.w, kf[3], s);
        s = fmaf(qb.x, kf[4], s); s = fmaf(qb.y, kf[5], s);
        s = fmaf(qb.z, kf[6], s); s = fmaf(qb.w, kf[7], s);
        z[hh] = s;
      }
    }
    const bool valid = row >= 0;
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      const float zz = z[hh] + __shfl_xor_sync(0xffffffffu, z[hh], 1);
      const float y = valid ? zz * a.scale_log2 : -INFINITY;
      const float mn = fmaxf(m[hh], wmax_pairs(y));
      const float alpha = (m[hh] == -INFINITY) ? 0.f : exp2f(m[hh] - mn);
      const float p = valid ? exp2f(y - mn) : 0.f;
      lsum[hh] = lsum[hh] * alpha + wsum_pairs(p);
#pragma unroll
      for (int e = 0; e < DPL; ++e) acc[hh][e] *= alpha;
      m[hh] = mn;
      if (half == 0) sm.p[warp][lane >> 1][hh] = p;
    }
    __syncwarp();
    // ---- P.V: lane owns DPL dims of every row
#pragma unroll
    for (int kk = 0; kk < kKeysPerWarp; ++kk) {
      float vf[DPL];
#pragma unroll
      for (int e = 0; e < DPL / 2; ++e) {
        vf[2 * e] = bf16_lo(vr[kk][e]);
        vf[2 * e + 1] = bf16_hi(vr[kk][e]);
      }
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        const float p = sm.p[warp][kk][hh];
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[hh][e] = fmaf(p, vf[e], acc[hh][e]);
      }
    }
    __syncwarp();
  }

  // ---- merge the four warps in a fixed order
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    if (lane == 0) {
      sm.wm[warp][hh] = m[hh];
      sm.wl[warp][hh] = lsum[hh];
    }
#pragma unroll
    for (int e = 0; e < DPL; ++e) sm.wo[warp][hh][lane * DPL + e] = acc[hh][e];
  }
  __syncthreads();
  const bool direct = n_splits <= 1;
  const size_t slot = (static_cast<size_t>(b) * a.Hkv + g) * a.max_splits + split;
  float* wsl = direct ? nullptr : a.ws + slot * G * (D + 2);
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
      wsl[2 * G + hh * D + dim] = o;
      if (dim == 0) {
        wsl[hh] = M;
        wsl[G + hh] = Lh;
      }
    }
  }
}

// Combine the splits of one (pair, head): block (pair, head), thread = dim.
template <int D, int G>
__global__ void __launch_bounds__(D) sparse_merge_kernel(const SParams a) {
  __shared__ float wgt[kMaxSplits];
  __shared__ float inv_l;
  const int pair = blockIdx.x;
  const int hh = blockIdx.y;
  const int b = pair / a.Hkv, g = pair - (pair / a.Hkv) * a.Hkv;
  ptx::pdl_wait_primary();  // every split has written its partial
  const SList L = attended_list(a, b, false);
  const int n_splits = (L.total + a.split_len - 1) / a.split_len;
  if (n_splits <= 1) return;  // written directly by the split kernel
  const size_t stride = static_cast<size_t>(G) * (D + 2);
  const float* ws = a.ws + static_cast<size_t>(pair) * a.max_splits * stride;
  if (threadIdx.x < 32) {
    float M = -INFINITY;
    for (int s = threadIdx.x; s < n_splits; s += 32) M = fmaxf(M, ws[s * stride + hh]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float Ls = 0.f;
    for (int s = threadIdx.x; s < n_splits; s += 32) {
      const float ms = ws[s * stride + hh];
      const float w = (ms == -INFINITY) ? 0.f : exp2f(ms - M);
      wgt[s] = w;
      Ls += w * ws[s * stride + G + hh];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
    if (threadIdx.x == 0) inv_l = Ls > 0.f ? 1.f / Ls : 0.f;
  }
  __syncthreads();
  const int dim = threadIdx.x;
  const float* po = ws + 2 * G + hh * D + dim;
  float acc = 0.f;
  for (int s0 = 0; s0 < n_splits; s0 += 8) {
    float x[8];  // eight partials in flight, summed in split order
#pragma unroll
    for (int u = 0; u < 8; ++u) x[u] = s0 + u < n_splits ? po[(s0 + u) * stride] : 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (s0 + u < n_splits) acc += wgt[s0 + u] * x[u];
  }
  const __nv_bfloat16 bv = __float2bfloat16_rn(acc * inv_l);
  a.out[(static_cast<size_t>(b) * a.Hq + g * G + hh) * D + dim] =
      *reinterpret_cast<const uint16_t*>(&bv);
}

template <int D, int G>
cudaError_t launch_dg(const SParams& p, int B, int Hkv, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.max_splits, Hkv, B);
  cfg.blockDim = dim3(kSThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, sparse_decode_kernel<D, G>, p);
  if (e != cudaSuccess || p.max_splits <= 1) return e;
  cfg.gridDim = dim3(B * Hkv, G, 1);
  cfg.blockDim = dim3(D, 1, 1);
  return cudaLaunchKernelEx(&cfg, sparse_merge_kernel<D, G>, p);
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

size_t sparse_workspace_bytes(const SparsePlan& plan, int B, int Hkv, int G, int head_dim) {
  if (plan.max_splits <= 1) return 0;
  return static_cast<size_t>(B) * Hkv * plan.max_splits * G * (head_dim + 2) * sizeof(float);
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
  p.status = sa.status;
  p.Hq = sa.Hq;
  p.Hkv = sa.Hkv;
  p.max_blocks = sa.max_blocks;
  p.num_blocks = sa.num_blocks;
  p.k_max = sa.k_max;
  p.split_len = plan.split_len;
  p.max_splits = plan.max_splits;
  p.scale_log2 = sa.scale * kLog2e;
#define VSD_SPARSE_CASE(DD, GG) \
  if (sa.d == DD && sa.G == GG) return launch_dg<DD, GG>(p, sa.B, sa.Hkv, stream);
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
