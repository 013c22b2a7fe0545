// sparse_decode.cu -- sparse draft-step attention on sm_103a.
//
// What it computes ("Vegas" technical summary, sec. 2 drafting phase and sec. 3
// sparse execution): one query row per head attends only the selected positions
// (paged attention with page size 1 whose page indices are the selected token
// indices) plus the tokens appended after the selection (dense tail).
//
// How (GB300 design): the work of one (sequence, KV head) pair is the list
// idx[0 .. n_sel) ++ [tail_start, seq_len).  A thread-block cluster of up to 16 CTAs
// takes one pair; each CTA takes a contiguous slice of the list and its 8 warps take
// batches of 32 positions.  Per batch:
//   * each lane translates one position through the block table and gathers that
//     key's K row (head_dim x bf16, 16-byte loads) while the warp also issues the V
//     loads of all 32 rows (each lane a slice of every row, so V reads are coalesced);
//   * lane = key: the G query heads' logits are plain fp32 dot products (q in shared
//     memory, broadcast reads); one warp max per head gives the online-softmax update;
//   * lane = dims: V rows are accumulated with the batch's probabilities.
// Warps merge in shared memory in a fixed order; CTAs of the cluster merge through
// distributed shared memory in rank order, so results are bit-reproducible.  No
// global workspace, no atomics on results, no inter-CTA waits beyond the cluster
// barrier.
#include <cooperative_groups.h>

#include <cfloat>

#include "common.cuh"
#include "launch.h"

namespace cg = cooperative_groups;

namespace vsd {
namespace {

constexpr int kWarps = 8;
constexpr int kThreadsS = kWarps * 32;
constexpr int kPageS = 16;
constexpr int kMaxCluster = 16;

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
  unsigned* status;
  int Hq, Hkv, max_blocks, num_blocks, k_max;
  float scale_log2;
};

template <int D, int G>
struct SSmem {
  float q[G][D];
  uint32_t rows[kWarps][32];
  float p[kWarps][32][G];
  float wm[kWarps][G];
  float wl[kWarps][G];
  float part_m[G];
  float part_l[G];
  float part_o[G][D];
};

__device__ __forceinline__ float wmax(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float wsum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <int D, int G>
__global__ void __launch_bounds__(kThreadsS, 1) sparse_decode_kernel(const SParams a) {
  constexpr int DPL = D / 32;  // dims per lane when lanes own dims
  constexpr uint32_t kNoRow = 0xFFFFFFFFu;
  __shared__ __align__(16) SSmem<D, G> sm;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int C = static_cast<int>(cluster.num_blocks());
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // queries of the group, widened to fp32
  for (int i = threadIdx.x; i < G * D; i += kThreadsS) {
    const int hh = i / D, dim = i % D;
    const uint16_t raw = a.q[(static_cast<size_t>(b) * a.Hq + g * G + hh) * D + dim];
    sm.q[hh][dim] = __uint_as_float(static_cast<uint32_t>(raw) << 16);
  }

  // the attended list of this pair: idx[0 .. ns) then tail_start .. seq_len-1
  int ns = a.n_sel != nullptr ? __ldg(a.n_sel + b) : 0;
  const int t0 = __ldg(a.tail_start + b);
  const int t1 = __ldg(a.seq_len + b);
  bool ok_len = ns >= 0 && ns <= a.k_max && t0 >= 0 && t0 <= t1 &&
                static_cast<long long>(t1) <= static_cast<long long>(a.max_blocks) * kPageS;
  if (!ok_len) {
    if (threadIdx.x == 0 && rank == 0 && g == 0) flag_status(a.status, VSD_DEV_BAD_LENGTH);
    ns = 0;
  }
  const int total = ok_len ? ns + (t1 - t0) : 0;
  const int per = (total + C - 1) / C;
  const int lo = rank * per;
  const int hi = min(lo + per, total);
  __syncthreads();

  float m[G], lpart[G], acc[G][DPL];
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    m[hh] = -INFINITY;
    lpart[hh] = 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[hh][e] = 0.f;
  }

  for (int start = lo + warp * 32; start < hi; start += kWarps * 32) {
    const int pos = start + lane;
    uint32_t my_row = kNoRow;
    if (pos < hi) {
      const int j = pos < ns ? __ldg(a.idx + static_cast<size_t>(b) * a.k_max + pos) : t0 + (pos - ns);
      if (j < 0 || j >= t1) {
        flag_status(a.status, VSD_DEV_BAD_INDEX);
      } else {
        const int blk = __ldg(a.block_table + static_cast<size_t>(b) * a.max_blocks + j / kPageS);
        if (blk < 0 || blk >= a.num_blocks) {
          flag_status(a.status, VSD_DEV_BAD_BLOCK);
        } else {
          my_row = (static_cast<uint32_t>(blk) * a.Hkv + g) * kPageS + (j % kPageS);
        }
      }
    }
    sm.rows[warp][lane] = my_row;
    __syncwarp();
    // K row of this lane's key
    uint4 kr[D / 8];
    if (my_row != kNoRow) {
      const uint16_t* src = a.k_cache + static_cast<size_t>(my_row) * D;
#pragma unroll
      for (int i = 0; i < D / 8; ++i) kr[i] = ldg_stream16(src + i * 8);
    } else {
#pragma unroll
      for (int i = 0; i < D / 8; ++i) kr[i] = make_uint4(0, 0, 0, 0);
    }
    // this lane's slice of the V rows of all 32 keys
    uint32_t vr[32][DPL / 2];
#pragma unroll
    for (int kk = 0; kk < 32; ++kk) {
      const uint32_t r = sm.rows[warp][kk];
      if (r != kNoRow) {
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
    // logits of this lane's key for the G heads
    float z[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) z[hh] = 0.f;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      float kf[8];
      kf[0] = bf16_lo(kr[i].x); kf[1] = bf16_hi(kr[i].x);
      kf[2] = bf16_lo(kr[i].y); kf[3] = bf16_hi(kr[i].y);
      kf[4] = bf16_lo(kr[i].z); kf[5] = bf16_hi(kr[i].z);
      kf[6] = bf16_lo(kr[i].w); kf[7] = bf16_hi(kr[i].w);
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        const float4 qa = *reinterpret_cast<const float4*>(&sm.q[hh][i * 8]);
        const float4 qb = *reinterpret_cast<const float4*>(&sm.q[hh][i * 8 + 4]);
        float s = z[hh];
        s = fmaf(qa.x, kf[0], s); s = fmaf(qa.y, kf[1], s);
        s = fmaf(qa.z, kf[2], s); s = fmaf(qa.w, kf[3], s);
        s = fmaf(qb.x, kf[4], s); s = fmaf(qb.y, kf[5], s);
        s = fmaf(qb.z, kf[6], s); s = fmaf(qb.w, kf[7], s);
        z[hh] = s;
      }
    }
    const bool valid = my_row != kNoRow;
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      const float y = valid ? z[hh] * a.scale_log2 : -INFINITY;
      const float mn = fmaxf(m[hh], wmax(y));
      const float alpha = (m[hh] == -INFINITY) ? 0.f : exp2f(m[hh] - mn);
      const float p = valid ? exp2f(y - mn) : 0.f;
      lpart[hh] = lpart[hh] * alpha + p;
#pragma unroll
      for (int e = 0; e < DPL; ++e) acc[hh][e] *= alpha;
      m[hh] = mn;
      sm.p[warp][lane][hh] = p;
    }
    __syncwarp();
#pragma unroll
    for (int kk = 0; kk < 32; ++kk) {
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

  // ---- merge the warps of this CTA in a fixed order
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    const float lw = wsum(lpart[hh]);
    if (lane == 0) {
      sm.wm[warp][hh] = m[hh];
      sm.wl[warp][hh] = lw;
    }
  }
  __syncthreads();
  float f[G];
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.wm[w][hh]);
    f[hh] = (sm.wm[warp][hh] == -INFINITY) ? 0.f : exp2f(sm.wm[warp][hh] - M);
    if (warp == 0 && lane == 0) {
      float L = 0.f;
      for (int w = 0; w < kWarps; ++w)
        if (sm.wm[w][hh] != -INFINITY) L += sm.wl[w][hh] * exp2f(sm.wm[w][hh] - M);
      sm.part_m[hh] = M;
      sm.part_l[hh] = L;
    }
  }
  for (int w = 0; w < kWarps; ++w) {
    if (warp == w) {
#pragma unroll
      for (int hh = 0; hh < G; ++hh)
#pragma unroll
        for (int e = 0; e < DPL; ++e) {
          const float val = acc[hh][e] * f[hh];
          float* dst = &sm.part_o[hh][lane * DPL + e];
          *dst = (w == 0) ? val : *dst + val;
        }
    }
    __syncthreads();
  }

  // ---- merge the CTAs of the cluster through distributed shared memory
  cluster.sync();
  if (rank == 0) {
    for (int i = threadIdx.x; i < G * D; i += kThreadsS) {
      const int hh = i / D, dim = i % D;
      float M = -INFINITY;
      for (int r = 0; r < C; ++r) {
        const SSmem<D, G>* other = cluster.map_shared_rank(&sm, r);
        M = fmaxf(M, other->part_m[hh]);
      }
      float L = 0.f, o = 0.f;
      if (M != -INFINITY) {
        for (int r = 0; r < C; ++r) {
          const SSmem<D, G>* other = cluster.map_shared_rank(&sm, r);
          const float mr = other->part_m[hh];
          if (mr == -INFINITY) continue;
          const float w = exp2f(mr - M);
          L += w * other->part_l[hh];
          o += w * other->part_o[hh][dim];
        }
      }
      const float val = L > 0.f ? o / L : 0.f;
      const __nv_bfloat16 bv = __float2bfloat16_rn(val);
      a.out[(static_cast<size_t>(b) * a.Hq + g * G + hh) * D + dim] =
          *reinterpret_cast<const uint16_t*>(&bv);
    }
  }
  cluster.sync();  // keep every CTA's shared memory alive until rank 0 has read it
}

template <int D, int G>
cudaError_t launch_dg(const SParams& p, int B, int Hkv, int C, cudaStream_t stream) {
  auto kern = sparse_decode_kernel<D, G>;
  if (C > 8) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, Hkv, B);
  cfg.blockDim = dim3(kThreadsS, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

// Cluster size: enough CTAs that each warp sees about two batches of 32 positions.
static int sparse_cluster_size(int max_len) {
  const int per_cta = kWarps * 32 * 2;
  int C = (max_len + per_cta - 1) / per_cta;
  if (C < 1) C = 1;
  if (C > kMaxCluster) C = kMaxCluster;
  return C;
}

cudaError_t launch_sparse(const SparseArgs& sa, cudaStream_t stream) {
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
  p.status = sa.status;
  p.Hq = sa.Hq;
  p.Hkv = sa.Hkv;
  p.max_blocks = sa.max_blocks;
  p.num_blocks = sa.num_blocks;
  p.k_max = sa.k_max;
  p.scale_log2 = sa.scale * kLog2e;
  if (sa.B == 0) return cudaSuccess;
  const int C = sparse_cluster_size(sa.k_max + sa.max_tail);
#define VSD_SPARSE_CASE(DD, GG) \
  if (sa.d == DD && sa.G == GG) return launch_dg<DD, GG>(p, sa.B, sa.Hkv, C, stream);
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
