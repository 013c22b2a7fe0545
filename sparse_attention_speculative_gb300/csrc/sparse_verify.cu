// sparse_verify.cu -- the compressed cache of sparse verification on sm_103a.
//
// What it computes (Dustin technical summary, "Verification workflow", steps 3-4): a
// compressed target KV cache is formed from the selected tokens only, and the draft
// block is verified against it.  Verify row t of sequence b then attends
// idx[b, 0 .. n_sel[b]) followed by the verify block P_b .. P_b + t.
//
// How (GB300 design).  This kernel writes that compressed cache as an ordinary paged
// cache in the workspace: sequence b's compact position p holds the K and V rows of
// token idx[b, p] for p < n_sel[b] and of token P_b + (p - n_sel[b]) for the R verify
// rows after them, pages numbered b * pages_per_seq + p / 16.  The verification
// kernel then runs unchanged on it with prefix length n_sel[b]: the selected tokens
// are its prefix and the verify block keeps its causal structure.  So sparse
// verification uses the same TMA-streamed tcgen05 tiles as full verification, over
// n_sel + R keys instead of P + R.
//
// The gather: one CTA per 64 compact positions of one (sequence, KV head); a row of
// head_dim bf16 is copied by head_dim / 8 lanes with 16-byte loads and stores, and
// all loads of a CTA are issued before any store.  The CTA that owns the first
// positions of a sequence also writes its block-table row and its compact prefix
// length.
#include "common.cuh"
#include "launch.h"

namespace vsd {
namespace {

constexpr int kGThreads = 256;
constexpr int kGPositions = 64;  // compact positions per CTA
constexpr int kPageG = 16;

template <int D>
__global__ void __launch_bounds__(kGThreads) sparse_verify_gather_kernel(const SparseVerifyArgs a,
                                                                         int pages_per_seq) {
  constexpr int LPR = D / 8;                  // lanes (16-byte chunks) per row
  constexpr int kRows = kGThreads / LPR;      // rows per pass
  constexpr int kPasses = kGPositions / kRows;
  const int b = blockIdx.z, g = blockIdx.y;
  const int p0 = blockIdx.x * kGPositions;
  const int t = threadIdx.x;
  const int r_in = t / LPR, ch = t % LPR;
  const uint16_t* kc = static_cast<const uint16_t*>(a.k_cache);
  const uint16_t* vc = static_cast<const uint16_t*>(a.v_cache);
  uint16_t* ck = a.compact_k;
  uint16_t* cv = a.compact_v;

  int ns = a.n_sel != nullptr ? __ldcg(a.n_sel + b) : 0;
  const int P = __ldcg(a.prefix_len + b);
  const bool ok = ns >= 0 && ns <= a.k_max && P >= 0 &&
                  static_cast<long long>(P) + a.R <= static_cast<long long>(a.max_blocks) * kPageG;
  if (!ok) {
    if (t == 0 && g == 0 && blockIdx.x == 0) flag_status(a.status, VSD_DEV_BAD_LENGTH);
    ns = 0;
  }
  const int n_used = ok ? ns + a.R : 0;  // compact positions holding a token
  if (blockIdx.x == 0 && g == 0) {
    for (int i = t; i < pages_per_seq; i += kGThreads)
      a.compact_table[static_cast<size_t>(b) * pages_per_seq + i] = b * pages_per_seq + i;
    if (t == 0) a.compact_prefix[b] = ns;
  }

  uint4 kv[kPasses], vv[kPasses];
  size_t dst[kPasses];
  bool have[kPasses];
#pragma unroll
  for (int u = 0; u < kPasses; ++u) {
    const int p = p0 + u * kRows + r_in;
    have[u] = false;
    kv[u] = vv[u] = make_uint4(0, 0, 0, 0);
    dst[u] = 0;
    if (p < n_used) {
      const int j = p < ns ? __ldcg(a.idx + static_cast<size_t>(b) * a.k_max + p) : P + (p - ns);
      if (j < 0 || j >= P + a.R) {
        if (ch == 0) flag_status(a.status, VSD_DEV_BAD_INDEX);
      } else {
        const int blk = __ldcg(a.block_table + static_cast<size_t>(b) * a.max_blocks + j / kPageG);
        if (blk < 0 || blk >= a.num_blocks) {
          if (ch == 0) flag_status(a.status, VSD_DEV_BAD_BLOCK);
        } else {
          const size_t src = ((static_cast<size_t>(blk) * a.Hkv + g) * kPageG + j % kPageG) * D +
                             ch * 8;
          kv[u] = ldg_stream16(kc + src);
          vv[u] = ldg_stream16(vc + src);
        }
      }
      // an invalid token leaves a zero row (its sequence's output is unspecified)
      have[u] = true;
      dst[u] = ((static_cast<size_t>(b) * pages_per_seq + p / kPageG) * a.Hkv + g) * kPageG * D +
               static_cast<size_t>(p % kPageG) * D + ch * 8;
    }
  }
#pragma unroll
  for (int u = 0; u < kPasses; ++u) {
    if (have[u]) {
      *reinterpret_cast<uint4*>(ck + dst[u]) = kv[u];
      *reinterpret_cast<uint4*>(cv + dst[u]) = vv[u];
    }
  }
}

}  // namespace

int sparse_verify_pages(int k_max, int R) { return (k_max + R + kPageG - 1) / kPageG; }

cudaError_t launch_sparse_verify_gather(const SparseVerifyArgs& a, cudaStream_t stream) {
  if (a.B == 0) return cudaSuccess;
  const int pps = sparse_verify_pages(a.k_max, a.R);
  dim3 grid((pps * kPageG + kGPositions - 1) / kGPositions, a.Hkv, a.B);
  if (a.d == 128)
    sparse_verify_gather_kernel<128><<<grid, kGThreads, 0, stream>>>(a, pps);
  else if (a.d == 64)
    sparse_verify_gather_kernel<64><<<grid, kGThreads, 0, stream>>>(a, pps);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace vsd
