// kv_append.cu -- the cache bookkeeping of a decode iteration, as kernels.
//
// What it does ("Vegas" technical summary, sec. 2 core mechanism: every iteration
// verifies the drafts with a full forward pass, selects from that pass and drafts from
// the selection; sec. 3 integration: the draft tokens come from repeated forward
// passes of the target model).  Each forward pass writes the keys and values of the
// tokens it processes into the paged cache before their attention reads them, and the
// accepted count of a verification moves every sequence's prefix forward.
//   * append_kv_kernel: K/V rows of n_new tokens per sequence stored at consecutive
//     positions through the block table (one 16-byte chunk per thread).
//   * advance_kernel: prefix_len += accepted + 1, and the draft steps' dense tail
//     [old prefix, old prefix + accepted + 2 + i) for draft step i.
// Both are programmatic dependents that wait for their predecessor before touching
// memory and release their own dependents only after that wait, so a kernel that
// follows them can rely on everything issued before them being complete.
#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace vsd {
namespace {

constexpr int kAppendThreads = 256;
constexpr int kPageA = 16;

struct AppendParams {
  const uint4* k_new;  // [B][n_new][Hkv][d] bf16, as 16-byte chunks
  const uint4* v_new;
  const int32_t* block_table;
  const int32_t* pos_base;
  uint4* k_cache;  // [num_blocks][Hkv][16][d] bf16, as 16-byte chunks
  uint4* v_cache;
  unsigned* status;
  int B, n_new, Hkv, chunks;  // chunks: 16-byte pieces of one row (d / 8)
  int max_blocks, num_blocks, pos_offset;
};

__global__ void __launch_bounds__(kAppendThreads) append_kv_kernel(const AppendParams a) {
  ptx::pdl_wait_primary();  // the rows and positions may come from the preceding kernel
  ptx::pdl_launch_dependents();
  const long long total = static_cast<long long>(a.B) * a.n_new * a.Hkv * a.chunks;
  for (long long i = static_cast<long long>(blockIdx.x) * kAppendThreads + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * kAppendThreads) {
    // i = ((b * n_new + t) * Hkv + g) * chunks + c: the source order
    const int c = static_cast<int>(i % a.chunks);
    const long long row = i / a.chunks;
    const int g = static_cast<int>(row % a.Hkv);
    const long long bt = row / a.Hkv;
    const int t = static_cast<int>(bt % a.n_new);
    const int b = static_cast<int>(bt / a.n_new);
    const long long pos = static_cast<long long>(__ldcg(a.pos_base + b)) + a.pos_offset + t;
    if (pos < 0 || pos >= static_cast<long long>(a.max_blocks) * kPageA) {
      if (c == 0) flag_status(a.status, VSD_DEV_BAD_LENGTH);
      continue;
    }
    const int blk = __ldcg(a.block_table + static_cast<size_t>(b) * a.max_blocks +
                          static_cast<int>(pos / kPageA));
    if (blk < 0 || blk >= a.num_blocks) {
      if (c == 0) flag_status(a.status, VSD_DEV_BAD_BLOCK);
      continue;
    }
    const size_t dst =
        ((static_cast<size_t>(blk) * a.Hkv + g) * kPageA + static_cast<size_t>(pos % kPageA)) *
            a.chunks + c;
    a.k_cache[dst] = a.k_new[i];
    a.v_cache[dst] = a.v_new[i];
  }
}

struct AdvanceParams {
  const int32_t* accepted;
  int32_t* prefix_len;
  int32_t* tail_start;
  int32_t* seq_len;        // [gamma][B]
  int32_t* prefix_copies;  // [n_copies][B] or NULL
  unsigned* status;
  int B, gamma, max_prefix, n_copies;
};

__global__ void __launch_bounds__(kAppendThreads) advance_kernel(const AdvanceParams a) {
  ptx::pdl_wait_primary();  // every reader of the old lengths has completed
  ptx::pdl_launch_dependents();
  for (int b = blockIdx.x * kAppendThreads + threadIdx.x; b < a.B;
       b += gridDim.x * kAppendThreads) {
    const int P = a.prefix_len[b];
    const int acc = __ldcg(a.accepted + b);
    // the accepted drafts and the verify block's first token join the prefix; a count
    // outside [0, gamma] or a prefix past max_prefix is refused (lengths unchanged)
    const bool ok = acc >= 0 && acc <= a.gamma && P >= 0 &&
                    static_cast<long long>(P) + acc + 1 <= a.max_prefix;
    if (!ok) flag_status(a.status, VSD_DEV_BAD_LENGTH);
    const int grow = ok ? acc + 1 : 0;
    a.tail_start[b] = P;
    for (int i = 0; i < a.gamma; ++i) a.seq_len[static_cast<size_t>(i) * a.B + b] = P + grow + 1 + i;
    a.prefix_len[b] = P + grow;
    for (int r = 0; r < a.n_copies; ++r) a.prefix_copies[static_cast<size_t>(r) * a.B + b] = P + grow;
  }
}

cudaLaunchConfig_t pdl_config(cudaLaunchAttribute* attr, int blocks, cudaStream_t stream) {
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(kAppendThreads, 1, 1);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

}  // namespace

cudaError_t launch_append_kv(const AppendArgs& x, cudaStream_t stream) {
  AppendParams p;
  p.k_new = static_cast<const uint4*>(x.k_new);
  p.v_new = static_cast<const uint4*>(x.v_new);
  p.block_table = x.block_table;
  p.pos_base = x.pos_base;
  p.k_cache = static_cast<uint4*>(x.k_cache);
  p.v_cache = static_cast<uint4*>(x.v_cache);
  p.status = x.status;
  p.B = x.B;
  p.n_new = x.n_new;
  p.Hkv = x.Hkv;
  p.chunks = x.d / 8;
  p.max_blocks = x.max_blocks;
  p.num_blocks = x.num_blocks;
  p.pos_offset = x.pos_offset;
  const long long total = static_cast<long long>(x.B) * x.n_new * x.Hkv * p.chunks;
  if (total == 0) return cudaSuccess;
  long long blocks = (total + kAppendThreads - 1) / kAppendThreads;
  if (blocks > 1024) blocks = 1024;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(attr, static_cast<int>(blocks), stream);
  return cudaLaunchKernelEx(&cfg, append_kv_kernel, p);
}

cudaError_t launch_advance(const AdvanceArgs& x, cudaStream_t stream) {
  if (x.B == 0) return cudaSuccess;
  AdvanceParams p;
  p.accepted = x.accepted;
  p.prefix_len = x.prefix_len;
  p.tail_start = x.tail_start;
  p.seq_len = x.seq_len;
  p.prefix_copies = x.prefix_copies;
  p.status = x.status;
  p.B = x.B;
  p.gamma = x.gamma;
  p.max_prefix = x.max_prefix;
  p.n_copies = x.prefix_copies != nullptr ? x.n_copies : 0;
  const int blocks = (x.B + kAppendThreads - 1) / kAppendThreads;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(attr, blocks, stream);
  return cudaLaunchKernelEx(&cfg, advance_kernel, p);
}

}  // namespace vsd
