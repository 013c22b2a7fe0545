// vsd_noalloc.cu -- the verification call for callers that cannot provide a workspace.
//
// vsd_verify_attn_collect needs device scratch for the split-K partial results of
// pairs that several CTAs share.  Normally the caller allocates it.  Some callers
// cannot: an engine that reserves all free HBM for its paged KV cache at start-up
// and has nothing left to hand out, or a host program that forbids cudaMalloc on the
// decode path because it can synchronize the whole device.  For them this file keeps
// the scratch in a fixed device array that lives as long as the library is loaded,
// and the entry point below allocates nothing.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/vsd.h"

namespace {

constexpr size_t kScratchBytes = static_cast<size_t>(VSD_NOALLOC_SCRATCH_BYTES);
constexpr int kMaxDevices = 64;

// The scratch itself.  Its host-side name is only a handle: host code must use the
// device address obtained from cudaGetSymbolAddress, never &g_noalloc_scratch.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch on the current device, looked up once per device.
vsd_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return VSD_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return VSD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return VSD_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return VSD_OK;
}

}  // namespace

extern "C" {

vsd_status vsd_verify_attn_collect_noalloc(const vsd_geom* geom, int R, const void* q,
                                           const void* k_cache, const void* v_cache,
                                           const int32_t* block_table,
                                           const int32_t* prefix_len, int collect_row0,
                                           int collect_row1, int P_max, float scale,
                                           float* logits, float* partial_scores, void* out,
                                           void* stream) {
  size_t need = 0;
  vsd_status st = vsd_verify_workspace_size(geom, R, P_max, &need);
  if (st != VSD_OK) return st;
  if (need > kScratchBytes) return VSD_ERR_WORKSPACE;  // larger than the fixed scratch
  void* scratch = nullptr;
  if (need > 0) {
    st = scratch_address(&scratch);
    if (st != VSD_OK) return st;
  }
  // The partial-result slots are written before they are read in every call, so
  // nothing in the scratch has to start at zero.
  return vsd_verify_attn_collect(geom, R, q, k_cache, v_cache, block_table, prefix_len,
                                 collect_row0, collect_row1, P_max, scale, logits,
                                 partial_scores, out, scratch, need > 0 ? kScratchBytes : 0,
                                 stream);
}

}  // extern "C"
