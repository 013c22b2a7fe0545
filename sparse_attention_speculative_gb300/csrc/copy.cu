// copy.cu -- the copies between pinned host memory and device memory of a decode
// iteration, as a kernel.
//
// Host memory that is pinned is addressable from the GPU (unified addressing over the
// CPU-GPU link).  A kernel that moves the iteration's inputs in and its results out
// 16 bytes per thread replaces a DMA copy node, and as a programmatic dependent its
// launch overlaps the tail of the preceding kernel.
#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace vsd {
namespace {

constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads) copy16_kernel(uint4* __restrict__ dst,
                                                              const uint4* __restrict__ src,
                                                              size_t n16) {
  ptx::pdl_wait_primary();  // the source may come from the preceding kernel
  ptx::pdl_launch_dependents();
  for (size_t i = static_cast<size_t>(blockIdx.x) * kCopyThreads + threadIdx.x; i < n16;
       i += static_cast<size_t>(gridDim.x) * kCopyThreads)
    dst[i] = src[i];
}

}  // namespace

cudaError_t launch_copy16(void* dst, const void* src, size_t bytes, cudaStream_t stream) {
  const size_t n16 = bytes / 16;
  if (n16 == 0) return cudaSuccess;
  int blocks = static_cast<int>((n16 + kCopyThreads - 1) / kCopyThreads);
  if (blocks > 1024) blocks = 1024;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks, 1, 1);
  cfg.blockDim = dim3(kCopyThreads, 1, 1);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, copy16_kernel, static_cast<uint4*>(dst),
                            static_cast<const uint4*>(src), n16);
}

}  // namespace vsd
