// common.cuh -- small device helpers shared by the three kernels of libvsd.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/vsd.h"

namespace vsd {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void flag_status(unsigned* status, unsigned bits) {
  if (status != nullptr) atomicOr(status, bits);
}

__device__ __forceinline__ float bf16_lo(uint32_t packed) {
  return __uint_as_float(packed << 16);
}

__device__ __forceinline__ float bf16_hi(uint32_t packed) {
  return __uint_as_float(packed & 0xFFFF0000u);
}

// Round two floats to bf16 (nearest even) and pack them, `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float fast_exp2(float x) { return exp2f(x); }

// Loads of anything a preceding kernel may have written.  Every kernel here is a
// programmatic dependent of its predecessor, so such data is read only after the wait
// for it, and never through the non-coherent read-only path: a load the compiler treats
// as read-only for the kernel's lifetime may be moved above that wait.  These go to L2
// (the data is used once or is small).
__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

__device__ __forceinline__ uint2 ldg_stream8(const void* p) {
  uint2 v;
  asm volatile("ld.global.cg.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ldg_stream4(const void* p) {
  uint32_t v;
  asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

}  // namespace vsd
