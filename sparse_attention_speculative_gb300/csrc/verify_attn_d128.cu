// verify_attn_d128.cu -- verification kernels instantiated for head_dim 128.
#include "verify_attn.cuh"

namespace vsd {
namespace verify_detail {

cudaError_t launch_verify_d128(const VerifyArgs& a, const VerifyPlan& plan, cudaStream_t s) {
  return launch_verify_d<128>(a, plan, s);
}

}  // namespace verify_detail
}  // namespace vsd
