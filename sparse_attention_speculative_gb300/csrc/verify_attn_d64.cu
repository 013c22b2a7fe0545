// verify_attn_d64.cu -- verification kernels instantiated for head_dim 64.
#include "verify_attn.cuh"

namespace vsd {
namespace verify_detail {

cudaError_t launch_verify_d64(const VerifyArgs& a, const VerifyPlan& plan, cudaStream_t s) {
  return launch_verify_d<64>(a, plan, s);
}

}  // namespace verify_detail
}  // namespace vsd
