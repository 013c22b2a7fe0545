// verify_attn.cu -- host side of the verification kernel: the persistent grid plan,
// the split-K workspace size and the dispatch to the per-head-dimension
// instantiations (verify_attn_d128.cu, verify_attn_d64.cu).  The kernels themselves
// are in verify_attn.cuh.
#include "launch.h"

namespace vsd {

namespace verify_detail {
cudaError_t launch_verify_d128(const VerifyArgs& a, const VerifyPlan& plan, cudaStream_t s);
cudaError_t launch_verify_d64(const VerifyArgs& a, const VerifyPlan& plan, cudaStream_t s);
}  // namespace verify_detail

namespace {
constexpr int kTile = 128;
constexpr int kMaxCtas = 256;  // the merge kernel weighs at most this many partials
}  // namespace

VerifyPlan plan_verify(int B, int Hkv, int R, int G, int P_max, int num_sms) {
  VerifyPlan plan;
  plan.pairs = B * Hkv;
  plan.t_max = (P_max + R + kTile - 1) / kTile;
  const long long W = static_cast<long long>(plan.pairs) * plan.t_max;
  const int cap = num_sms < kMaxCtas ? num_sms : kMaxCtas;
  plan.ctas = static_cast<int>(W < cap ? W : cap);
  if (plan.ctas < 1) plan.ctas = 1;
  plan.nq = ((R * G + 15) / 16) * 16;
  // slots per pair: the most CTAs whose ranges [c W / C, (c+1) W / C) meet one pair
  int mc = 1;
  if (W > 0) {
    for (int p = 0; p < plan.pairs; ++p) {
      const long long f = static_cast<long long>(p) * plan.t_max;
      const long long l = f + plan.t_max - 1;
      const int cf = static_cast<int>(((f + 1) * plan.ctas - 1) / W);
      const int cl = static_cast<int>(((l + 1) * plan.ctas - 1) / W);
      if (cl - cf + 1 > mc) mc = cl - cf + 1;
    }
  }
  plan.max_chunks = mc;
  return plan;
}

size_t verify_workspace_bytes(const VerifyPlan& plan, int head_dim) {
  if (plan.max_chunks <= 1) return 0;
  return static_cast<size_t>(plan.pairs) * plan.max_chunks * plan.nq * (head_dim + 2) *
         sizeof(float);
}

cudaError_t launch_verify(const VerifyArgs& va, const VerifyPlan& plan, cudaStream_t stream) {
  if (plan.pairs == 0) return cudaSuccess;
  if (va.d == 128) return verify_detail::launch_verify_d128(va, plan, stream);
  if (va.d == 64) return verify_detail::launch_verify_d64(va, plan, stream);
  return cudaErrorInvalidValue;
}

}  // namespace vsd
