// cq_permute_f16.cu -- permute-quantise kernels for fp16 tokens (see
// cq_permute_impl.cuh); compiled apart from the bf16 ones to keep builds
// parallel.
#include "cq_permute_impl.cuh"

namespace cq {

cudaError_t launch_permute_f16(const PermuteArgs& a, cudaStream_t s) {
  return permute_detail::launch_typed<permute_detail::F16>(a, s);
}

}  // namespace cq
