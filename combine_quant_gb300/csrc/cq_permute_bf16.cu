// cq_permute_bf16.cu -- permute-quantise kernels for bf16 tokens, and the
// launcher that picks the token type (see cq_permute_impl.cuh).
#include "cq_permute_impl.cuh"

namespace cq {

cudaError_t launch_permute_f16(const PermuteArgs& a, cudaStream_t s);  // cq_permute_f16.cu

cudaError_t launch_permute(const PermuteArgs& a, cudaStream_t s) {
  if (a.d.x_dtype == 1) return launch_permute_f16(a, s);
  return permute_detail::launch_typed<permute_detail::BF16>(a, s);
}

}  // namespace cq
