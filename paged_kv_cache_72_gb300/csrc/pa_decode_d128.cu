// Decode / gather kernels for head_dim 128.
#include "pa_decode_variants.cuh"

namespace pa {
int decode_ctas_per_sm_d128(const DecodePlan& p, int* ctas) {
  return ctas_per_sm_impl<128, false>(p, ctas);
}
int decode_launch_d128(const DecodePlan& p, const CUtensorMap& tk, const CUtensorMap& tv,
                       const DecodeArgs& a, cudaStream_t s) {
  return launch_impl<128, false>(p, tk, tv, a, s);
}
}  // namespace pa
