// decode_bf16_d256.cu -- decode kernels for bf16 pools with head_dim 256.
#include "decode_impl.cuh"

namespace pa {
cudaError_t decode_bf16_d256(const DecodeArgs& a, int group, cudaStream_t stream) {
  return dispatch_decode_d<__nv_bfloat16, 256>(a, group, stream);
}
}  // namespace pa
