// decode_f32_d64.cu -- decode kernels for f32 pools with head_dim 64.
#include "decode_impl.cuh"

namespace pa {
cudaError_t decode_f32_d64(const DecodeArgs& a, int group, cudaStream_t stream) {
  return dispatch_decode_d<float, 64>(a, group, stream);
}
}  // namespace pa
