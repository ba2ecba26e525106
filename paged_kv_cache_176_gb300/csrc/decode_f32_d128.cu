// decode_f32_d128.cu -- decode kernels for f32 pools with head_dim 128.
#include "decode_impl.cuh"

namespace pa {
cudaError_t decode_f32_d128(const DecodeArgs& a, int group, cudaStream_t stream) {
  return dispatch_decode_d<float, 128>(a, group, stream);
}
}  // namespace pa
