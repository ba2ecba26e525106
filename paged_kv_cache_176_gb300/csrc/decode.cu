// decode.cu -- host side of the decode path: workspace size, support
// matrix, and dispatch to the per-(dtype, head_dim) kernels.
#include "pa_internal.h"

namespace pa {

size_t decode_workspace_bytes(int num_seqs, int num_q_heads, int head_dim) {
  return decode_workspace_bytes_slots(num_seqs, num_q_heads, head_dim,
                                      static_cast<size_t>(kMaxDecodeCtas) + num_seqs);
}

size_t decode_workspace_bytes_slots(int num_seqs, int num_q_heads, int head_dim, size_t slots) {
  // [num_seqs + 1] block prefix, then per partial slot (CTA c, sequence s at
  // slot c + s without sibling groups) the (max, sum) pair and the fp32
  // accumulator of every head
  const size_t prefix_bytes = align_up_sz((num_seqs + 1) * 4, 256);
  const size_t ml = align_up_sz(slots * num_q_heads * 8, 256);
  const size_t acc = slots * num_q_heads * static_cast<size_t>(head_dim) * 4;
  return prefix_bytes + ml + acc;
}

bool decode_supported(int dtype, int head_dim, int group, int num_kv_heads) {
  if (dtype != PA_F32 && dtype != PA_BF16) return false;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return false;
  if (group != 1 && group != 2 && group != 4 && group != 8) return false;
  return num_kv_heads == 1 || num_kv_heads == 2 || num_kv_heads == 4 || num_kv_heads == 8;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.num_seqs == 0) return cudaSuccess;
  const int group = a.num_q_heads / a.pool.num_kv_heads;
  const int d = a.pool.head_dim;
  if (a.pool.dtype == PA_BF16) {
    if (d == 64) return decode_bf16_d64(a, group, stream);
    if (d == 128) return decode_bf16_d128(a, group, stream);
    if (d == 256) return decode_bf16_d256(a, group, stream);
  } else {
    if (d == 64) return decode_f32_d64(a, group, stream);
    if (d == 128) return decode_f32_d128(a, group, stream);
    if (d == 256) return decode_f32_d256(a, group, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace pa
