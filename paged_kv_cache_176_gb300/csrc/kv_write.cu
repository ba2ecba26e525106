// kv_write.cu -- the KV write ("reshape and cache").
//
// Token t with slot_mapping[t] >= 0 lands in physical block slot / 16 at
// offset slot % 16; its K (and V) row of num_kv_heads * head_dim values is
// contiguous in both k_new and the pool, so the write is a byte copy of one
// row per token, done with 16-byte vector stores. The cache of a sequence
// grows this way block by block ("Chunked Prefill" page, how chunked prefill
// works; "vLLM serving internals", PagedAttention as a virtual memory system).
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

// One CTA per token; each thread moves 16-byte vectors of K and V.
__global__ void __launch_bounds__(128) kv_write_kernel(uint4* __restrict__ k_pool,
                                                       uint4* __restrict__ v_pool,
                                                       int64_t num_slots, int vecs_per_token,
                                                       const uint4* __restrict__ k_new,
                                                       const uint4* __restrict__ v_new,
                                                       const int64_t* __restrict__ slot_mapping,
                                                       int* d_status) {
  const int t = blockIdx.x;
  const int64_t slot = slot_mapping[t];
  if (slot < 0) return;  // padding token
  if (slot >= num_slots) {
    if (threadIdx.x == 0) status_or(d_status, PA_STATUS_BAD_SLOT);
    return;
  }
  const int64_t block = slot / kBlockSize;
  const int64_t offset = slot - block * kBlockSize;
  const int64_t dst = (block * kBlockSize + offset) * vecs_per_token;
  const int64_t src = static_cast<int64_t>(t) * vecs_per_token;
  for (int i = threadIdx.x; i < vecs_per_token; i += blockDim.x) {
    const uint4 kv = __ldg(k_new + src + i);
    const uint4 vv = __ldg(v_new + src + i);
    k_pool[dst + i] = kv;
    v_pool[dst + i] = vv;
  }
}

}  // namespace

cudaError_t launch_kv_write(const KvWriteArgs& a, cudaStream_t stream) {
  if (a.num_tokens == 0) return cudaSuccess;
  const int elt = a.pool.dtype == PA_BF16 ? 2 : 4;
  const int token_bytes = a.pool.num_kv_heads * a.pool.head_dim * elt;
  const int vecs = token_bytes / 16;
  const int threads = vecs >= 128 ? 128 : ((vecs + 31) / 32) * 32;
  kv_write_kernel<<<a.num_tokens, threads, 0, stream>>>(
      static_cast<uint4*>(a.pool.k), static_cast<uint4*>(a.pool.v), a.pool.num_blocks * kBlockSize,
      vecs, static_cast<const uint4*>(a.k_new), static_cast<const uint4*>(a.v_new), a.slot_mapping,
      a.d_status);
  return cudaGetLastError();
}

}  // namespace pa
