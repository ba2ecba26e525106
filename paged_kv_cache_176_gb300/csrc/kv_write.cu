// kv_write.cu -- the KV write ("reshape and cache").
//
// Token t with slot_mapping[t] >= 0 lands in physical block slot / 16 at
// offset slot % 16; its K (and V) row of num_kv_heads * head_dim values is
// contiguous in both k_new and the pool, so the write is a byte copy of one
// row per token, done with 16-byte vector stores. The cache of a sequence
// grows this way block by block ("Chunked Prefill" page, how chunked prefill
// works; "vLLM serving internals", PagedAttention as a virtual memory system).
#include "../../include/pa_serving.h"
#include "pa_common.cuh"
#include "pa_internal.h"
#include "pa_trace.h"

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

// One CTA per (src, dst) pair: copy block src of the K and V pools onto
// block dst (copy-on-write of a shared block).
__global__ void __launch_bounds__(256) copy_blocks_kernel(uint4* __restrict__ k_pool,
                                                          uint4* __restrict__ v_pool,
                                                          int64_t num_blocks, int vecs_per_block,
                                                          const int32_t* __restrict__ src,
                                                          const int32_t* __restrict__ dst,
                                                          int* d_status) {
  const int i = blockIdx.x;
  const int64_t s = src[i], d = dst[i];
  if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
    if (threadIdx.x == 0) status_or(d_status, PA_STATUS_BAD_BLOCK);
    return;
  }
  for (int v = threadIdx.x; v < vecs_per_block; v += blockDim.x) {
    k_pool[d * vecs_per_block + v] = k_pool[s * vecs_per_block + v];
    v_pool[d * vecs_per_block + v] = v_pool[s * vecs_per_block + v];
  }
}

// One launch for a step's KV write and its copy-on-write copies. CTAs
// 0 .. num_tokens-1 write one new token each (as kv_write_kernel); CTA
// num_tokens + i copies the first ntok[i] token slots of block src[i] onto
// block dst[i], the filled part of a shared block that is about to receive
// new tokens at offsets >= ntok[i]. The copies and the writes touch disjoint
// slots, so they need no ordering inside the launch.
__global__ void __launch_bounds__(128) kv_write_cow_kernel(
    uint4* __restrict__ k_pool, uint4* __restrict__ v_pool, int64_t num_blocks, int vecs_per_token,
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
    const int64_t* __restrict__ slot_mapping, int num_tokens, const int32_t* __restrict__ src,
    const int32_t* __restrict__ dst, const int32_t* __restrict__ ntok, int* d_status) {
  const int b = blockIdx.x;
  if (b < num_tokens) {
    const int64_t slot = slot_mapping[b];
    if (slot < 0) return;  // padding token
    if (slot >= num_blocks * kBlockSize) {
      if (threadIdx.x == 0) status_or(d_status, PA_STATUS_BAD_SLOT);
      return;
    }
    const int64_t dst_v = slot * vecs_per_token;
    const int64_t src_v = static_cast<int64_t>(b) * vecs_per_token;
    for (int i = threadIdx.x; i < vecs_per_token; i += blockDim.x) {
      const uint4 kv = __ldg(k_new + src_v + i);
      const uint4 vv = __ldg(v_new + src_v + i);
      k_pool[dst_v + i] = kv;
      v_pool[dst_v + i] = vv;
    }
    return;
  }
  const int i = b - num_tokens;
  const int64_t s = src[i], d = dst[i];
  const int n = ntok[i];
  if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks || n < 0 || n > kBlockSize) {
    if (threadIdx.x == 0) status_or(d_status, PA_STATUS_BAD_BLOCK);
    return;
  }
  const int vecs = n * vecs_per_token;
  const int64_t so = s * kBlockSize * vecs_per_token, dof = d * kBlockSize * vecs_per_token;
  for (int v = threadIdx.x; v < vecs; v += blockDim.x) {
    k_pool[dof + v] = k_pool[so + v];
    v_pool[dof + v] = v_pool[so + v];
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

extern "C" int pa_copy_blocks(const pa_kv_pool* pool, const int32_t* src, const int32_t* dst,
                              int n, int* d_status, void* stream) {
  pa::TraceRange trace("pa_copy_blocks");
  if (pool == nullptr || pool->k == nullptr || pool->v == nullptr || n < 0) return PA_EINVAL;
  if ((reinterpret_cast<uintptr_t>(pool->k) & 15u) || (reinterpret_cast<uintptr_t>(pool->v) & 15u))
    return PA_EINVAL;
  if (pool->num_blocks <= 0 || pool->block_size != pa::kBlockSize) return PA_EUNSUPPORTED;
  if (pool->dtype != PA_F32 && pool->dtype != PA_BF16) return PA_EUNSUPPORTED;
  if (n == 0) return PA_OK;
  if (src == nullptr || dst == nullptr) return PA_EINVAL;
  const int64_t elt = pool->dtype == PA_BF16 ? 2 : 4;
  const int64_t bytes = static_cast<int64_t>(pa::kBlockSize) * pool->num_kv_heads * pool->head_dim * elt;
  if (bytes % 16 != 0) return PA_EUNSUPPORTED;
  pa::copy_blocks_kernel<<<n, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4*>(pool->k), static_cast<uint4*>(pool->v), pool->num_blocks,
      static_cast<int>(bytes / 16), src, dst, d_status);
  if (cudaGetLastError() != cudaSuccess) return PA_ECUDA;
  return PA_OK;
}

extern "C" int pa_reshape_and_cache_cow(const pa_kv_pool* pool, const void* k_new,
                                        const void* v_new, const int64_t* slot_mapping,
                                        int num_tokens, const int32_t* cow_src,
                                        const int32_t* cow_dst, const int32_t* cow_ntok,
                                        int n_cow, int* d_status, void* stream) {
  pa::TraceRange trace("pa_reshape_and_cache_cow");
  if (pool == nullptr || pool->k == nullptr || pool->v == nullptr || num_tokens < 0 || n_cow < 0)
    return PA_EINVAL;
  if ((reinterpret_cast<uintptr_t>(pool->k) & 15u) || (reinterpret_cast<uintptr_t>(pool->v) & 15u))
    return PA_EINVAL;
  if (pool->num_blocks <= 0 || pool->num_kv_heads <= 0 || pool->head_dim <= 0) return PA_EINVAL;
  if (pool->block_size != pa::kBlockSize) return PA_EUNSUPPORTED;
  if (pool->dtype != PA_F32 && pool->dtype != PA_BF16) return PA_EUNSUPPORTED;
  const int64_t elt = pool->dtype == PA_BF16 ? 2 : 4;
  const int64_t token_bytes = static_cast<int64_t>(pool->num_kv_heads) * pool->head_dim * elt;
  if (token_bytes % 16 != 0) return PA_EUNSUPPORTED;
  if (num_tokens > 0) {
    if (k_new == nullptr || v_new == nullptr || slot_mapping == nullptr) return PA_EINVAL;
    if ((reinterpret_cast<uintptr_t>(k_new) & 15u) || (reinterpret_cast<uintptr_t>(v_new) & 15u))
      return PA_EINVAL;
  }
  if (n_cow > 0 && (cow_src == nullptr || cow_dst == nullptr || cow_ntok == nullptr)) return PA_EINVAL;
  if (num_tokens + n_cow == 0) return PA_OK;
  const int vecs = static_cast<int>(token_bytes / 16);
  pa::kv_write_cow_kernel<<<num_tokens + n_cow, 128, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4*>(pool->k), static_cast<uint4*>(pool->v), pool->num_blocks, vecs,
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slot_mapping, num_tokens,
      cow_src, cow_dst, cow_ntok, d_status);
  if (cudaGetLastError() != cudaSuccess) return PA_ECUDA;
  return PA_OK;
}
