// tmap.h -- host-side TMA tensor maps for the tensor-core kernels: the
// driver's cuTensorMapEncodeTiled, looked up once through the runtime (no
// libcuda link), and a 3-D bf16 map with 128-byte swizzled boxes.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

namespace pa {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// 3-D bf16 tensor {inner, mid, outer} (row-major) with box {box_inner,
// box_mid, box_outer} and 128-byte swizzle.
inline bool make_tmap(CUtensorMap* map, const void* base, uint64_t inner, uint64_t mid,
                      uint64_t outer, uint32_t box_inner, uint32_t box_mid, uint32_t box_outer) {
  EncodeTiledFn fn = encode_tiled();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {inner, mid, outer};
  const cuuint64_t strides[2] = {inner * 2, inner * mid * 2};  // bytes, dims 1 and 2
  const cuuint32_t box[3] = {box_inner, box_mid, box_outer};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 paged pool [blocks][16 tokens][heads][d] seen as the 4-D tensor
// {d, token, head, block}: a box {64, 16, heads, 1} lands in shared memory as
// [head][token][64 elements], one KV head's 16 token rows contiguous, with
// 128-byte swizzle.
inline bool make_tmap_pool_heads(CUtensorMap* map, const void* base, uint64_t d, uint64_t heads,
                                 uint64_t blocks) {
  EncodeTiledFn fn = encode_tiled();
  if (fn == nullptr) return false;
  const cuuint64_t dims[4] = {d, 16, heads, blocks};
  const cuuint64_t strides[3] = {heads * d * 2, d * 2, 16 * heads * d * 2};  // bytes, dims 1..3
  const cuuint32_t box[4] = {64, 16, static_cast<cuuint32_t>(heads), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace pa
