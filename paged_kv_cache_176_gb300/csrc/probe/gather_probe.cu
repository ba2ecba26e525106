// gather_probe.cu -- the measurement aid of include/pa_probe.h (libpa_probe):
// stream a list of pool blocks (K and V) into a ring of shared-memory stages
// with the decode kernel's bulk copies and compute nothing.
#include "../../../include/pa_probe.h"
#include "../pa_common.cuh"
#include "../pa_trace.h"

namespace pa {
namespace {

constexpr int kProbeMaxStages = 8;

__global__ void __launch_bounds__(256, 1) gather_probe_kernel(const char* k, const char* v,
                                                              int64_t num_blocks,
                                                              const int32_t* blocks, int n,
                                                              int stages, int block_bytes,
                                                              int* d_status) {
  extern __shared__ __align__(128) char smem[];
  __shared__ __align__(8) uint64_t bars[kProbeMaxStages];
  const int tid = threadIdx.x;
  const int lo = static_cast<int>(static_cast<int64_t>(blockIdx.x) * n / gridDim.x);
  const int hi = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * n / gridDim.x);
  const int cnt = hi - lo;
  if (tid == 0) {
    for (int i = 0; i < stages; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  __syncthreads();
  auto issue = [&](int j) {
    const int st = j % stages;
    int64_t b = blocks[lo + j];
    if (b < 0 || b >= num_blocks) {
      status_or(d_status, PA_STATUS_BAD_BLOCK);
      b = 0;  // keep the copy in bounds
    }
    const int64_t off = b * block_bytes;
    mbar_arrive_expect_tx(&bars[st], 2u * static_cast<uint32_t>(block_bytes));
    bulk_g2s(smem + st * 2 * block_bytes, k + off, block_bytes, &bars[st]);
    bulk_g2s(smem + st * 2 * block_bytes + block_bytes, v + off, block_bytes, &bars[st]);
  };
  if (tid == 0)
    for (int j = 0; j < stages && j < cnt; ++j) issue(j);
  int i = 0;
  bool ok = true;
  for (; i < cnt; ++i) {
    ok = __syncthreads_and(mbar_wait_bounded(&bars[i % stages], (i / stages) & 1));
    if (!ok) break;
    if (tid == 0 && i + stages < cnt) issue(i + stages);
  }
  if (!ok && tid == 0) {
    status_or(d_status, PA_STATUS_TIMEOUT);
    for (int j = i; j < cnt && j < i + stages; ++j)  // copies still in flight
      mbar_wait_bounded(&bars[j % stages], (j / stages) & 1);
  }
}

}  // namespace
}  // namespace pa

extern "C" int pa_gather_probe(const pa_kv_pool* pool, const int32_t* blocks, int n, int stages,
                               int ctas, int* d_status, void* stream) {
  pa::TraceRange trace("pa_gather_probe");
  if (pool == nullptr || pool->k == nullptr || pool->v == nullptr || n < 0) return PA_EINVAL;
  if ((reinterpret_cast<uintptr_t>(pool->k) & 15u) || (reinterpret_cast<uintptr_t>(pool->v) & 15u))
    return PA_EINVAL;
  if (pool->num_blocks <= 0 || pool->num_kv_heads <= 0 || pool->head_dim <= 0) return PA_EINVAL;
  if (pool->block_size != pa::kBlockSize) return PA_EUNSUPPORTED;
  if (pool->dtype != PA_F32 && pool->dtype != PA_BF16) return PA_EUNSUPPORTED;
  const int64_t elt = pool->dtype == PA_BF16 ? 2 : 4;
  const int64_t bytes = static_cast<int64_t>(pa::kBlockSize) * pool->num_kv_heads * pool->head_dim * elt;
  if (bytes % 16 != 0) return PA_EUNSUPPORTED;
  if (stages < 1 || stages > pa::kProbeMaxStages || stages * 2 * bytes > 227 * 1024) return PA_EINVAL;
  if (n == 0) return PA_OK;
  if (blocks == nullptr) return PA_EINVAL;
  const int smem = static_cast<int>(stages * 2 * bytes);
  if (cudaFuncSetAttribute(pa::gather_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return PA_ECUDA;
  int grid = ctas;
  if (grid <= 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&grid, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return PA_ECUDA;
    }
  }
  pa::gather_probe_kernel<<<grid, 256, smem, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const char*>(pool->k), static_cast<const char*>(pool->v), pool->num_blocks, blocks,
      n, stages, static_cast<int>(bytes), d_status);
  if (cudaGetLastError() != cudaSuccess) return PA_ECUDA;
  return PA_OK;
}
