// wait_probe.cu -- the test aid of include/pa_probe.h (libpa_probe): one CTA
// that goes through the kernels' bounded wait and give-up path, with no copy
// in flight.
//
// The attention kernels wait on mbarriers that their TMA / bulk copies
// complete. Each wait is bounded (mbar_wait_bounded_ns, pa_common.cuh); when it
// gives up, the kernel records PA_STATUS_TIMEOUT, stops, releases the TMEM it
// holds and returns. A copy that never completes cannot be produced safely on
// purpose, so this kernel arms its barrier for a transfer it never starts: the
// wait then runs out exactly as it would for a lost copy, and nothing is left
// in flight when the CTA exits.
#include "../../../include/pa_probe.h"
#include "../pa_common.cuh"
#include "../pa_trace.h"
#include "../tc_common.cuh"

namespace pa {
namespace {

constexpr uint32_t kProbeBytes = 1024;   // one bulk copy
constexpr uint32_t kProbeTmemCols = 32;  // the smallest TMEM allocation
constexpr int kProbeThreads = 128;

__global__ void __launch_bounds__(kProbeThreads, 1)
    wait_probe_kernel(const uint4* src, int starve, unsigned long long limit_ns, int* d_status) {
  __shared__ __align__(128) uint4 buf[kProbeBytes / 16];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {  // hold TMEM like the tensor-core kernels do
    tc::tmem_alloc(&tmem_base, kProbeTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  if (tid == 0) {
    mbar_arrive_expect_tx(&bar, kProbeBytes);
    if (!starve) bulk_g2s(buf, src, kProbeBytes, &bar);  // starve: armed, never started
  }
  // every warp waits on the stage, as the consumer warps of the kernels do
  if (!mbar_wait_bounded_ns(&bar, 0, limit_ns)) atomicOr(&abort_flag, 1);
  __syncthreads();
  if (abort_flag != 0) {
    if (tid == 0) status_or(d_status, PA_STATUS_TIMEOUT);
  } else if (tid < static_cast<int>(kProbeBytes / 16)) {
    // the copy landed: check its bytes (a mismatch would be a copy error)
    const uint4 a = buf[tid], b = src[tid];
    if (a.x != b.x || a.y != b.y || a.z != b.z || a.w != b.w) status_or(d_status, PA_STATUS_BAD_BLOCK);
  }
  // the give-up path and the normal path both release TMEM before returning
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, kProbeTmemCols);
}

}  // namespace
}  // namespace pa

extern "C" int pa_wait_probe(const void* src, int starve, unsigned long long limit_ns,
                             int* d_status, void* stream) {
  pa::TraceRange trace("pa_wait_probe");
  if (src == nullptr || (reinterpret_cast<uintptr_t>(src) & 15u) != 0) return PA_EINVAL;
  if (limit_ns == 0 || limit_ns > pa::kWaitLimitNs) return PA_EINVAL;
  pa::wait_probe_kernel<<<1, pa::kProbeThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(src), starve ? 1 : 0, limit_ns, d_status);
  if (cudaGetLastError() != cudaSuccess) return PA_ECUDA;
  return PA_OK;
}
