// decode_static.cu -- pa_decode_static_ws: decode attention for callers that
// cannot hand the library a workspace.
//
// Some callers cannot allocate device memory around a decode call: a host
// framework that plans every device buffer up front and forbids its plugins to
// call cudaMalloc, or a latency-critical loop where cudaMalloc (which may
// synchronize the device and may fail under memory pressure) is not allowed.
// This entry point runs the same kernels as pa_decode, with the split-K
// scratch taken from a fixed array that lives in the library itself.
//
// The array is a file-scope static __device__ buffer of kStaticScratchBytes
// (32 MiB). Every GPU that loads this library keeps it allocated until the
// process exits. Host code cannot use the array's name as a device address, so
// the first call on each device looks the address up with
// cudaGetSymbolAddress (with that device current) and caches it; make that
// first call before any stream capture. The call allocates nothing.
//
// All calls share the one array and it keeps whatever the last call left in
// it. Nothing in it has to start at zero: on every path that completes, each
// value the merge kernel reads is written earlier by the same call. A call
// whose status word gets PA_STATUS_TIMEOUT (a copy that never completed) may
// leave partial slots unwritten, so its output is undefined, as for pa_decode.
// Calls whose work overlaps on the GPU (concurrent streams, or several host
// threads) race on the array; run them one after another.
//
// The cached address belongs to the CUDA context that was current when it was
// looked up. cudaDeviceReset (or anything else that destroys the device's
// primary context) unloads the module, so the cache is then stale: a process
// that resets a device must not call this entry point on it again.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/pa.h"
#include "pa_internal.h"
#include "pa_trace.h"

namespace pa {
namespace {

constexpr size_t kStaticScratchBytes = PA_DECODE_STATIC_WS_BYTES;

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device (looked up once).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    err = cudaGetSymbolAddress(&ptr, g_decode_scratch);
    if (err != cudaSuccess) return err;
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" {

int pa_decode_static_ws(const pa_kv_pool* pool, void* out, const void* q, int num_seqs,
                        int num_q_heads, const int32_t* block_tables, int max_blocks_per_seq,
                        const int32_t* context_lens, float scale, int* d_status, void* stream) {
  pa::TraceRange trace("pa_decode_static_ws");
  // pa_decode's own argument checks first, so that a bad or unsupported call
  // gets the same status as from pa_decode; then the size limit of the array
  int rc = check_decode_args(pool, out, q, num_seqs, num_q_heads, block_tables,
                             max_blocks_per_seq, context_lens);
  if (rc != PA_OK || num_seqs == 0) return rc;
  const size_t need = pa_decode_workspace_size(num_seqs, num_q_heads, pool->head_dim,
                                               max_blocks_per_seq);
  if (need > kStaticScratchBytes) return PA_EWORKSPACE;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) {
    cudaGetLastError();
    return PA_ECUDA;
  }
  return pa_decode(pool, out, q, num_seqs, num_q_heads, block_tables, max_blocks_per_seq,
                   context_lens, scale, scratch, kStaticScratchBytes, d_status, stream);
}

}  // extern "C"
