// api.cu -- the C ABI declared in include/pa.h: host-side validation of the
// scalar arguments, workspace size queries, and dispatch to the kernels.
// Host validation never dereferences a device pointer; data-dependent checks
// happen in the kernels (see pa.h).
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "../../include/pa.h"
#include "pa_internal.h"
#include "pa_trace.h"

namespace pa {

int device_sm_count() {
  // cached per device: the attribute query is cheap but not free
  static std::mutex mu;
  static std::vector<int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  std::lock_guard<std::mutex> lock(mu);
  if (static_cast<int>(cache.size()) <= dev) cache.resize(dev + 1, 0);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Pool checks shared by every entry point (the KV write needs no more).
int check_pool_storage(const pa_kv_pool* pool) {
  if (pool == nullptr || pool->k == nullptr || pool->v == nullptr) return PA_EINVAL;
  if (!aligned16(pool->k) || !aligned16(pool->v)) return PA_EINVAL;
  if (pool->num_blocks <= 0 || pool->num_kv_heads <= 0 || pool->head_dim <= 0) return PA_EINVAL;
  if (pool->block_size != 16) return PA_EUNSUPPORTED;
  if (pool->dtype != PA_F32 && pool->dtype != PA_BF16) return PA_EUNSUPPORTED;
  const int64_t elt = pool->dtype == PA_BF16 ? 2 : 4;
  if ((pool->num_kv_heads * pool->head_dim * elt) % 16 != 0) return PA_EUNSUPPORTED;
  return PA_OK;
}

// Attention kernels are built for head_dim 64, 128 and 256.
int check_pool(const pa_kv_pool* pool) {
  int rc = check_pool_storage(pool);
  if (rc != PA_OK) return rc;
  if (pool->head_dim != 64 && pool->head_dim != 128 && pool->head_dim != 256) return PA_EUNSUPPORTED;
  return PA_OK;
}

PoolView view(const pa_kv_pool* pool) {
  PoolView v;
  v.k = pool->k;
  v.v = pool->v;
  v.num_blocks = pool->num_blocks;
  v.num_kv_heads = pool->num_kv_heads;
  v.head_dim = pool->head_dim;
  v.dtype = pool->dtype;
  return v;
}

int check_heads(const pa_kv_pool* pool, int num_q_heads) {
  if (num_q_heads <= 0) return PA_EINVAL;
  if (num_q_heads % pool->num_kv_heads != 0) return PA_EINVAL;
  const int group = num_q_heads / pool->num_kv_heads;
  if (group != 1 && group != 2 && group != 4 && group != 8) return PA_EUNSUPPORTED;
  return PA_OK;
}

int to_status(cudaError_t err) {
  if (err == cudaSuccess) return PA_OK;
  cudaGetLastError();  // clear a sticky launch error so the caller's next launch is clean
  return PA_ECUDA;
}

int validate_kv_write(const pa_kv_pool* pool, const void* k_new, const void* v_new,
                      const int64_t* slot_mapping, int num_tokens) {
  int rc = check_pool_storage(pool);
  if (rc != PA_OK) return rc;
  if (num_tokens < 0) return PA_EINVAL;
  if (num_tokens == 0) return PA_OK;
  if (k_new == nullptr || v_new == nullptr || slot_mapping == nullptr) return PA_EINVAL;
  if (!aligned16(k_new) || !aligned16(v_new)) return PA_EINVAL;
  return PA_OK;
}

}  // namespace

int check_decode_args(const pa_kv_pool* pool, const void* out, const void* q, int num_seqs,
                      int num_q_heads, const int32_t* block_tables, int max_blocks_per_seq,
                      const int32_t* context_lens) {
  int rc = check_pool(pool);
  if (rc != PA_OK) return rc;
  if (num_seqs < 0 || max_blocks_per_seq <= 0) return PA_EINVAL;
  rc = check_heads(pool, num_q_heads);
  if (rc != PA_OK) return rc;
  if (!decode_supported(pool->dtype, pool->head_dim, num_q_heads / pool->num_kv_heads,
                        pool->num_kv_heads))
    return PA_EUNSUPPORTED;
  if (num_seqs == 0) return PA_OK;
  if (out == nullptr || q == nullptr || block_tables == nullptr || context_lens == nullptr)
    return PA_EINVAL;
  if (!aligned16(out) || !aligned16(q)) return PA_EINVAL;
  return PA_OK;
}

}  // namespace pa

using namespace pa;

extern "C" {

const char* pa_strerror(int status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_EINVAL: return "invalid argument (null or misaligned pointer, bad size)";
    case PA_EUNSUPPORTED: return "unsupported configuration (block size, head_dim, head ratio or dtype)";
    case PA_EWORKSPACE: return "workspace missing or too small";
    case PA_EBUDGET: return "num_tokens exceeds token_budget";
    case PA_ECUDA: return "CUDA launch failed";
    default: return "unknown status";
  }
}

int pa_version(void) { return (1 << 16) | 0; }

int pa_reshape_and_cache(const pa_kv_pool* pool, const void* k_new, const void* v_new,
                         const int64_t* slot_mapping, int num_tokens, int* d_status,
                         void* stream) {
  pa::TraceRange trace("pa_reshape_and_cache");
  int rc = validate_kv_write(pool, k_new, v_new, slot_mapping, num_tokens);
  if (rc != PA_OK || num_tokens == 0) return rc;
  KvWriteArgs a;
  a.pool = view(pool);
  a.k_new = k_new;
  a.v_new = v_new;
  a.slot_mapping = slot_mapping;
  a.num_tokens = num_tokens;
  a.d_status = d_status;
  return to_status(launch_kv_write(a, static_cast<cudaStream_t>(stream)));
}

size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int head_dim,
                                int max_blocks_per_seq) {
  if (num_seqs < 0 || num_q_heads <= 0 || head_dim <= 0 || max_blocks_per_seq <= 0) return 0;
  return decode_workspace_bytes(num_seqs, num_q_heads, head_dim);
}

int pa_decode_with_ctas(const pa_kv_pool* pool, void* out, const void* q, int num_seqs,
                        int num_q_heads, const int32_t* block_tables, int max_blocks_per_seq,
                        const int32_t* context_lens, float scale, int num_ctas, void* workspace,
                        size_t workspace_bytes, int* d_status, void* stream) {
  pa::TraceRange trace("pa_decode");
  if (num_ctas < 0) return PA_EINVAL;
  int rc = check_decode_args(pool, out, q, num_seqs, num_q_heads, block_tables,
                             max_blocks_per_seq, context_lens);
  if (rc != PA_OK || num_seqs == 0) return rc;
  const size_t need = pa_decode_workspace_size(num_seqs, num_q_heads, pool->head_dim,
                                               max_blocks_per_seq);
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return PA_EWORKSPACE;
  DecodeArgs a = {};
  a.pool = view(pool);
  a.out = out;
  a.q = q;
  a.cu_q_lens = nullptr;
  a.num_seqs = num_seqs;
  a.num_rows = num_seqs;
  a.num_q_heads = num_q_heads;
  a.block_tables = block_tables;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.context_lens = context_lens;
  a.scale = scale;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.d_status = d_status;
  a.grid_override = num_ctas;
  return to_status(launch_decode(a, static_cast<cudaStream_t>(stream)));
}

int pa_decode(const pa_kv_pool* pool, void* out, const void* q, int num_seqs, int num_q_heads,
              const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
              float scale, void* workspace, size_t workspace_bytes, int* d_status, void* stream) {
  return pa_decode_with_ctas(pool, out, q, num_seqs, num_q_heads, block_tables, max_blocks_per_seq,
                             context_lens, scale, 0, workspace, workspace_bytes, d_status, stream);
}

namespace {
// Cascade workspace: the decode workspace (`slots` partial slots), then the
// prefix partials (max, sum) [num_seqs, hq] float2 and accumulators
// [num_seqs, hq, head_dim] fp32.
size_t cascade_ml_offset(int num_seqs, int num_q_heads, int head_dim, size_t slots) {
  return align_up_sz(decode_workspace_bytes_slots(num_seqs, num_q_heads, head_dim, slots), 256);
}
size_t cascade_acc_offset(int num_seqs, int num_q_heads, int head_dim, size_t slots) {
  return cascade_ml_offset(num_seqs, num_q_heads, head_dim, slots) +
         align_up_sz(static_cast<size_t>(num_seqs) * num_q_heads * 8, 256);
}
// ... then the decode kernel's per-sequence records for the merge, [num_seqs] uint32
size_t cascade_rec_offset(int num_seqs, int num_q_heads, int head_dim, size_t slots) {
  return cascade_acc_offset(num_seqs, num_q_heads, head_dim, slots) +
         align_up_sz(static_cast<size_t>(num_seqs) * num_q_heads * head_dim * 4, 256);
}
size_t cascade_bytes(int num_seqs, int num_q_heads, int head_dim, size_t slots) {
  return cascade_rec_offset(num_seqs, num_q_heads, head_dim, slots) +
         static_cast<size_t>(num_seqs) * 4;
}
size_t plain_slots(int num_seqs) { return static_cast<size_t>(kMaxDecodeCtas) + num_seqs; }
// Sibling entries of up to 16 / G members: a member of an entry that spans n
// CTAs leaves n partials, so the slots grow to num_seqs + (16 / G) * CTAs.
size_t nested_slots(int num_seqs, int group, int num_ctas) {
  const int ctas = num_ctas > 0 ? std::min(num_ctas, kMaxDecodeCtas) : kMaxDecodeCtas;
  return static_cast<size_t>(num_seqs) + static_cast<size_t>(16 / group) * ctas;
}

// Decode beside prefill: the decode kernel (HBM-bound) runs on a reduced set
// of persistent CTAs, and the tensor-core prefill or prefix kernel, launched
// right after it on the same stream as a programmatic dependent, takes the
// SMs it leaves free (it may start once every decode CTA has staged its
// blocks, and neither kernel waits for the other); the merge kernel, an
// ordinary launch, runs after both. On fewer SMs the decode no longer
// saturates HBM, so each of its SMs streams more bytes, and an SM a decode
// CTA leaves goes to the prefill.
//  - cascade decode: the decode streams the suffixes on all but
//    kCascadePrefixSms SMs beside the (short, latency-bound) prefix pass;
//  - mixed step: the decode takes kMixedDecodeSms SMs beside the prefill when
//    the prefill dominates the step. The host sees only counts: prefill
//    tokens P >= num_tokens - num_seqs, decode rows D <= num_seqs. A decode
//    row reads its whole context (a few to tens of MB), a prefill token costs
//    tensor work in proportion to its context, so the split is taken only
//    for P >= kMixedPrefillTokens and num_seqs <= P / kMixedTokensPerSeq
//    (a step of long prefill chunks and few decode rows); a decode-heavy
//    step (hundreds of decode rows beside short chunks) runs the prefill,
//    then the decode on all SMs.
constexpr int kCascadePrefixSms = 36;
constexpr int kMixedDecodeSms = 48;
constexpr int kMixedPrefillTokens = 1024;
constexpr int kMixedTokensPerSeq = 12;
}  // namespace

size_t pa_decode_cascade_workspace_size(int num_seqs, int num_q_heads, int head_dim,
                                        int max_blocks_per_seq) {
  if (num_seqs < 0 || num_q_heads <= 0 || head_dim <= 0 || max_blocks_per_seq <= 0) return 0;
  return cascade_bytes(num_seqs, num_q_heads, head_dim, plain_slots(num_seqs));
}

size_t pa_decode_cascade_nested_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                               int head_dim, int max_blocks_per_seq, int num_ctas) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      max_blocks_per_seq <= 0 || num_ctas < 0 || num_q_heads % num_kv_heads != 0)
    return 0;
  const int group = num_q_heads / num_kv_heads;
  if (group > 16) return 0;
  return cascade_bytes(num_seqs, num_q_heads, head_dim, nested_slots(num_seqs, group, num_ctas));
}

namespace {
// Both cascade entry points: the first level (cu_groups / prefix_lens, the
// tensor-core prefix pass) and, for the nested call, the second (cu_sib /
// shared_lens, sibling entries in the decode kernel).
int cascade_impl(const pa_kv_pool* pool, void* out, const void* q, int num_seqs, int num_q_heads,
                 const int32_t* block_tables, int max_blocks_per_seq,
                 const int32_t* context_lens, const int32_t* cu_groups,
                 const int32_t* prefix_lens, int num_groups, const int32_t* cu_sib,
                 const int32_t* shared_lens, int num_sib, bool nested, float scale, int num_ctas,
                 void* workspace, size_t workspace_bytes, int* d_status, void* stream) {
  if (num_ctas < 0) return PA_EINVAL;
  int rc = check_pool(pool);
  if (rc != PA_OK) return rc;
  if (num_seqs < 0 || max_blocks_per_seq <= 0 || num_groups < 0 || num_sib < 0) return PA_EINVAL;
  rc = check_heads(pool, num_q_heads);
  if (rc != PA_OK) return rc;
  const int group = num_q_heads / pool->num_kv_heads;
  if (!decode_supported(pool->dtype, pool->head_dim, group, pool->num_kv_heads) ||
      !prefix_supported(pool->dtype, pool->head_dim, group, num_groups))
    return PA_EUNSUPPORTED;
  if (num_seqs == 0) return PA_OK;
  if (out == nullptr || q == nullptr || block_tables == nullptr || context_lens == nullptr)
    return PA_EINVAL;
  if (num_groups > 0 && (cu_groups == nullptr || prefix_lens == nullptr)) return PA_EINVAL;
  if (num_sib > 0 && (cu_sib == nullptr || shared_lens == nullptr)) return PA_EINVAL;
  if (!aligned16(out) || !aligned16(q)) return PA_EINVAL;
  const size_t slots = nested ? nested_slots(num_seqs, group, num_ctas) : plain_slots(num_seqs);
  const size_t need = cascade_bytes(num_seqs, num_q_heads, pool->head_dim, slots);
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return PA_EWORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  void* pre_ml = ws + cascade_ml_offset(num_seqs, num_q_heads, pool->head_dim, slots);
  void* pre_acc = ws + cascade_acc_offset(num_seqs, num_q_heads, pool->head_dim, slots);
  DecodeArgs a = {};
  a.pool = view(pool);
  a.out = out;
  a.q = q;
  a.cu_q_lens = nullptr;
  a.num_seqs = num_seqs;
  a.num_rows = num_seqs;
  a.num_q_heads = num_q_heads;
  a.block_tables = block_tables;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.context_lens = context_lens;
  a.scale = scale;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.d_status = d_status;
  a.grid_override = num_ctas;
  a.ws_slots = slots;
  a.ws_rec = ws + cascade_rec_offset(num_seqs, num_q_heads, pool->head_dim, slots);
  if (num_sib > 0) {
    a.cu_sib = cu_sib;
    a.shared_lens = shared_lens;
    a.num_sib = num_sib;
  }
  if (num_groups == 0) return to_status(launch_decode(a, st));
  a.cu_groups = cu_groups;
  a.prefix_lens = prefix_lens;
  a.num_groups = num_groups;
  a.pre_ml = pre_ml;
  a.pre_acc = pre_acc;
  a.defer_prefix = 1;
  if (num_ctas == 0) a.grid_override = std::max(1, device_sm_count() - kCascadePrefixSms);
  // every group's decode rows against its shared prefix, once, on the tensor cores
  PrefillArgs pf = {};
  pf.pool = view(pool);
  pf.q = q;
  pf.cu_q_lens = cu_groups;
  pf.num_seqs = num_groups;
  pf.num_tokens = num_seqs;
  pf.num_q_heads = num_q_heads;
  pf.block_tables = block_tables;
  pf.max_blocks_per_seq = max_blocks_per_seq;
  pf.context_lens = prefix_lens;
  pf.scale = scale;
  pf.d_status = d_status;
  pf.prefix_mode = 1;
  pf.pre_ml = pre_ml;
  pf.pre_acc = pre_acc;
  pf.beside_previous = 1;
  pf.sm_budget = std::max(1, device_sm_count() - a.grid_override);
  // the suffix decode first (it takes its SMs), the prefix pass beside it,
  // then the merge, which folds the prefix partials in, after both
  a.launch_part = 1;
  rc = to_status(launch_decode(a, st));
  if (rc != PA_OK) return rc;
  rc = to_status(launch_prefix_partials(pf, st));
  if (rc != PA_OK) return rc;
  a.launch_part = 2;
  return to_status(launch_decode(a, st));
}
}  // namespace

int pa_decode_cascade_with_ctas(const pa_kv_pool* pool, void* out, const void* q, int num_seqs,
                                int num_q_heads, const int32_t* block_tables,
                                int max_blocks_per_seq, const int32_t* context_lens,
                                const int32_t* cu_groups, const int32_t* prefix_lens,
                                int num_groups, float scale, int num_ctas, void* workspace,
                                size_t workspace_bytes, int* d_status, void* stream) {
  pa::TraceRange trace("pa_decode_cascade");
  return cascade_impl(pool, out, q, num_seqs, num_q_heads, block_tables, max_blocks_per_seq,
                      context_lens, cu_groups, prefix_lens, num_groups, nullptr, nullptr, 0, false,
                      scale, num_ctas, workspace, workspace_bytes, d_status, stream);
}

int pa_decode_cascade_nested(const pa_kv_pool* pool, void* out, const void* q, int num_seqs,
                             int num_q_heads, const int32_t* block_tables, int max_blocks_per_seq,
                             const int32_t* context_lens, const int32_t* cu_groups,
                             const int32_t* prefix_lens, int num_groups,
                             const int32_t* cu_siblings, const int32_t* sibling_lens,
                             int num_sibling_groups, float scale, int num_ctas, void* workspace,
                             size_t workspace_bytes, int* d_status, void* stream) {
  pa::TraceRange trace("pa_decode_cascade_nested");
  return cascade_impl(pool, out, q, num_seqs, num_q_heads, block_tables, max_blocks_per_seq,
                      context_lens, cu_groups, prefix_lens, num_groups, cu_siblings, sibling_lens,
                      num_sibling_groups, true, scale, num_ctas, workspace, workspace_bytes,
                      d_status, stream);
}

int pa_decode_cascade(const pa_kv_pool* pool, void* out, const void* q, int num_seqs,
                      int num_q_heads, const int32_t* block_tables, int max_blocks_per_seq,
                      const int32_t* context_lens, const int32_t* cu_groups,
                      const int32_t* prefix_lens, int num_groups, float scale, void* workspace,
                      size_t workspace_bytes, int* d_status, void* stream) {
  return pa_decode_cascade_with_ctas(pool, out, q, num_seqs, num_q_heads, block_tables,
                                     max_blocks_per_seq, context_lens, cu_groups, prefix_lens,
                                     num_groups, scale, 0, workspace, workspace_bytes, d_status,
                                     stream);
}

size_t pa_mixed_workspace_size(int num_seqs, int num_tokens, int num_q_heads, int head_dim,
                               int max_blocks_per_seq) {
  if (num_seqs < 0 || num_tokens < 0 || num_q_heads <= 0 || head_dim <= 0 ||
      max_blocks_per_seq <= 0)
    return 0;
  return decode_workspace_bytes(num_seqs, num_q_heads, head_dim);
}

int pa_mixed_step_with_units(const pa_kv_pool* pool, void* out, const void* q,
                             const int32_t* cu_q_lens, int num_seqs, int num_tokens,
                             int num_q_heads, const int32_t* context_lens,
                             const int32_t* block_tables, int max_blocks_per_seq, float scale,
                             int token_budget, const void* k_new, const void* v_new,
                             const int64_t* slot_mapping, int prefill_q_tiles, void* workspace,
                             size_t workspace_bytes, int* d_status, void* stream) {
  pa::TraceRange trace("pa_mixed_step");
  int rc = check_pool(pool);
  if (rc != PA_OK) return rc;
  if (num_seqs < 0 || num_tokens < 0 || max_blocks_per_seq <= 0) return PA_EINVAL;
  if (prefill_q_tiles < 0 || prefill_q_tiles > 2) return PA_EINVAL;
  rc = check_heads(pool, num_q_heads);
  if (rc != PA_OK) return rc;
  if (num_tokens > token_budget) return PA_EBUDGET;
  if (!decode_supported(pool->dtype, pool->head_dim, num_q_heads / pool->num_kv_heads,
                        pool->num_kv_heads) ||
      !prefill_supported(pool->dtype, pool->head_dim, num_q_heads / pool->num_kv_heads))
    return PA_EUNSUPPORTED;
  const bool write = k_new != nullptr || v_new != nullptr || slot_mapping != nullptr;
  if (write) {
    rc = validate_kv_write(pool, k_new, v_new, slot_mapping, num_tokens);
    if (rc != PA_OK) return rc;
  }
  if (num_seqs == 0 || num_tokens == 0) return PA_OK;
  if (out == nullptr || q == nullptr || cu_q_lens == nullptr || block_tables == nullptr ||
      context_lens == nullptr)
    return PA_EINVAL;
  if (!aligned16(out) || !aligned16(q)) return PA_EINVAL;
  const size_t need = pa_mixed_workspace_size(num_seqs, num_tokens, num_q_heads, pool->head_dim,
                                              max_blocks_per_seq);
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return PA_EWORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (write) {
    KvWriteArgs w;
    w.pool = view(pool);
    w.k_new = k_new;
    w.v_new = v_new;
    w.slot_mapping = slot_mapping;
    w.num_tokens = num_tokens;
    w.d_status = d_status;
    rc = to_status(launch_kv_write(w, st));
    if (rc != PA_OK) return rc;
  }
  PrefillArgs pf = {};
  pf.pool = view(pool);
  pf.out = out;
  pf.q = q;
  pf.cu_q_lens = cu_q_lens;
  pf.num_seqs = num_seqs;
  pf.num_tokens = num_tokens;
  pf.num_q_heads = num_q_heads;
  pf.block_tables = block_tables;
  pf.max_blocks_per_seq = max_blocks_per_seq;
  pf.context_lens = context_lens;
  pf.scale = scale;
  pf.d_status = d_status;
  pf.q_tiles = prefill_q_tiles;
  DecodeArgs a = {};
  a.pool = view(pool);
  a.out = out;
  a.q = q;
  a.cu_q_lens = cu_q_lens;
  a.num_seqs = num_seqs;
  a.num_rows = num_tokens;
  a.num_q_heads = num_q_heads;
  a.block_tables = block_tables;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.context_lens = context_lens;
  a.scale = scale;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.d_status = d_status;
  a.grid_override = 0;
  // prefill rows are at least num_tokens - num_seqs (every sequence that is
  // not a decode row contributes two or more)
  const int prefill_min = num_tokens - num_seqs;
  if (prefill_min >= kMixedPrefillTokens && num_seqs * kMixedTokensPerSeq <= prefill_min &&
      prefill_on_tensor_cores(pf)) {
    // decode on kMixedDecodeSms CTAs, the prefill beside it, then the merge
    a.grid_override = std::min(kMixedDecodeSms, device_sm_count());
    a.launch_part = 1;
    rc = to_status(launch_decode(a, st));
    if (rc != PA_OK) return rc;
    pf.beside_previous = 1;
    pf.sm_budget = std::max(1, device_sm_count() - a.grid_override);
    rc = to_status(launch_prefill(pf, st));
    if (rc != PA_OK) return rc;
    a.launch_part = 2;
    return to_status(launch_decode(a, st));
  }
  rc = to_status(launch_prefill(pf, st));
  if (rc != PA_OK) return rc;
  return to_status(launch_decode(a, st));
}

int pa_mixed_step(const pa_kv_pool* pool, void* out, const void* q, const int32_t* cu_q_lens,
                  int num_seqs, int num_tokens, int num_q_heads, const int32_t* context_lens,
                  const int32_t* block_tables, int max_blocks_per_seq, float scale,
                  int token_budget, const void* k_new, const void* v_new,
                  const int64_t* slot_mapping, void* workspace, size_t workspace_bytes,
                  int* d_status, void* stream) {
  return pa_mixed_step_with_units(pool, out, q, cu_q_lens, num_seqs, num_tokens, num_q_heads,
                                  context_lens, block_tables, max_blocks_per_seq, scale,
                                  token_budget, k_new, v_new, slot_mapping, 0, workspace,
                                  workspace_bytes, d_status, stream);
}

}  // extern "C"
