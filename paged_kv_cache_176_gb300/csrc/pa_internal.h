// pa_internal.h -- launch parameters shared between the C-ABI layer (api.cu)
// and the kernel translation units. Host code only; no device code here.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

constexpr int kMaxDecodeCtas = 1024;  // decode workspace holds this many CTA partial slots

inline size_t align_up_sz(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct PoolView {
  void* k;
  void* v;
  int64_t num_blocks;
  int num_kv_heads;
  int head_dim;
  int dtype;
};

// ---- KV write
struct KvWriteArgs {
  PoolView pool;
  const void* k_new;
  const void* v_new;
  const int64_t* slot_mapping;
  int num_tokens;
  int* d_status;
};
cudaError_t launch_kv_write(const KvWriteArgs& a, cudaStream_t stream);

// ---- decode (q_len == 1 rows)
struct DecodeArgs {
  PoolView pool;
  void* out;                 // rows indexed by seq (or by cu_q_lens[s] when given)
  const void* q;
  const int32_t* cu_q_lens;  // NULL: row of sequence s is s; else cu_q_lens[s], and
                             // only sequences with q_len == 1 are processed
  int num_seqs;
  int num_rows;              // rows of q/out (num_seqs, or num_tokens of a mixed step)
  int num_q_heads;
  const int32_t* block_tables;
  int max_blocks_per_seq;
  const int32_t* context_lens;
  float scale;
  void* workspace;
  size_t workspace_bytes;
  int* d_status;
  int grid_override;         // > 0: number of persistent CTAs (tuning / tests)
  // shared-prefix (cascade) decode, all NULL / 0 otherwise: sequences
  // cu_groups[g] .. cu_groups[g+1]-1 share their first prefix_lens[g] tokens
  // (whole blocks), whose attention partials (max, sum) and fp32 accumulators
  // are already in pre_ml [num_seqs, hq] (float2) and pre_acc [num_seqs, hq, D]
  const int32_t* cu_groups;
  const int32_t* prefix_lens;
  int num_groups;
  const void* pre_ml;
  const void* pre_acc;
  int defer_prefix;  // 1: the prefix partials are written concurrently; only the merge folds them
  int launch_part;   // 0: decode kernel and merge; 1: the decode kernel only; 2: the merge only
  // nested cascade, second level (NULL / 0 otherwise): sequences cu_sib[j] ..
  // cu_sib[j+1]-1 share their first shared_lens[j] tokens (whole blocks,
  // including any first-level prefix); the tensor-core path reads those
  // blocks once per entry of up to 16 / G members
  const int32_t* cu_sib;
  const int32_t* shared_lens;
  int num_sib;
  size_t ws_slots;   // partial slots the workspace holds (0: kMaxDecodeCtas + num_seqs)
  void* ws_rec;      // cascade calls: [num_seqs] uint32 per-sequence records for the merge
};
size_t decode_workspace_bytes(int num_seqs, int num_q_heads, int head_dim);
// The same for a workspace of `slots` partial slots.
size_t decode_workspace_bytes_slots(int num_seqs, int num_q_heads, int head_dim, size_t slots);
// per (dtype, head_dim) entry points, one translation unit each
cudaError_t decode_f32_d64(const DecodeArgs& a, int group, cudaStream_t stream);
cudaError_t decode_f32_d128(const DecodeArgs& a, int group, cudaStream_t stream);
cudaError_t decode_f32_d256(const DecodeArgs& a, int group, cudaStream_t stream);
cudaError_t decode_bf16_d64(const DecodeArgs& a, int group, cudaStream_t stream);
cudaError_t decode_bf16_d128(const DecodeArgs& a, int group, cudaStream_t stream);
cudaError_t decode_bf16_d256(const DecodeArgs& a, int group, cudaStream_t stream);
bool decode_supported(int dtype, int head_dim, int group, int num_kv_heads);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

// ---- prefill chunks (q_len > 1 rows of a mixed step)
struct PrefillArgs {
  PoolView pool;
  void* out;
  const void* q;
  const int32_t* cu_q_lens;
  int num_seqs;
  int num_tokens;
  int num_q_heads;
  const int32_t* block_tables;
  int max_blocks_per_seq;
  const int32_t* context_lens;
  float scale;
  int* d_status;
  // prefix mode (cascade decode): "sequence" i is group i of decode rows
  // cu_q_lens[i] .. cu_q_lens[i+1]-1, context_lens[i] is the group's shared
  // prefix length, its table is the row of its first member, every row sees
  // every prefix key, and the result goes to pre_ml / pre_acc (see DecodeArgs)
  int prefix_mode;
  void* pre_ml;
  void* pre_acc;
  // 1: launched as a programmatic dependent of the kernel before it on the
  // stream (a decode kernel that signals early), so that it runs beside that
  // kernel on the SMs it leaves free; the prefill reads nothing that kernel
  // writes and never waits for it
  int beside_previous;
  // SMs the prefill can expect to run on (0: all of them); with fewer, it
  // favours more, smaller units
  int sm_budget;
  // Q tiles of 128 rows per tensor-core unit (1 or 2); 0: chosen from the sizes
  int q_tiles;
};
bool prefill_supported(int dtype, int head_dim, int group);
// the tensor-core kernel in prefix mode (bf16, head_dim 128)
bool prefix_supported(int dtype, int head_dim, int group, int num_groups);
cudaError_t launch_prefix_partials(const PrefillArgs& a, cudaStream_t stream);
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream);
// true when launch_prefill takes the tensor-core kernel for these arguments
bool prefill_on_tensor_cores(const PrefillArgs& a);
cudaError_t launch_prefill_simt(const PrefillArgs& a, cudaStream_t stream);

int device_sm_count();

// Host validation of pa_decode's arguments other than the workspace (api.cu):
// PA_OK, or the pa_status pa_decode would return.
int check_decode_args(const pa_kv_pool* pool, const void* out, const void* q, int num_seqs,
                      int num_q_heads, const int32_t* block_tables, int max_blocks_per_seq,
                      const int32_t* context_lens);

}  // namespace pa
