/*
 * pa.h -- C ABI of libpa: attention over a paged KV cache on one GB300 (sm_103a).
 *
 * The KV cache is a pool of fixed-size physical blocks; every sequence owns a
 * block table mapping its logical blocks to physical block IDs ("vLLM serving
 * internals", section "PagedAttention as a virtual memory system"; the page
 * table of "Inference engine core techniques", section 1.2). Attention gathers
 * each sequence's K/V through its table (K_r = gather(K_pool, table_r), the
 * gather figure of "C13 L2 serving: continuous batching and PagedAttention").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers marked "device" are CUDA device pointers owned by the caller; the
 *    library allocates no memory and keeps no state between calls that could
 *    change a result (it caches only per-device facts: the SM count, and the
 *    address of pa_decode_static_ws's array).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream). PA_OK means "validated and enqueued".
 *  - Host-side validation looks only at scalars and pointer values; on any
 *    failure the call returns a negative pa_status and enqueues nothing.
 *  - Data-dependent errors (a table entry outside the pool, a context longer
 *    than the table, q_len > context, a slot outside the pool) are found on
 *    the device: the kernel ORs a PA_STATUS_* bit into *d_status (when
 *    d_status is not NULL), skips the bad access and writes zeros for the
 *    affected output rows. Nothing traps.
 *  - Every wait of a kernel on an asynchronous copy is bounded (2 s); if one
 *    gives up, the kernel ORs PA_STATUS_TIMEOUT into *d_status, stops, and
 *    the call's outputs are undefined.
 *  - Layouts are row-major and contiguous:
 *      K/V pool     [num_blocks, block_size, num_kv_heads, head_dim]
 *      q, out       [num_tokens, num_q_heads, head_dim]
 *      k_new, v_new [num_tokens, num_kv_heads, head_dim]
 *      block_tables int32 [num_seqs, max_blocks_per_seq]
 *    Query head h reads KV head h / (num_q_heads / num_kv_heads).
 *  - Supported: block_size 16; head_dim 64, 128 or 256; num_q_heads a multiple
 *    of num_kv_heads with a ratio of 1, 2, 4 or 8; num_kv_heads <= 8 for
 *    decode; dtype PA_F32 or PA_BF16. Accumulation is fp32; outputs are
 *    written in the input dtype (bf16 with round-to-nearest-even).
 *  - Every device pointer must be 16-byte aligned.
 *  - Calls are re-entrant; concurrent calls must not share a workspace.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PA_OK = 0,
  PA_EINVAL = -1,        /* null/misaligned pointer, negative or inconsistent size */
  PA_EUNSUPPORTED = -2,  /* block size, head_dim, head ratio or dtype not built */
  PA_EWORKSPACE = -3,    /* workspace NULL or smaller than the size query */
  PA_EBUDGET = -4,       /* num_tokens > token_budget */
  PA_ECUDA = -5          /* a kernel launch failed (the CUDA error is cleared) */
} pa_status;

typedef enum { PA_F32 = 0, PA_BF16 = 1 } pa_dtype;

/* Bits ORed into *d_status by the kernels. */
#define PA_STATUS_BAD_BLOCK 1u   /* block table entry outside [0, num_blocks) */
#define PA_STATUS_BAD_LENGTH 2u  /* context <= 0, context > max_blocks_per_seq * block_size,
                                    q_len > context, or inconsistent cu_q_lens */
#define PA_STATUS_BAD_SLOT 4u    /* slot_mapping entry >= num_blocks * block_size */
#define PA_STATUS_TIMEOUT 8u     /* a bounded wait on an asynchronous copy gave up */

/* The KV pool of one layer: borrowed device memory, never freed by libpa. */
typedef struct {
  void* k;              /* device, [num_blocks, block_size, num_kv_heads, head_dim] */
  void* v;              /* device, same shape as k */
  int64_t num_blocks;   /* N_blk */
  int32_t block_size;   /* b, tokens per block: 16 */
  int32_t num_kv_heads; /* Hkv */
  int32_t head_dim;     /* d */
  int32_t dtype;        /* pa_dtype */
} pa_kv_pool;

/* Human-readable text for a pa_status value (static storage). */
PA_API const char* pa_strerror(int status);

/* ABI version: (major << 16) | minor. */
PA_API int pa_version(void);

/*
 * KV write ("reshape and cache"): for every token t with slot_mapping[t] >= 0,
 * copy k_new[t] and v_new[t] into the pool at physical block slot / block_size,
 * offset slot % block_size. slot_mapping[t] == -1 marks a padding token and is
 * skipped. The copy is byte-exact for either dtype. The cache grows this way,
 * block by block ("Chunked Prefill" page, section on how chunked prefill works).
 *
 *  pool          K/V pool (written in place)
 *  k_new, v_new  device, [num_tokens, num_kv_heads, head_dim], pool dtype
 *  slot_mapping  device int64 [num_tokens]
 *  num_tokens    >= 0 (0 enqueues nothing)
 *  Any head_dim works here as long as a token row (num_kv_heads * head_dim
 *  elements) is a multiple of 16 bytes.
 *  d_status      device int32 or NULL; PA_STATUS_BAD_SLOT for slots past the pool
 */
PA_API int pa_reshape_and_cache(const pa_kv_pool* pool, const void* k_new, const void* v_new,
                         const int64_t* slot_mapping, int num_tokens, int* d_status,
                         void* stream);

/* Bytes of workspace pa_decode needs for these sizes (0 on invalid sizes). */
PA_API size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int head_dim,
                                int max_blocks_per_seq);

/*
 * Decode attention: one query token per sequence attends to the whole cached
 * context of that sequence (decode reads the entire cache each step: "Chunked
 * Prefill" page, section on prefill, decode and generation stalls). The block
 * loop follows the paged_attn pseudo-kernel of "Inference engine core
 * techniques", section 1.4: per page, look up the physical page, read its K/V,
 * accumulate with an online softmax. Long contexts are split over several
 * CTAs and the partial (max, sum, accumulator) triples are merged by a second
 * kernel; the split depends only on the context lengths, so results are
 * bit-identical under any relabelling of physical blocks.
 *
 *  out           device, [num_seqs, num_q_heads, head_dim], pool dtype
 *  q             device, [num_seqs, num_q_heads, head_dim], pool dtype
 *  block_tables  device int32 [num_seqs, max_blocks_per_seq]
 *  context_lens  device int32 [num_seqs]; tokens attended (>= 1)
 *  scale         softmax scale applied to q.k (e.g. 1/sqrt(head_dim))
 *  workspace     device, >= pa_decode_workspace_size(...) bytes, 16-byte aligned
 */
PA_API int pa_decode(const pa_kv_pool* pool, void* out, const void* q, int num_seqs,
              int num_q_heads, const int32_t* block_tables, int max_blocks_per_seq,
              const int32_t* context_lens, float scale, void* workspace,
              size_t workspace_bytes, int* d_status, void* stream);

/*
 * pa_decode without a workspace argument, for callers that cannot allocate
 * device memory around the call (for example a host framework that plans all
 * device buffers itself and does not let libraries call cudaMalloc, or a
 * latency-critical loop where an allocation, which can synchronize the device
 * or fail under memory pressure, is not allowed). The pages describe no such
 * entry point; it has no counterpart there.
 *
 * Same arguments, kernels and results as pa_decode, minus workspace and
 * workspace_bytes. The split-K scratch is a static device array of
 * PA_DECODE_STATIC_WS_BYTES inside libpa, held on every GPU that loads the
 * library until the process exits; the call allocates nothing.
 *  - Sizes whose pa_decode_workspace_size() exceeds PA_DECODE_STATIC_WS_BYTES
 *    are rejected with PA_EWORKSPACE before anything is enqueued.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and caches it; make the
 *    first call on a device before any stream capture.
 *  - Every call uses the same array, which keeps the previous call's
 *    contents; nothing in it needs to start at zero (a call whose status gets
 *    PA_STATUS_TIMEOUT has undefined outputs, as for every entry point).
 *    Calls that overlap on the GPU (other streams, other host threads) race
 *    on it: serialize them.
 *  - The cached address is that of the device's context at the first call;
 *    after cudaDeviceReset on a device, do not call this entry point on it
 *    again in the same process.
 *  - Argument errors return what pa_decode would return; the size limit is
 *    checked after them.
 */
#define PA_DECODE_STATIC_WS_BYTES (((size_t)32) << 20)
PA_API int pa_decode_static_ws(const pa_kv_pool* pool, void* out, const void* q, int num_seqs,
                               int num_q_heads, const int32_t* block_tables,
                               int max_blocks_per_seq, const int32_t* context_lens, float scale,
                               int* d_status, void* stream);

/*
 * Decode over sequences that share a prompt prefix, reading the shared blocks
 * once per group instead of once per sequence. Paging lets several sequences
 * point their block tables at the same physical blocks: the replies of one
 * request share its prompt's blocks ("C13 L2 serving", parallel sampling
 * paragraph), and requests with a common prefix share its full pages by
 * reference count ("Inference engine core techniques", section 3.2). The
 * result is the same attention as pa_decode (up to floating-point summation
 * order): softmax over all of a sequence's keys splits exactly into a part
 * over the shared prefix and a part over the rest, merged through their
 * (max, sum, accumulator) triples, the identity pa_decode's split-K uses.
 *
 * Groups: sequences cu_groups[g] .. cu_groups[g+1]-1 form group g; their
 * first prefix_lens[g] tokens (a multiple of 16, at most each member's
 * context) are held by the same physical blocks, i.e. the first
 * prefix_lens[g]/16 entries of every member's block-table row are equal. The
 * shared blocks are read through the group's first member's row; the caller
 * guarantees the equality (it is not checked). Sequences outside every group,
 * and groups with prefix_lens[g] == 0, are plain decode.
 *
 * Steps: (1) one tensor-core pass per group and KV head computes the
 * partials of every member's query rows against the shared prefix (a dense
 * contraction: members x heads rows by prefix keys); (2) the decode kernel
 * walks each sequence's remaining blocks; (3) a merge kernel folds the prefix
 * partials in. All three run on the caller's stream, (1) and (2) side by
 * side: (2) is launched first on all but 36 SMs, (1) right after it as a
 * programmatic dependent launch that takes the SMs (2) leaves free (neither
 * waits for the other), and (3) after both. With num_groups == 0 the call is
 * pa_decode.
 *
 *  cu_groups     device int32 [num_groups + 1], non-decreasing, within [0, num_seqs]
 *  prefix_lens   device int32 [num_groups], tokens; multiple of 16
 *  other arguments as pa_decode; workspace >= pa_decode_cascade_workspace_size()
 *
 * Supported: bf16 with head_dim 128 (the tensor-core prefix pass), the
 * query/KV head ratios and KV head counts of pa_decode; otherwise
 * PA_EUNSUPPORTED. A prefix length that is not a multiple of 16 or exceeds a
 * member's context sets PA_STATUS_BAD_LENGTH in *d_status and that member's
 * output row is zeros.
 */
PA_API size_t pa_decode_cascade_workspace_size(int num_seqs, int num_q_heads, int head_dim,
                                               int max_blocks_per_seq);
PA_API int pa_decode_cascade(const pa_kv_pool* pool, void* out, const void* q, int num_seqs,
                             int num_q_heads, const int32_t* block_tables, int max_blocks_per_seq,
                             const int32_t* context_lens, const int32_t* cu_groups,
                             const int32_t* prefix_lens, int num_groups, float scale,
                             void* workspace, size_t workspace_bytes, int* d_status, void* stream);

/*
 * Two-level cascade decode: pa_decode_cascade's groups (first level: a
 * prefix shared by many sequences, e.g. a system prompt, read once per group
 * by the tensor-core prefix pass) plus sibling groups (second level: a few
 * sequences that share a longer prefix, e.g. the replies of one request,
 * which share all of its prompt's full pages; "C13 L2 serving", parallel
 * sampling paragraph). A sibling group's shared blocks after the first-level
 * prefix are read once per entry of up to 16 / (num_q_heads / num_kv_heads)
 * members: the decode kernel puts the members' query rows together in one
 * 16-row tensor-core tile, so each such block is loaded and multiplied once
 * for all of them. Each member's own blocks are read for that member only (the
 * other rows of the tile are masked). The result is the same attention as
 * pa_decode, up to floating-point summation order.
 *
 * Sibling groups: sequences cu_siblings[j] .. cu_siblings[j+1]-1 form
 * sibling group j; their first sibling_lens[j] tokens (a multiple of 16, at
 * most each member's context, at least the member's first-level prefix) are
 * held by the same physical blocks, read through the first row of each entry
 * (entries are consecutive runs of members from cu_siblings[j]); the caller
 * guarantees the block equality (not checked). Members of one sibling group
 * must have the same first-level prefix length. cu_siblings is non-decreasing
 * within [0, num_seqs]. num_sibling_groups == 0 gives pa_decode_cascade (with
 * this call's workspace); num_groups == 0 leaves out the first level.
 *
 * The sibling entries run on the tensor-core decode path (bf16, head_dim 64 or
 * 128, 8 KV heads); with fewer KV heads the decode walks every sequence on
 * its own (same result, no second-level saving).
 *
 * Errors: a sibling length that is not whole blocks, is shorter than the
 * member's first-level prefix or longer than its context, or a member whose
 * entry's first member has lengths that cannot hold the shared blocks, sets
 * PA_STATUS_BAD_LENGTH in *d_status and zeroes that member's output row (a
 * bad first member of an entry makes every member of the entry bad).
 *
 *  cu_siblings    device int32 [num_sibling_groups + 1]
 *  sibling_lens   device int32 [num_sibling_groups], tokens
 *  num_ctas       persistent decode CTAs as in pa_decode_cascade_with_ctas
 *                 (0: the default); the workspace depends on it
 *  other arguments as pa_decode_cascade; workspace >=
 *  pa_decode_cascade_nested_workspace_size(num_seqs, num_q_heads,
 *  num_kv_heads, head_dim, max_blocks_per_seq, num_ctas)
 */
PA_API size_t pa_decode_cascade_nested_workspace_size(int num_seqs, int num_q_heads,
                                                      int num_kv_heads, int head_dim,
                                                      int max_blocks_per_seq, int num_ctas);
PA_API int pa_decode_cascade_nested(const pa_kv_pool* pool, void* out, const void* q, int num_seqs,
                                    int num_q_heads, const int32_t* block_tables,
                                    int max_blocks_per_seq, const int32_t* context_lens,
                                    const int32_t* cu_groups, const int32_t* prefix_lens,
                                    int num_groups, const int32_t* cu_siblings,
                                    const int32_t* sibling_lens, int num_sibling_groups,
                                    float scale, int num_ctas, void* workspace,
                                    size_t workspace_bytes, int* d_status, void* stream);

/*
 * pa_decode and pa_decode_cascade with an explicit number of persistent
 * decode CTAs instead of the default of one per SM of the current device
 * (num_ctas == 0 keeps the default; values above 1024 are clamped; negative
 * values return PA_EINVAL). The CTA count sets where the balanced split-K
 * cuts the batch's blocks, so it changes the floating-point summation order
 * and nothing else. For tuning and for tests that make sequences straddle
 * many CTAs; the count is an argument, never library state.
 */
PA_API int pa_decode_with_ctas(const pa_kv_pool* pool, void* out, const void* q, int num_seqs,
                               int num_q_heads, const int32_t* block_tables,
                               int max_blocks_per_seq, const int32_t* context_lens, float scale,
                               int num_ctas, void* workspace, size_t workspace_bytes,
                               int* d_status, void* stream);
PA_API int pa_decode_cascade_with_ctas(const pa_kv_pool* pool, void* out, const void* q,
                                       int num_seqs, int num_q_heads, const int32_t* block_tables,
                                       int max_blocks_per_seq, const int32_t* context_lens,
                                       const int32_t* cu_groups, const int32_t* prefix_lens,
                                       int num_groups, float scale, int num_ctas, void* workspace,
                                       size_t workspace_bytes, int* d_status, void* stream);

/* Bytes of workspace pa_mixed_step needs for these sizes (0 on invalid sizes). */
PA_API size_t pa_mixed_workspace_size(int num_seqs, int num_tokens, int num_q_heads, int head_dim,
                               int max_blocks_per_seq);

/*
 * Mixed step: one call for a batch of decode tokens and prefill chunks under a
 * token budget (the step of iteration-level scheduling with chunked prefill:
 * "Chunked Prefill" page, section on how it works; "vLLM serving internals",
 * scheduler loop, "one fused GPU call"). Sequence s owns query rows
 * cu_q_lens[s] .. cu_q_lens[s+1]-1; its q_len = cu_q_lens[s+1] - cu_q_lens[s]
 * rows are the LAST q_len positions of its context_lens[s] tokens, so row i
 * sits at absolute position context_lens[s] - q_len + i and attends keys
 * 0 .. that position (causal over absolute positions, as in the glossary
 * page's chunked-prefill example). q_len == 1 rows take the decode kernel;
 * q_len > 1 rows take the prefill kernel (tcgen05 tensor cores for bf16). The
 * result equals one-pass causal prefill for any chunk split. When the step
 * is dominated by prefill on the tensor-core path (with P = num_tokens -
 * num_seqs: P >= 1024 and num_seqs <= P / 12), the decode rows run on 48 SMs
 * and the prefill beside them on the other SMs (a programmatic dependent
 * launch on the same stream; neither kernel waits for the other); otherwise
 * the prefill runs first on all SMs, then the decode. The tensor-core prefill
 * serves two 128-row query tiles from each K/V tile when one-tile units would
 * not all fit on the SMs it gets at once, else one
 * (pa_mixed_step_with_units fixes the choice).
 *
 *  cu_q_lens     device int32 [num_seqs + 1], cu_q_lens[0] = 0, non-decreasing,
 *                cu_q_lens[num_seqs] = num_tokens
 *  context_lens  device int32 [num_seqs]; includes this step's tokens
 *  token_budget  num_tokens must not exceed it (PA_EBUDGET otherwise)
 *  k_new, v_new, slot_mapping
 *                NULL, or the step's new K/V ([num_tokens, Hkv, d]) and slots:
 *                when given, the KV write runs first, on the same stream
 *  workspace     device, >= pa_mixed_workspace_size(...) bytes
 */
PA_API int pa_mixed_step(const pa_kv_pool* pool, void* out, const void* q, const int32_t* cu_q_lens,
                  int num_seqs, int num_tokens, int num_q_heads, const int32_t* context_lens,
                  const int32_t* block_tables, int max_blocks_per_seq, float scale,
                  int token_budget, const void* k_new, const void* v_new,
                  const int64_t* slot_mapping, void* workspace, size_t workspace_bytes,
                  int* d_status, void* stream);

/*
 * pa_mixed_step with the size of the tensor-core prefill units fixed:
 * prefill_q_tiles = 1 or 2 query tiles of 128 rows per unit (0: the library
 * chooses from the sizes, as pa_mixed_step does; other values return
 * PA_EINVAL). Two-tile units share each K/V tile between both tiles and
 * overlap one tile's softmax with the other's products; one-tile units give
 * twice as many units for small steps. Both compute the same attention; a
 * row's last bits can differ between them where a tile's first row decides
 * whether the row's exponents take the masked form. For tuning and for tests
 * that run both unit shapes on the same inputs; an argument, never library
 * state.
 */
PA_API int pa_mixed_step_with_units(const pa_kv_pool* pool, void* out, const void* q,
                                    const int32_t* cu_q_lens, int num_seqs, int num_tokens,
                                    int num_q_heads, const int32_t* context_lens,
                                    const int32_t* block_tables, int max_blocks_per_seq,
                                    float scale, int token_budget, const void* k_new,
                                    const void* v_new, const int64_t* slot_mapping,
                                    int prefill_q_tiles, void* workspace, size_t workspace_bytes,
                                    int* d_status, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* PA_H */
