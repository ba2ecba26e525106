/*
 * oracle.h -- plain, slow, fp64 CPU oracle for attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the library path may call, link or
 * load this code; only the tests, the package's smoke check and the benchmark's
 * CPU-baseline leg do. It shares no code, header, table or helper with the
 * CUDA path.
 *
 * What it computes (no blocking, no online softmax, no reordering):
 *
 *  - oracle_reshape_and_cache: the KV write. Token t goes to physical block
 *    slot/b at offset slot%b of the pool (the per-sequence page table maps
 *    logical token positions to physical blocks: "vLLM serving internals",
 *    section "PagedAttention as a virtual memory system", and the page-table
 *    example of "Inference engine core techniques", section 1.2). Slot -1 is
 *    skipped. The copy is byte-exact.
 *
 *  - oracle_copy_blocks: the copy-on-write copy. Several sequences may point
 *    their tables at one physical block (the replies of one request share the
 *    prompt's blocks; beams share their prefix pages); before a sequence
 *    writes into a shared block, that block is copied and the sequence's
 *    table points at the copy ("C13 L2 serving", parallel-sampling paragraph;
 *    "Inference engine core techniques", section 1.5). Pair i copies the
 *    first ntok[i] token slots (all slots when ntok is NULL) of block src[i]
 *    onto block dst[i] of both pools, byte for byte, pairs in order.
 *
 *  - oracle_paged_attention: for every query row, gather the sequence's K/V
 *    through its block table (K_r = gather(K_pool, table_r), the gather figure
 *    of "C13 L2 serving: continuous batching and PagedAttention"), then plain
 *    softmax attention in fp64 over the keys the row may see. A row at absolute
 *    position P sees keys 0..P (causal over absolute positions, the chunked
 *    prefill example of the "Chunked Prefill" glossary page); a decode row has
 *    P = ctx - 1 and sees the whole context ("Chunked Prefill" page, section on
 *    prefill and decode: decode reads the whole cache every step).
 *
 * Parity status: every function here is pinned by the CPU tests (brute force,
 * library SDPA on the gathered cache, the chunked == one-pass experiment,
 * permutation and copy-on-write invariance, closed forms, the worked page
 * table, planted-mistake checks). No function is "parity unpinned".
 */
#ifndef PAGED_ATTN_ORACLE_H
#define PAGED_ATTN_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element types of the pool and of q */
#define ORACLE_F32 0
#define ORACLE_BF16 1

/* error codes (0 = ok) */
#define ORACLE_OK 0
#define ORACLE_EARG 1     /* bad argument */
#define ORACLE_ERANGE 2   /* slot / block id / length out of range */

/*
 * k_pool, v_pool: [num_blocks, block_size, token_bytes] raw bytes.
 * k_new, v_new:   [num_tokens, token_bytes] raw bytes.
 * slot_mapping:   [num_tokens]; -1 skips the token.
 */
int oracle_reshape_and_cache(void* k_pool, void* v_pool, int64_t num_blocks,
                             int block_size, int64_t token_bytes,
                             const void* k_new, const void* v_new,
                             const int64_t* slot_mapping, int num_tokens);

/*
 * k_pool, v_pool: [num_blocks, block_size, token_bytes] raw bytes.
 * src, dst:       [n] physical block ids.
 * ntok:           [n] slots to copy per pair (0..block_size), or NULL for
 *                 whole blocks.
 * A pair with an id outside [0, num_blocks) or ntok outside [0, block_size]
 * is skipped; the others are still applied, and the call then returns
 * ORACLE_ERANGE.
 */
int oracle_copy_blocks(void* k_pool, void* v_pool, int64_t num_blocks,
                       int block_size, int64_t token_bytes,
                       const int32_t* src, const int32_t* dst,
                       const int32_t* ntok, int n);

/*
 * out:          [num_tokens, num_q_heads, head_dim] fp64.
 * q:            [num_tokens, num_q_heads, head_dim] of `dtype`.
 * k_pool/v_pool:[num_blocks, block_size, num_kv_heads, head_dim] of `dtype`.
 * cu_q_lens:    [num_seqs + 1]; sequence s owns query rows cu[s]..cu[s+1]-1.
 * context_lens: [num_seqs]; tokens cached for s, including its query rows.
 * block_tables: [num_seqs, max_blocks_per_seq].
 * row_mask:     [num_tokens] or NULL; rows with mask 0 are left untouched.
 * num_threads:  worker threads over (row, head) pairs (<= 0: 1).
 */
int oracle_paged_attention(double* out, const void* q, const void* k_pool,
                           const void* v_pool, int dtype, int64_t num_blocks,
                           int block_size, int num_kv_heads, int head_dim,
                           int num_q_heads, int num_seqs,
                           const int32_t* cu_q_lens,
                           const int32_t* context_lens,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           double scale, const uint8_t* row_mask,
                           int num_threads);

#ifdef __cplusplus
}
#endif
#endif
