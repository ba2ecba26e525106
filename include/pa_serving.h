/*
 * pa_serving.h -- host-side block manager and iteration-level scheduler that
 * drive the paged-attention kernels of pa.h.
 *
 * Block manager ("vLLM serving internals", PagedAttention as a virtual memory
 * system): the KV pool is a set of fixed-size physical blocks; each sequence
 * owns a block table; a block is appended when a sequence outgrows its last
 * block and returned to the pool when the sequence is released, so at most
 * block_size - 1 slots of a sequence are ever unused and there is no external
 * fragmentation ("C13 L2 serving", the waste bound of paging). Blocks are
 * reference counted: a forked sequence (parallel sampling, beam search)
 * shares every block of its parent, and the first write into a shared,
 * partially filled block copies it first (copy-on-write: "C13 L2 serving",
 * parallel sampling; "Inference engine core techniques", section 1.5).
 *
 * Scheduler (the scheduler loop of "vLLM serving internals"; "Inference engine
 * core techniques", section 2.3; the token budget of the "Chunked Prefill"
 * page): every step removes finished sequences and releases their blocks,
 * admits waiting requests while their blocks fit, schedules one token for
 * every running decode first and then fills the rest of the token budget with
 * prefill chunks of at most chunk_size tokens. Admission reserves the blocks
 * a request can reach (prompt + max_new_tokens), so a running sequence never
 * runs out of blocks (no preemption).
 *
 * All functions are host-only and allocate host memory only. An object is
 * not thread safe; distinct objects are independent. Return values are
 * pa_status codes (pa.h) unless stated otherwise; PA_ENOSPACE (-6) means the
 * pool has too few free blocks and nothing was changed.
 */
#ifndef PA_SERVING_H
#define PA_SERVING_H

#include <stddef.h>
#include <stdint.h>

#include "pa.h"

#ifdef __cplusplus
extern "C" {
#endif

#define PA_ENOSPACE (-6)

typedef struct pa_block_manager pa_block_manager;
typedef struct pa_scheduler pa_scheduler;

/* A pool of num_blocks blocks of block_size tokens; NULL on bad sizes. */
PA_API pa_block_manager* pa_bm_create(int64_t num_blocks, int block_size);
PA_API void pa_bm_destroy(pa_block_manager* bm);
PA_API int64_t pa_bm_num_free(const pa_block_manager* bm);

/* Register an empty sequence (PA_EINVAL if the id exists). */
PA_API int pa_bm_add(pa_block_manager* bm, int64_t seq);

/* child shares every block of parent (reference counts + 1). */
PA_API int pa_bm_fork(pa_block_manager* bm, int64_t parent, int64_t child);

/*
 * Reserve slots for n new tokens of seq. slots_out[i] receives the pool slot
 * (block * block_size + offset) of the i-th new token. If the last block is
 * shared and partially filled it is first replaced by a fresh copy: the
 * (source, destination) block pair is written to cow_src/cow_dst (capacity 1
 * is enough), the number of filled slots to copy to cow_ntok (nullable), and
 * *n_cow is set to the number of pairs. The caller copies the filled slots on
 * the device (pa_reshape_and_cache_cow, fused with the token writes, or
 * pa_copy_blocks) before the attention reads the block.
 */
PA_API int pa_bm_append(pa_block_manager* bm, int64_t seq, int n, int64_t* slots_out,
                        int32_t* cow_src, int32_t* cow_dst, int32_t* cow_ntok, int* n_cow);

/*
 * One beam-search step ("Inference engine core techniques", section 1.5: the
 * beams share their prefix pages and copy only where they diverge). New beam
 * i continues old beam old_ids[parents[i]]: it shares every block of that
 * beam (reference counts + 1); then every old beam is released, so the
 * blocks of beams that left no child return to the pool. A new id may reuse
 * an old beam's id. The next pa_bm_append of each new beam copies a shared
 * partial last block (copy-on-write); the last holder writes in place.
 * PA_EINVAL (nothing changed) on unknown or repeated old ids, a parent index
 * outside [0, n_old), repeated new ids, or a new id held by a live sequence
 * that is not an old beam.
 */
PA_API int pa_bm_beam_step(pa_block_manager* bm, int n_old, const int64_t* old_ids, int n_new,
                           const int32_t* parents, const int64_t* new_ids);

/*
 * Prefix cache ("Inference engine core techniques", section 3.2: split the
 * prompt into pages, hash each page, look the hash up, share the physical
 * pages that hit by reference count, prefill only the rest). Only full pages
 * are cached. A page's key is a chain hash: page j of a token sequence hashes
 * (key of page j-1, its 16 token ids), with key 0 before page 0, so a key
 * names the whole prefix up to and including the page. The hash is 64-bit
 * FNV-1a over the 8 little-endian bytes of the previous key and then each
 * token id as 4 little-endian bytes (pa_page_hash). A lookup also compares
 * the page's tokens and its parent block, so a hash collision cannot share a
 * wrong page. A cached block that nobody holds any more stays cached (and
 * counts as free) until an allocation finds no never-used or uncached free
 * block and evicts the least recently released one.
 */
PA_API uint64_t pa_page_hash(uint64_t parent_key, const int32_t* tokens, int n);

/* Turn the prefix cache on or off (off drops every entry). Default: off. */
PA_API int pa_bm_set_prefix_cache(pa_block_manager* bm, int enable);

/* Pages currently in the cache (-1 on a NULL manager). */
PA_API int64_t pa_bm_num_cached(const pa_block_manager* bm);

/*
 * Register seq, whose first n tokens are tokens[0..n), sharing the longest
 * run of its leading full pages found in the cache, at most (n-1)/16 pages so
 * that at least one token is left to compute. *hit_tokens (nullable) receives
 * the tokens covered (a multiple of 16); the sequence starts with that many
 * tokens. With the cache off this is pa_bm_add.
 */
PA_API int pa_bm_add_cached(pa_block_manager* bm, int64_t seq, const int32_t* tokens, int64_t n,
                            int64_t* hit_tokens);

/*
 * Enter seq's full pages among its first n tokens (tokens[0..n), all already
 * written to the pool) into the cache, after the ones entered before. A page
 * whose key is already cached (another block with the same prefix) is not
 * entered twice. n <= pa_bm_num_tokens(seq).
 */
PA_API int pa_bm_cache_pages(pa_block_manager* bm, int64_t seq, const int32_t* tokens, int64_t n);

/* Release seq: blocks whose count reaches zero return to the pool. */
PA_API int pa_bm_free(pa_block_manager* bm, int64_t seq);

/* Tokens held by seq (-1 if unknown). */
PA_API int64_t pa_bm_num_tokens(const pa_block_manager* bm, int64_t seq);

/* Writes seq's block table (at most max_blocks entries); returns its length
 * or a negative status. */
PA_API int pa_bm_block_table(const pa_block_manager* bm, int64_t seq, int32_t* out, int max_blocks);

/* Reference count of a physical block (-1 if out of range). */
PA_API int pa_bm_refcount(const pa_block_manager* bm, int32_t block);

/* Tokens that the n sequences seqs[0..n-1] (a request's beams or sampled
 * replies) share as a sibling group of pa_decode_cascade_nested: the leading
 * blocks that are the same physical blocks in every one's table, whole pages
 * within every one's context, times the block size. Returns that count (0
 * when they share no page), or PA_EINVAL for n < 1, a null array or an
 * unknown sequence. */
PA_API int64_t pa_bm_shared_prefix(const pa_block_manager* bm, const int64_t* seqs, int n);

/* A scheduler over bm: token_budget tokens per step, prefill chunks of at
 * most chunk_size tokens, at most max_running sequences. */
PA_API pa_scheduler* pa_sched_create(pa_block_manager* bm, int token_budget, int chunk_size,
                                     int max_running);
PA_API void pa_sched_destroy(pa_scheduler* s);

/* Queue a request (FIFO): prompt_len >= 1 prompt tokens, then max_new_tokens
 * generated tokens (>= 1). PA_EINVAL on a duplicate id or bad lengths. */
PA_API int pa_sched_submit(pa_scheduler* s, int64_t req_id, int prompt_len, int max_new_tokens);

/* The same with the prompt's token ids (copied). Such a request goes
 * through the prefix cache when its first prefill chunk is scheduled (not at
 * admission, so pages written by requests ahead of it in the meantime count):
 * its cached leading pages are shared and only the rest is prefilled. Its
 * step tokens appear in the plan's token_ids, its completed pages are entered
 * into the cache at each commit, and every token it generates must be
 * supplied to pa_sched_commit_tokens. */
PA_API int pa_sched_submit_tokens(pa_scheduler* s, int64_t req_id, const int32_t* prompt_tokens,
                                  int prompt_len, int max_new_tokens);

/* One step's batch, in caller-owned host buffers of the stated capacities.
 * Sequences are ordered decode first (q_len 1), then prefill chunks. The
 * block tables are packed: row j starts at j * table_stride, where
 * table_stride (<= max_blocks_per_seq) is the largest block count of any
 * sequence in the step, and is padded with -1 up to table_stride. */
typedef struct {
  int max_seqs, max_tokens, max_blocks_per_seq, max_cow; /* capacities (in) */
  int num_seqs, num_tokens, num_decode, num_cow;         /* counts (out) */
  int table_stride;                                      /* (out) */
  int64_t* seq_ids;       /* [max_seqs] */
  int32_t* cu_q_lens;     /* [max_seqs + 1] */
  int32_t* context_lens;  /* [max_seqs], including this step's tokens */
  int32_t* block_tables;  /* [num_seqs * table_stride] used of max_seqs * max_blocks_per_seq */
  int64_t* slot_mapping;  /* [max_tokens] */
  int32_t* cow_src;       /* [max_cow] blocks to copy before the KV write */
  int32_t* cow_dst;       /* [max_cow] */
  int32_t* cow_ntok;      /* [max_cow] filled slots of cow_src to copy (nullable) */
  int32_t* token_ids;     /* [max_tokens] ids of the step's tokens, -1 for requests
                             submitted without tokens (nullable) */
} pa_step_plan;

/* Build the next step (removing finished sequences, admitting requests,
 * reserving slots). Returns PA_OK with num_seqs == 0 when nothing is left
 * to run, PA_EINVAL if a capacity is too small (finished sequences are still
 * released and waiting ones admitted, but no slot is reserved). */
PA_API int pa_sched_step(pa_scheduler* s, pa_step_plan* plan);

/* Mark the last planned step as executed: prefill progress advances; a
 * decode step, and the step that finishes a prompt, yield one token. */
PA_API int pa_sched_commit(pa_scheduler* s);

/* pa_sched_commit for steps with token-mode requests: next_tokens[j] is the
 * token generated by plan row j (read only for rows that yield one). PA_EINVAL
 * and nothing changed when next_tokens is NULL and the step holds a token-mode
 * request. */
PA_API int pa_sched_commit_tokens(pa_scheduler* s, const int32_t* next_tokens);

/* Prompt tokens admitted from the prefix cache so far (not prefilled). */
PA_API int64_t pa_sched_cached_tokens(const pa_scheduler* s);

/* Counters: waiting, running, finished requests and the tokens processed. */
PA_API int pa_sched_stats(const pa_scheduler* s, int64_t* waiting, int64_t* running,
                          int64_t* finished, int64_t* prefill_tokens, int64_t* decode_tokens);

/*
 * Device copy of whole blocks of the K and V pools: block dst[i] <- src[i]
 * for i < n (src/dst are device int32 arrays). Used for copy-on-write.
 */
PA_API int pa_copy_blocks(const pa_kv_pool* pool, const int32_t* src, const int32_t* dst, int n,
                          int* d_status, void* stream);

/*
 * The KV write of a step (pa_reshape_and_cache) and its copy-on-write copies
 * in one launch: for i < n_cow the first cow_ntok[i] token slots of block
 * cow_src[i] are copied onto block cow_dst[i] (only the filled part of the
 * shared block, not all 16 slots), and token t is written to slot
 * slot_mapping[t] (-1 skips). The new tokens that land in a copied block must
 * sit at offsets >= its cow_ntok, which pa_bm_append guarantees: the copies
 * and the writes then touch disjoint slots and need no ordering. A pair with
 * a block outside the pool or cow_ntok outside [0, 16] sets
 * PA_STATUS_BAD_BLOCK and is skipped; a slot outside the pool sets
 * PA_STATUS_BAD_SLOT. cow_* are device int32 arrays.
 */
PA_API int pa_reshape_and_cache_cow(const pa_kv_pool* pool, const void* k_new, const void* v_new,
                                    const int64_t* slot_mapping, int num_tokens,
                                    const int32_t* cow_src, const int32_t* cow_dst,
                                    const int32_t* cow_ntok, int n_cow, int* d_status,
                                    void* stream);

#ifdef __cplusplus
}
#endif
#endif /* PA_SERVING_H */
