/*
 * oracle.c -- plain fp64 CPU oracle for attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY: see oracle.h for what it computes, which passages
 * it follows and who may call it. Written for a reader checking it against the
 * pages by eye: one query row and one head at a time, two passes over the keys
 * (scores, then weights and output), fp64 throughout.
 */
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* The stored value of element `idx` of an array of `dtype`, widened to fp64.
 * bf16 is the top half of an IEEE binary32, so widening is exact. */
static double load_value(const void* base, int dtype, int64_t idx) {
  if (dtype == ORACLE_F32) return (double)((const float*)base)[idx];
  uint16_t half = ((const uint16_t*)base)[idx];
  uint32_t bits = ((uint32_t)half) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

int oracle_reshape_and_cache(void* k_pool, void* v_pool, int64_t num_blocks,
                             int block_size, int64_t token_bytes,
                             const void* k_new, const void* v_new,
                             const int64_t* slot_mapping, int num_tokens) {
  if (!k_pool || !v_pool || block_size <= 0 || token_bytes <= 0 ||
      num_tokens < 0 || (num_tokens > 0 && (!k_new || !v_new || !slot_mapping)))
    return ORACLE_EARG;
  for (int t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue; /* padding token: nothing to write */
    int64_t block = slot / block_size;  /* physical block */
    int64_t offset = slot % block_size; /* position inside the block */
    if (block >= num_blocks) return ORACLE_ERANGE;
    int64_t dst = (block * block_size + offset) * token_bytes;
    memcpy((char*)k_pool + dst, (const char*)k_new + (int64_t)t * token_bytes,
           (size_t)token_bytes);
    memcpy((char*)v_pool + dst, (const char*)v_new + (int64_t)t * token_bytes,
           (size_t)token_bytes);
  }
  return ORACLE_OK;
}

int oracle_copy_blocks(void* k_pool, void* v_pool, int64_t num_blocks,
                       int block_size, int64_t token_bytes,
                       const int32_t* src, const int32_t* dst,
                       const int32_t* ntok, int n) {
  if (!k_pool || !v_pool || block_size <= 0 || token_bytes <= 0 || n < 0 ||
      (n > 0 && (!src || !dst)))
    return ORACLE_EARG;
  int status = ORACLE_OK;
  const int64_t block_bytes = (int64_t)block_size * token_bytes;
  for (int i = 0; i < n; ++i) {
    int64_t from = src[i], to = dst[i];
    int slots = ntok ? ntok[i] : block_size; /* the filled part of the block */
    if (from < 0 || from >= num_blocks || to < 0 || to >= num_blocks ||
        slots < 0 || slots > block_size) {
      status = ORACLE_ERANGE; /* skipped */
      continue;
    }
    size_t bytes = (size_t)(slots * token_bytes);
    memcpy((char*)k_pool + to * block_bytes, (const char*)k_pool + from * block_bytes, bytes);
    memcpy((char*)v_pool + to * block_bytes, (const char*)v_pool + from * block_bytes, bytes);
  }
  return status;
}

typedef struct {
  double* out;
  const void* q;
  const void* k_pool;
  const void* v_pool;
  int dtype;
  int64_t num_blocks;
  int block_size, num_kv_heads, head_dim, num_q_heads;
  const int32_t* block_tables;
  int max_blocks_per_seq;
  double scale;
  const uint8_t* row_mask;
  /* per query row: owning sequence, absolute position */
  const int32_t* row_seq;
  const int64_t* row_pos;
  int64_t num_rows; /* tokens * heads */
  int64_t max_pos;  /* largest absolute position of any row */
  int64_t first, stride;
  int status;
} job_t;

/* Attention of one query row (token t, head h): plain softmax over keys
 * 0..P of the gathered cache. */
static int attend_row(const job_t* j, int64_t t, int h, double* scores) {
  const int d = j->head_dim;
  const int b = j->block_size;
  const int group = j->num_q_heads / j->num_kv_heads; /* query heads per KV head */
  const int g = h / group;                            /* this head's KV head */
  const int s = j->row_seq[t];
  const int64_t P = j->row_pos[t];
  const int64_t q_base = (t * j->num_q_heads + h) * (int64_t)d;
  double* o = j->out + q_base;

  /* pass 1: scores x_p = scale * <q, K_s[p]> for p = 0..P */
  for (int64_t p = 0; p <= P; ++p) {
    int64_t block = j->block_tables[(int64_t)s * j->max_blocks_per_seq + p / b];
    if (block < 0 || block >= j->num_blocks) return ORACLE_ERANGE;
    int64_t k_base = ((block * b + p % b) * j->num_kv_heads + g) * (int64_t)d;
    double dot = 0.0;
    for (int i = 0; i < d; ++i)
      dot += load_value(j->q, j->dtype, q_base + i) *
             load_value(j->k_pool, j->dtype, k_base + i);
    scores[p] = j->scale * dot;
  }
  /* pass 2: softmax weights w_p = exp(x_p - max x), output sum w_p V_s[p] / sum w_p */
  double m = scores[0];
  for (int64_t p = 1; p <= P; ++p)
    if (scores[p] > m) m = scores[p];
  for (int i = 0; i < d; ++i) o[i] = 0.0;
  double l = 0.0;
  for (int64_t p = 0; p <= P; ++p) {
    double w = exp(scores[p] - m);
    l += w;
    int64_t block = j->block_tables[(int64_t)s * j->max_blocks_per_seq + p / b];
    int64_t v_base = ((block * b + p % b) * j->num_kv_heads + g) * (int64_t)d;
    for (int i = 0; i < d; ++i) o[i] += w * load_value(j->v_pool, j->dtype, v_base + i);
  }
  for (int i = 0; i < d; ++i) o[i] /= l;
  return ORACLE_OK;
}

static void* run_job(void* arg) {
  job_t* j = (job_t*)arg;
  double* scores = (double*)malloc(sizeof(double) * (size_t)(j->max_pos + 1));
  if (!scores) {
    j->status = ORACLE_EARG;
    return NULL;
  }
  /* worker w takes (row, head) pairs w, w + n, w + 2n, ... so that long and
   * short rows are spread over the workers */
  for (int64_t r = j->first; r < j->num_rows && j->status == ORACLE_OK; r += j->stride) {
    int64_t t = r / j->num_q_heads;
    int h = (int)(r % j->num_q_heads);
    if (j->row_mask && !j->row_mask[t]) continue;
    j->status = attend_row(j, t, h, scores);
  }
  free(scores);
  return NULL;
}

int oracle_paged_attention(double* out, const void* q, const void* k_pool,
                           const void* v_pool, int dtype, int64_t num_blocks,
                           int block_size, int num_kv_heads, int head_dim,
                           int num_q_heads, int num_seqs,
                           const int32_t* cu_q_lens,
                           const int32_t* context_lens,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           double scale, const uint8_t* row_mask,
                           int num_threads) {
  if (!out || !q || !k_pool || !v_pool || !cu_q_lens || !context_lens ||
      !block_tables || (dtype != ORACLE_F32 && dtype != ORACLE_BF16) ||
      block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      num_q_heads <= 0 || num_q_heads % num_kv_heads != 0 || num_seqs < 0 ||
      max_blocks_per_seq <= 0)
    return ORACLE_EARG;
  int64_t num_tokens = cu_q_lens[num_seqs];
  int32_t* row_seq = (int32_t*)malloc(sizeof(int32_t) * (size_t)(num_tokens + 1));
  int64_t* row_pos = (int64_t*)malloc(sizeof(int64_t) * (size_t)(num_tokens + 1));
  if (!row_seq || !row_pos) {
    free(row_seq);
    free(row_pos);
    return ORACLE_EARG;
  }
  int status = ORACLE_OK;
  for (int s = 0; s < num_seqs && status == ORACLE_OK; ++s) {
    int64_t q_len = (int64_t)cu_q_lens[s + 1] - cu_q_lens[s];
    int64_t ctx = context_lens[s];
    if (q_len < 0 || q_len > ctx ||
        ctx > (int64_t)max_blocks_per_seq * block_size) {
      status = ORACLE_ERANGE;
      break;
    }
    for (int64_t i = 0; i < q_len; ++i) {
      /* query row i of the chunk sits at absolute position ctx - q_len + i */
      row_seq[cu_q_lens[s] + i] = s;
      row_pos[cu_q_lens[s] + i] = ctx - q_len + i;
    }
  }
  if (status != ORACLE_OK) {
    free(row_seq);
    free(row_pos);
    return status;
  }
  int64_t max_pos = 0;
  for (int64_t t = 0; t < num_tokens; ++t)
    if (row_pos[t] > max_pos) max_pos = row_pos[t];
  if (num_threads <= 0) num_threads = 1;
  int64_t num_rows = num_tokens * num_q_heads;
  if (num_threads > num_rows) num_threads = (int)(num_rows > 0 ? num_rows : 1);
  job_t* jobs = (job_t*)calloc((size_t)num_threads, sizeof(job_t));
  pthread_t* tids = (pthread_t*)calloc((size_t)num_threads, sizeof(pthread_t));
  for (int w = 0; w < num_threads; ++w) {
    job_t* j = &jobs[w];
    j->out = out;
    j->q = q;
    j->k_pool = k_pool;
    j->v_pool = v_pool;
    j->dtype = dtype;
    j->num_blocks = num_blocks;
    j->block_size = block_size;
    j->num_kv_heads = num_kv_heads;
    j->head_dim = head_dim;
    j->num_q_heads = num_q_heads;
    j->block_tables = block_tables;
    j->max_blocks_per_seq = max_blocks_per_seq;
    j->scale = scale;
    j->row_mask = row_mask;
    j->row_seq = row_seq;
    j->row_pos = row_pos;
    j->num_rows = num_rows;
    j->max_pos = max_pos;
    j->first = w;
    j->stride = num_threads;
    j->status = ORACLE_OK;
  }
  if (num_threads == 1) {
    run_job(&jobs[0]);
  } else {
    for (int w = 0; w < num_threads; ++w) pthread_create(&tids[w], NULL, run_job, &jobs[w]);
    for (int w = 0; w < num_threads; ++w) pthread_join(tids[w], NULL);
  }
  for (int w = 0; w < num_threads; ++w)
    if (jobs[w].status != ORACLE_OK) status = jobs[w].status;
  free(jobs);
  free(tids);
  free(row_seq);
  free(row_pos);
  return status;
}
