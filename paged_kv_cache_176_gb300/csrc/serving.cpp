// serving.cpp -- host-side block manager and iteration-level scheduler
// (include/pa_serving.h). Plain C++17, no CUDA calls.
#include <algorithm>
#include <array>
#include <deque>
#include <list>
#include <new>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "../../include/pa_serving.h"
#include "pa_trace.h"

// 64-bit FNV-1a (Fowler, Noll, Vo), fed byte by byte.
static inline uint64_t fnv1a_byte(uint64_t h, uint8_t b) { return (h ^ b) * 0x100000001b3ull; }

static uint64_t page_hash(uint64_t parent, const int32_t* tokens, int n) {
  uint64_t h = 0xcbf29ce484222325ull;
  for (int i = 0; i < 8; ++i) h = fnv1a_byte(h, static_cast<uint8_t>(parent >> (8 * i)));
  for (int t = 0; t < n; ++t) {
    const uint32_t v = static_cast<uint32_t>(tokens[t]);
    for (int i = 0; i < 4; ++i) h = fnv1a_byte(h, static_cast<uint8_t>(v >> (8 * i)));
  }
  return h;
}

struct pa_block_manager {
  struct Seq {
    std::vector<int32_t> blocks;
    int64_t tokens = 0;
    int64_t pages_cached = 0;  // leading full pages registered in (or taken from) the cache
    uint64_t last_hash = 0;    // chain hash of page pages_cached - 1
  };
  // a full page in the prefix cache: its chain hash, tokens and parent block
  struct Page {
    uint64_t hash = 0;
    int32_t parent = -1;
    std::vector<int32_t> tokens;
    bool cached = false;
  };
  int64_t num_blocks = 0;
  int block_size = 0;
  std::vector<int32_t> free_list;  // a stack: the most recently freed block is reused first
  std::vector<int32_t> refcount;
  std::unordered_map<int64_t, Seq> seqs;
  // prefix cache ("Inference engine core techniques", section 3.2)
  bool prefix_cache = false;
  std::vector<Page> pages;                       // per block
  std::unordered_map<uint64_t, int32_t> cached;  // chain hash -> block
  std::list<int32_t> lru;                        // cached blocks nobody holds, oldest first
  std::vector<std::list<int32_t>::iterator> lru_pos;

  int64_t blocks_for(int64_t tokens) const { return (tokens + block_size - 1) / block_size; }
  int64_t available() const { return static_cast<int64_t>(free_list.size() + lru.size()); }

  void uncache(int32_t b) {
    cached.erase(pages[b].hash);
    pages[b].cached = false;
    pages[b].tokens.clear();
  }
  // A free block: the free stack first, else the least recently released
  // cached block (evicted from the cache).
  int32_t take() {
    int32_t b;
    if (!free_list.empty()) {
      b = free_list.back();
      free_list.pop_back();
    } else {
      b = lru.front();
      lru.pop_front();
      uncache(b);
    }
    refcount[b] = 1;
    return b;
  }
  void release(int32_t b) {
    if (--refcount[b] > 0) return;
    if (prefix_cache && pages[b].cached) {
      lru_pos[b] = lru.insert(lru.end(), b);  // still a cache hit until evicted
    } else {
      free_list.push_back(b);
    }
  }
  // share a cached block (it leaves the LRU list when nobody held it)
  void hold(int32_t b) {
    if (refcount[b]++ == 0) lru.erase(lru_pos[b]);
  }
  // Blocks an append of n tokens to s needs (a copy of a shared partial last
  // block counts as one).
  int64_t append_cost(const Seq& s, int n) const {
    int64_t need = blocks_for(s.tokens + n) - blocks_for(s.tokens);
    if (n > 0 && s.tokens % block_size != 0 && refcount[s.blocks.back()] > 1) need += 1;
    return need;
  }
};

extern "C" {

pa_block_manager* pa_bm_create(int64_t num_blocks, int block_size) {
  if (num_blocks <= 0 || num_blocks > INT32_MAX || block_size <= 0) return nullptr;
  auto* bm = new (std::nothrow) pa_block_manager();
  if (bm == nullptr) return nullptr;
  bm->num_blocks = num_blocks;
  bm->block_size = block_size;
  bm->refcount.assign(static_cast<size_t>(num_blocks), 0);
  bm->pages.resize(static_cast<size_t>(num_blocks));
  bm->lru_pos.resize(static_cast<size_t>(num_blocks));
  bm->free_list.reserve(static_cast<size_t>(num_blocks));
  // block 0 on top of the stack: allocation order 0, 1, 2, ...
  for (int64_t b = num_blocks - 1; b >= 0; --b) bm->free_list.push_back(static_cast<int32_t>(b));
  return bm;
}

void pa_bm_destroy(pa_block_manager* bm) { delete bm; }

int64_t pa_bm_num_free(const pa_block_manager* bm) { return bm ? bm->available() : -1; }

uint64_t pa_page_hash(uint64_t parent, const int32_t* tokens, int n) {
  if (tokens == nullptr || n < 0) return 0;
  return page_hash(parent, tokens, n);
}

int pa_bm_set_prefix_cache(pa_block_manager* bm, int enable) {
  if (bm == nullptr) return PA_EINVAL;
  if (!enable) {
    // drop every cache entry; cached blocks nobody holds become free
    for (int32_t b : bm->lru) bm->free_list.push_back(b);
    bm->lru.clear();
    for (int64_t b = 0; b < bm->num_blocks; ++b)
      if (bm->pages[b].cached) bm->uncache(static_cast<int32_t>(b));
    for (auto& kv : bm->seqs) kv.second.pages_cached = 0;
  }
  bm->prefix_cache = enable != 0;
  return PA_OK;
}

int64_t pa_bm_num_cached(const pa_block_manager* bm) {
  return bm ? static_cast<int64_t>(bm->cached.size()) : -1;
}

// Share the cached leading pages of tokens[0..n) into the empty sequence sq.
static void share_cached_prefix(pa_block_manager* bm, pa_block_manager::Seq& sq,
                                const int32_t* tokens, int64_t n) {
  const int bs = bm->block_size;
  if (bm->prefix_cache) {
    // walk the prompt's full pages while the chain hits; keep >= 1 token to compute
    const int64_t max_pages = n > 0 ? (n - 1) / bs : 0;
    uint64_t h = 0;
    int32_t parent = -1;
    for (int64_t j = 0; j < max_pages; ++j) {
      const int32_t* pt = tokens + j * bs;
      const uint64_t hj = page_hash(h, pt, bs);
      auto it = bm->cached.find(hj);
      if (it == bm->cached.end()) break;
      const auto& pg = bm->pages[it->second];
      if (pg.parent != parent || !std::equal(pg.tokens.begin(), pg.tokens.end(), pt)) break;
      bm->hold(it->second);
      sq.blocks.push_back(it->second);
      parent = it->second;
      h = hj;
    }
    sq.tokens = static_cast<int64_t>(sq.blocks.size()) * bs;
    sq.pages_cached = static_cast<int64_t>(sq.blocks.size());
    sq.last_hash = h;
  }
}

int pa_bm_add_cached(pa_block_manager* bm, int64_t seq, const int32_t* tokens, int64_t n,
                     int64_t* hit_tokens) {
  if (bm == nullptr || bm->seqs.count(seq) || n < 0 || (n > 0 && tokens == nullptr)) return PA_EINVAL;
  pa_block_manager::Seq sq;
  share_cached_prefix(bm, sq, tokens, n);
  if (hit_tokens != nullptr) *hit_tokens = sq.tokens;
  bm->seqs.emplace(seq, std::move(sq));
  return PA_OK;
}

int pa_bm_cache_pages(pa_block_manager* bm, int64_t seq, const int32_t* tokens, int64_t n) {
  if (bm == nullptr || n < 0 || (n > 0 && tokens == nullptr)) return PA_EINVAL;
  auto it = bm->seqs.find(seq);
  if (it == bm->seqs.end() || n > it->second.tokens) return PA_EINVAL;
  if (!bm->prefix_cache) return PA_OK;
  auto& sq = it->second;
  const int bs = bm->block_size;
  for (int64_t j = sq.pages_cached; j < n / bs; ++j) {
    const int32_t* pt = tokens + j * bs;
    const uint64_t hj = page_hash(sq.last_hash, pt, bs);
    const int32_t b = sq.blocks[static_cast<size_t>(j)];
    auto& pg = bm->pages[b];
    if (!pg.cached && !bm->cached.count(hj)) {  // the first block with this content wins
      pg.hash = hj;
      pg.parent = j > 0 ? sq.blocks[static_cast<size_t>(j - 1)] : -1;
      pg.tokens.assign(pt, pt + bs);
      pg.cached = true;
      bm->cached.emplace(hj, b);
    }
    sq.last_hash = hj;
    sq.pages_cached = j + 1;
  }
  return PA_OK;
}

int pa_bm_add(pa_block_manager* bm, int64_t seq) {
  if (bm == nullptr || bm->seqs.count(seq)) return PA_EINVAL;
  bm->seqs.emplace(seq, pa_block_manager::Seq());
  return PA_OK;
}

int pa_bm_fork(pa_block_manager* bm, int64_t parent, int64_t child) {
  if (bm == nullptr || !bm->seqs.count(parent) || bm->seqs.count(child)) return PA_EINVAL;
  pa_block_manager::Seq copy = bm->seqs.at(parent);
  for (int32_t b : copy.blocks) ++bm->refcount[b];
  bm->seqs.emplace(child, std::move(copy));
  return PA_OK;
}

int pa_bm_append(pa_block_manager* bm, int64_t seq, int n, int64_t* slots_out, int32_t* cow_src,
                 int32_t* cow_dst, int32_t* cow_ntok, int* n_cow) {
  if (bm == nullptr || n < 0 || (n > 0 && slots_out == nullptr)) return PA_EINVAL;
  auto it = bm->seqs.find(seq);
  if (it == bm->seqs.end()) return PA_EINVAL;
  auto& s = it->second;
  if (n_cow != nullptr) *n_cow = 0;
  if (n == 0) return PA_OK;
  if (bm->append_cost(s, n) > bm->available()) return PA_ENOSPACE;
  const int b = bm->block_size;
  if (s.tokens % b != 0 && bm->refcount[s.blocks.back()] > 1) {
    // the last block is shared and partially filled: give this sequence its
    // own copy before writing into it
    if (cow_src == nullptr || cow_dst == nullptr || n_cow == nullptr) return PA_EINVAL;
    const int32_t old = s.blocks.back();
    const int32_t fresh = bm->take();
    bm->release(old);
    s.blocks.back() = fresh;
    cow_src[0] = old;
    cow_dst[0] = fresh;
    if (cow_ntok != nullptr) cow_ntok[0] = static_cast<int32_t>(s.tokens % b);
    *n_cow = 1;
  }
  for (int i = 0; i < n; ++i) {
    const int64_t pos = s.tokens + i;
    if (pos % b == 0) s.blocks.push_back(bm->take());  // the sequence outgrew its blocks
    slots_out[i] = static_cast<int64_t>(s.blocks[pos / b]) * b + pos % b;
  }
  s.tokens += n;
  return PA_OK;
}

int pa_bm_beam_step(pa_block_manager* bm, int n_old, const int64_t* old_ids, int n_new,
                    const int32_t* parents, const int64_t* new_ids) {
  if (bm == nullptr || n_old < 0 || n_new < 0) return PA_EINVAL;
  if ((n_old > 0 && old_ids == nullptr) || (n_new > 0 && (parents == nullptr || new_ids == nullptr)))
    return PA_EINVAL;
  // check everything first so that a rejected call changes nothing
  std::unordered_set<int64_t> olds, news;
  for (int i = 0; i < n_old; ++i)
    if (!bm->seqs.count(old_ids[i]) || !olds.insert(old_ids[i]).second) return PA_EINVAL;
  for (int i = 0; i < n_new; ++i) {
    if (parents[i] < 0 || parents[i] >= n_old) return PA_EINVAL;
    if (!news.insert(new_ids[i]).second) return PA_EINVAL;
    if (bm->seqs.count(new_ids[i]) && !olds.count(new_ids[i])) return PA_EINVAL;
  }
  // children share every block of their parent; then the old beams leave.
  // Children are built aside first, as a new id may reuse an old beam's id.
  std::vector<pa_block_manager::Seq> kids;
  kids.reserve(static_cast<size_t>(n_new));
  for (int i = 0; i < n_new; ++i) {
    kids.push_back(bm->seqs.at(old_ids[parents[i]]));
    for (int32_t b : kids.back().blocks) ++bm->refcount[b];
  }
  for (int i = 0; i < n_old; ++i) pa_bm_free(bm, old_ids[i]);
  for (int i = 0; i < n_new; ++i) bm->seqs.emplace(new_ids[i], std::move(kids[static_cast<size_t>(i)]));
  return PA_OK;
}

int pa_bm_free(pa_block_manager* bm, int64_t seq) {
  if (bm == nullptr) return PA_EINVAL;
  auto it = bm->seqs.find(seq);
  if (it == bm->seqs.end()) return PA_EINVAL;
  for (int32_t blk : it->second.blocks) bm->release(blk);
  bm->seqs.erase(it);
  return PA_OK;
}

int64_t pa_bm_num_tokens(const pa_block_manager* bm, int64_t seq) {
  if (bm == nullptr) return -1;
  auto it = bm->seqs.find(seq);
  return it == bm->seqs.end() ? -1 : it->second.tokens;
}

int pa_bm_block_table(const pa_block_manager* bm, int64_t seq, int32_t* out, int max_blocks) {
  if (bm == nullptr || out == nullptr || max_blocks < 0) return PA_EINVAL;
  auto it = bm->seqs.find(seq);
  if (it == bm->seqs.end()) return PA_EINVAL;
  const auto& blocks = it->second.blocks;
  if (static_cast<int64_t>(blocks.size()) > max_blocks) return PA_EINVAL;
  std::copy(blocks.begin(), blocks.end(), out);
  return static_cast<int>(blocks.size());
}

int pa_bm_refcount(const pa_block_manager* bm, int32_t block) {
  if (bm == nullptr || block < 0 || block >= bm->num_blocks) return -1;
  return bm->refcount[block];
}

int64_t pa_bm_shared_prefix(const pa_block_manager* bm, const int64_t* seqs, int n) {
  if (bm == nullptr || seqs == nullptr || n < 1) return PA_EINVAL;
  std::vector<const pa_block_manager::Seq*> members;
  members.reserve(n);
  int64_t pages = INT64_MAX;
  for (int i = 0; i < n; ++i) {
    auto it = bm->seqs.find(seqs[i]);
    if (it == bm->seqs.end()) return PA_EINVAL;
    members.push_back(&it->second);
    // whole pages inside this member's context
    pages = std::min(pages, it->second.tokens / bm->block_size);
  }
  int64_t j = 0;
  for (; j < pages; ++j) {
    const int32_t b = members[0]->blocks[j];
    bool same = true;
    for (int i = 1; i < n && same; ++i) same = members[i]->blocks[j] == b;
    if (!same) break;
  }
  return j * bm->block_size;
}

}  // extern "C"

// ------------------------------------------------------------------ scheduler

struct pa_scheduler {
  struct Req {
    int64_t id;
    int64_t prompt;
    int64_t max_new;
    int64_t prefilled = 0;
    int64_t generated = 0;
    int64_t reserve = 0;   // blocks the request may ever hold
    int64_t step_n = 0;    // tokens scheduled in the pending step
    int plan_pos = -1;     // its row in the pending plan
    bool step_prefill = false;
    bool has_tokens = false;
    bool looked_up = false;       // prefix cache consulted (at its first prefill chunk)
    std::vector<int32_t> tokens;  // prompt, then the generated tokens (token mode)
  };
  pa_block_manager* bm = nullptr;
  int budget = 0, chunk = 0, max_running = 0;
  std::deque<Req> waiting;
  std::vector<Req> running;
  std::unordered_map<int64_t, char> known;
  int64_t finished = 0, prefill_tokens = 0, decode_tokens = 0, cached_tokens = 0;
  bool pending = false;

  int64_t held(const Req& r) const {
    auto it = bm->seqs.find(r.id);
    return it == bm->seqs.end() ? 0 : static_cast<int64_t>(it->second.blocks.size());
  }
  // free blocks not promised to running requests
  int64_t spare() const {
    int64_t promised = 0;
    for (const Req& r : running) promised += std::max<int64_t>(0, r.reserve - held(r));
    return bm->available() - promised;
  }
};

extern "C" {

pa_scheduler* pa_sched_create(pa_block_manager* bm, int token_budget, int chunk_size,
                              int max_running) {
  if (bm == nullptr || token_budget <= 0 || chunk_size <= 0 || max_running <= 0) return nullptr;
  auto* s = new (std::nothrow) pa_scheduler();
  if (s == nullptr) return nullptr;
  s->bm = bm;
  s->budget = token_budget;
  s->chunk = chunk_size;
  s->max_running = max_running;
  return s;
}

void pa_sched_destroy(pa_scheduler* s) { delete s; }

int pa_sched_submit_tokens(pa_scheduler* s, int64_t req_id, const int32_t* prompt_tokens,
                          int prompt_len, int max_new_tokens) {
  if (prompt_tokens == nullptr) return PA_EINVAL;
  const int rc = pa_sched_submit(s, req_id, prompt_len, max_new_tokens);
  if (rc != PA_OK) return rc;
  auto& r = s->waiting.back();
  r.has_tokens = true;
  r.tokens.reserve(static_cast<size_t>(prompt_len) + max_new_tokens);
  r.tokens.assign(prompt_tokens, prompt_tokens + prompt_len);
  return PA_OK;
}

int pa_sched_submit(pa_scheduler* s, int64_t req_id, int prompt_len, int max_new_tokens) {
  if (s == nullptr || prompt_len < 1 || max_new_tokens < 1 || s->known.count(req_id)) return PA_EINVAL;
  pa_scheduler::Req r;
  r.id = req_id;
  r.prompt = prompt_len;
  r.max_new = max_new_tokens;
  r.reserve = s->bm->blocks_for(static_cast<int64_t>(prompt_len) + max_new_tokens);
  if (r.reserve > s->bm->num_blocks) return PA_ENOSPACE;  // can never fit
  s->known.emplace(req_id, 1);
  s->waiting.push_back(r);
  return PA_OK;
}

int pa_sched_step(pa_scheduler* s, pa_step_plan* plan) {
  pa::TraceRange trace("pa_sched_step");
  if (s == nullptr || plan == nullptr || s->pending) return PA_EINVAL;
  pa_block_manager* bm = s->bm;
  // 1. finished sequences leave and return their blocks
  for (size_t i = 0; i < s->running.size();) {
    if (s->running[i].generated >= s->running[i].max_new) {
      pa_bm_free(bm, s->running[i].id);
      ++s->finished;
      s->running.erase(s->running.begin() + static_cast<long>(i));
    } else {
      ++i;
    }
  }
  // 2. admit waiting requests (FIFO) while their blocks fit
  while (!s->waiting.empty() && static_cast<int>(s->running.size()) < s->max_running &&
         s->spare() >= s->waiting.front().reserve) {
    pa_scheduler::Req r = std::move(s->waiting.front());
    s->waiting.pop_front();
    pa_bm_add(bm, r.id);
    s->running.push_back(std::move(r));
  }
  // 3. one token per running decode, then prefill chunks, under the budget
  std::vector<size_t> order;
  int64_t tokens = 0;
  for (size_t i = 0; i < s->running.size(); ++i) {
    auto& r = s->running[i];
    r.step_n = 0;
    if (r.prefilled == r.prompt && r.generated < r.max_new && tokens + 1 <= s->budget) {
      r.step_n = 1;
      r.step_prefill = false;
      tokens += 1;
      order.push_back(i);
    }
  }
  const size_t num_decode = order.size();
  for (size_t i = 0; i < s->running.size(); ++i) {
    auto& r = s->running[i];
    if (r.has_tokens && !r.looked_up && tokens < s->budget) {
      // prefix cache, consulted when the prompt's first chunk is about to
      // run: pages that requests ahead of it have written since it was
      // admitted count too. Cached pages are shared, the rest is prefilled.
      r.looked_up = true;
      auto& sq = bm->seqs.at(r.id);
      if (sq.tokens == 0) {
        share_cached_prefix(bm, sq, r.tokens.data(), r.prompt);
        r.prefilled = sq.tokens;
        s->cached_tokens += sq.tokens;
      }
    }
    if (r.prefilled >= r.prompt) continue;
    const int64_t n = std::min<int64_t>({static_cast<int64_t>(s->chunk), r.prompt - r.prefilled,
                                         s->budget - tokens});
    if (n <= 0) break;
    r.step_n = n;
    r.step_prefill = true;
    tokens += n;
    order.push_back(i);
  }
  // capacities
  int64_t max_blocks = 0;
  for (size_t k : order) {
    const auto& r = s->running[k];
    const auto it = bm->seqs.find(r.id);
    max_blocks = std::max(max_blocks, bm->blocks_for(it->second.tokens + r.step_n));
  }
  if (static_cast<int64_t>(order.size()) > plan->max_seqs || tokens > plan->max_tokens ||
      max_blocks > plan->max_blocks_per_seq) {
    for (auto& r : s->running) r.step_n = 0;
    return PA_EINVAL;
  }
  // 4. reserve slots and fill the plan
  plan->num_seqs = static_cast<int>(order.size());
  plan->num_tokens = static_cast<int>(tokens);
  plan->num_decode = static_cast<int>(num_decode);
  plan->num_cow = 0;
  plan->table_stride = static_cast<int>(std::max<int64_t>(max_blocks, 1));
  plan->cu_q_lens[0] = 0;
  int64_t t = 0;
  for (size_t j = 0; j < order.size(); ++j) {
    const auto& r = s->running[order[j]];
    int32_t src = -1, dst = -1, ntok = 0;
    int n_cow = 0;
    const int rc = pa_bm_append(bm, r.id, static_cast<int>(r.step_n), plan->slot_mapping + t, &src,
                                &dst, &ntok, &n_cow);
    if (rc != PA_OK) return rc;  // cannot happen: admission reserved the blocks
    if (n_cow > 0) {
      if (plan->num_cow >= plan->max_cow) return PA_EINVAL;
      plan->cow_src[plan->num_cow] = src;
      plan->cow_dst[plan->num_cow] = dst;
      if (plan->cow_ntok != nullptr) plan->cow_ntok[plan->num_cow] = ntok;
      ++plan->num_cow;
    }
    if (plan->token_ids != nullptr) {
      const int64_t pos0 = bm->seqs.at(r.id).tokens - r.step_n;  // position of the first token
      for (int64_t i = 0; i < r.step_n; ++i)
        plan->token_ids[t + i] = r.has_tokens ? r.tokens[static_cast<size_t>(pos0 + i)] : -1;
    }
    s->running[order[j]].plan_pos = static_cast<int>(j);
    t += r.step_n;
    plan->seq_ids[j] = r.id;
    plan->cu_q_lens[j + 1] = static_cast<int32_t>(t);
    plan->context_lens[j] = static_cast<int32_t>(bm->seqs.at(r.id).tokens);
    int32_t* row = plan->block_tables + j * static_cast<int64_t>(plan->table_stride);
    const int nb = pa_bm_block_table(bm, r.id, row, plan->table_stride);
    for (int k = nb; k < plan->table_stride; ++k) row[k] = -1;
  }
  s->pending = plan->num_seqs > 0;
  return PA_OK;
}

int pa_sched_commit_tokens(pa_scheduler* s, const int32_t* next_tokens) {
  pa::TraceRange trace("pa_sched_commit_tokens");
  if (s == nullptr || !s->pending) return PA_EINVAL;
  if (next_tokens == nullptr)
    for (const auto& r : s->running)
      if (r.step_n > 0 && r.has_tokens) return PA_EINVAL;  // nothing changed
  for (auto& r : s->running) {
    if (r.step_n == 0) continue;
    bool yields;
    if (r.step_prefill) {
      r.prefilled += r.step_n;
      s->prefill_tokens += r.step_n;
      yields = r.prefilled == r.prompt;  // the last chunk yields the first token
    } else {
      s->decode_tokens += 1;
      yields = true;
    }
    if (yields) {
      r.generated += 1;
      if (r.has_tokens) r.tokens.push_back(next_tokens[r.plan_pos]);
    }
    // the pages this step completed are written: later requests may share them
    if (r.has_tokens) pa_bm_cache_pages(s->bm, r.id, r.tokens.data(), s->bm->seqs.at(r.id).tokens);
    r.step_n = 0;
    r.plan_pos = -1;
  }
  s->pending = false;
  return PA_OK;
}

int pa_sched_commit(pa_scheduler* s) { return pa_sched_commit_tokens(s, nullptr); }

int64_t pa_sched_cached_tokens(const pa_scheduler* s) { return s ? s->cached_tokens : -1; }

int pa_sched_stats(const pa_scheduler* s, int64_t* waiting, int64_t* running, int64_t* finished,
                   int64_t* prefill_tokens, int64_t* decode_tokens) {
  if (s == nullptr) return PA_EINVAL;
  if (waiting) *waiting = static_cast<int64_t>(s->waiting.size());
  if (running) *running = static_cast<int64_t>(s->running.size());
  if (finished) *finished = s->finished;
  if (prefill_tokens) *prefill_tokens = s->prefill_tokens;
  if (decode_tokens) *decode_tokens = s->decode_tokens;
  return PA_OK;
}

}  // extern "C"
