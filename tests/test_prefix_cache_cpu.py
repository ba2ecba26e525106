"""Prefix caching by page (include/pa_serving.h) against the plain reference
in oracle/prefix_cache.py, on the CPU."""
import numpy as np
import pytest

from oracle import prefix_cache as ref
from paged_kv_cache_176_gb300 import abi
from paged_kv_cache_176_gb300.serving import BlockManager, Scheduler, StepPlan, pa_page_hash

B = 16


def test_fnv1a64_published_vectors():
    # test vectors of the FNV specification (IETF draft "The FNV
    # Non-Cryptographic Hash Algorithm", FNV-1a, 64 bits)
    assert ref.fnv1a64(b"") == 0xCBF29CE484222325
    assert ref.fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert ref.fnv1a64(b"foobar") == 0x85944171F73967E8


def test_page_hash_matches_reference():
    rng = np.random.default_rng(0)
    for _ in range(50):
        toks = rng.integers(-2**31, 2**31, size=B, dtype=np.int64).astype(np.int32)
        parent = int(rng.integers(0, 2**63)) * 2 + int(rng.integers(0, 2))
        assert pa_page_hash(parent, toks) == ref.page_key(parent, toks.tolist())
    # a chain key depends on every token and on the parent
    toks = np.arange(B, dtype=np.int32)
    k = pa_page_hash(7, toks)
    assert pa_page_hash(8, toks) != k
    for i in range(B):
        t2 = toks.copy()
        t2[i] += 1
        assert pa_page_hash(7, t2) != k


def _prompts(rng, n, vocab=50):
    systems = [rng.integers(0, vocab, size=int(rng.integers(20, 120))).tolist() for _ in range(3)]
    out = []
    for _ in range(n):
        p = list(systems[int(rng.integers(0, 3))])
        if rng.random() < 0.3:  # sometimes a longer shared part (same question twice)
            p += systems[0][:32]
        p += rng.integers(0, vocab, size=int(rng.integers(1, 60))).tolist()
        out.append(p)
    return out


def test_hits_match_exact_prefix_reference():
    rng = np.random.default_rng(1)
    bm = BlockManager(4000, B)
    bm.set_prefix_cache(True)
    cache = ref.ExactPrefixCache()
    owner = {}       # prefix tuple -> block that first cached it
    live = []
    total_hit = 0
    for rid, prompt in enumerate(_prompts(rng, 120)):
        hit = bm.add_cached(rid, prompt)
        assert hit == cache.hit_tokens(prompt), rid
        total_hit += hit
        table = bm.block_table(rid)
        for j in range(hit // B):
            assert table[j] == owner[tuple(prompt[:B * (j + 1)])]
        bm.append(rid, len(prompt) - hit)          # prefill the rest
        bm.cache_pages(rid, prompt)
        cache.add(prompt)
        table = bm.block_table(rid)
        for j in range(len(prompt) // B):
            owner.setdefault(tuple(prompt[:B * (j + 1)]), int(table[j]))
        live.append(rid)
        if rng.random() < 0.4:                      # some requests finish
            bm.free(live.pop(int(rng.integers(0, len(live)))))
    assert total_hit > 0
    # reference counts: every block is held by exactly the live sequences using it
    held = {}
    for rid in live:
        for b in bm.block_table(rid):
            held[int(b)] = held.get(int(b), 0) + 1
    for b in range(4000):
        assert bm.refcount(b) == held.get(b, 0)
    for rid in live:
        bm.free(rid)
    assert bm.num_free == 4000  # cached blocks nobody holds count as free


def test_one_token_is_always_left_to_compute():
    bm = BlockManager(16, B)
    bm.set_prefix_cache(True)
    p = list(range(32))
    bm.add_cached(1, p)
    bm.append(1, 32)
    bm.cache_pages(1, p)
    assert bm.num_cached == 2
    assert bm.add_cached(2, p) == 16            # 2 cached pages, but one token must run
    assert bm.add_cached(3, p + [99]) == 32
    assert bm.add_cached(4, [5] + p[1:]) == 0   # a different first token misses everything


def test_eviction_takes_the_least_recently_released_page():
    bm = BlockManager(8, B)
    bm.set_prefix_cache(True)
    a = list(range(64))                          # 4 pages
    bm.add_cached(1, a)
    bm.append(1, 64)
    bm.cache_pages(1, a)
    bm.free(1)                                   # pages stay cached, blocks count as free
    assert bm.num_free == 8 and bm.num_cached == 4
    assert bm.add_cached(2, a + [1]) == 64       # a full hit
    bm.free(2)
    b = list(range(1000, 1096))                  # 6 pages: 4 free blocks + 2 evictions
    bm.add_cached(3, b)
    bm.append(3, 96)
    assert bm.num_cached == 2 and bm.num_free == 2
    # the first released page of a was evicted: its chain no longer hits
    assert bm.add_cached(4, a + [1]) == 0
    bm.free(3)
    bm.free(4)
    assert bm.num_free == 8


def test_cache_off_drops_entries():
    bm = BlockManager(8, B)
    bm.set_prefix_cache(True)
    p = list(range(40))
    bm.add_cached(1, p)
    bm.append(1, 40)
    bm.cache_pages(1, p)
    bm.free(1)
    bm.set_prefix_cache(False)
    assert bm.num_cached == 0 and bm.num_free == 8
    assert bm.add_cached(2, p) == 0


def test_scheduler_token_mode_plans_ids_and_shares_prefixes():
    rng = np.random.default_rng(3)
    system = rng.integers(0, 1000, size=100).tolist()
    reqs = [system + rng.integers(0, 1000, size=int(rng.integers(5, 40))).tolist() for _ in range(12)]
    bm = BlockManager(400, B)
    bm.set_prefix_cache(True)
    sched = Scheduler(bm, 64, 32, 4)
    news = {}
    for rid, p in enumerate(reqs):
        sched.submit(rid, len(p), 5, tokens=p)
    plan = StepPlan(4, 64, 64)
    toks = {rid: list(p) for rid, p in enumerate(reqs)}
    sched.step(plan)
    with pytest.raises(abi.PagedAttentionError):   # token-mode steps need their tokens
        sched.commit()
    while True:
        S, T = plan.num_seqs, plan.num_tokens
        cu = plan.cu_q_lens[:S + 1]
        for j in range(S):
            sid = int(plan.seq_ids[j])
            ctx = int(plan.context_lens[j])
            ql = int(cu[j + 1] - cu[j])
            assert plan.token_ids[cu[j]:cu[j + 1]].tolist() == toks[sid][ctx - ql:ctx]
        nxt = rng.integers(0, 1000, size=S).astype(np.int32)
        for j in range(S):
            sid = int(plan.seq_ids[j])
            ql = int(cu[j + 1] - cu[j])
            if j < plan.num_decode or int(plan.context_lens[j]) == len(reqs[sid]):
                toks[sid].append(int(nxt[j]))
                news[sid] = news.get(sid, 0) + 1
        sched.commit(nxt)
        sched.step(plan)
        if plan.num_seqs == 0:
            break
    st = sched.stats()
    assert st["finished"] == 12 and all(v == 5 for v in news.values())
    # the system prompt's 6 full pages were shared by the requests admitted
    # after its first prefill finished
    assert sched.cached_tokens >= 96 and sched.cached_tokens % 16 == 0
    assert st["prefill_tokens"] + sched.cached_tokens == sum(len(p) for p in reqs)
    assert bm.num_free == 400
