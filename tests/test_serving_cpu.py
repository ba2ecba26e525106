"""Native block manager and scheduler (include/pa_serving.h), on the CPU."""
import numpy as np
import pytest

from paged_kv_cache_176_gb300 import abi
from paged_kv_cache_176_gb300.serving import PA_ENOSPACE, BlockManager, Scheduler, StepPlan

B = 16


def test_append_grows_block_by_block():
    bm = BlockManager(10, B)
    bm.add(1)
    slots, cow = bm.append(1, 20)
    assert cow == []
    table = bm.block_table(1)
    assert len(table) == 2 and bm.num_free == 8
    # token p lives at table[p // 16] * 16 + p % 16
    assert list(slots) == [int(table[p // B]) * B + p % B for p in range(20)]
    slots2, _ = bm.append(1, 13)  # 4 fill block 1, 9 go to a new block
    table = bm.block_table(1)
    assert len(table) == 3 and bm.num_tokens(1) == 33
    assert list(slots2) == [int(table[p // B]) * B + p % B for p in range(20, 33)]
    # at most block_size - 1 unused slots per sequence
    assert len(table) * B - bm.num_tokens(1) <= B - 1
    bm.free(1)
    assert bm.num_free == 10


def test_fork_shares_and_copy_on_write():
    bm = BlockManager(8, B)
    bm.add(1)
    bm.append(1, 20)                      # blocks b0 (full), b1 (4 tokens)
    b0, b1 = bm.block_table(1)
    bm.fork(1, 2)                         # parallel sampling: reply 2 shares the prompt
    assert bm.refcount(b0) == 2 and bm.refcount(b1) == 2 and bm.num_free == 6
    slots, cow = bm.append(2, 1)          # first write into the shared partial block
    assert len(cow) == 1 and cow[0][0] == b1 and cow[0][2] == 4  # 4 filled slots to copy
    fresh = cow[0][1]
    assert list(bm.block_table(2)) == [b0, fresh]
    assert bm.refcount(b1) == 1 and bm.refcount(fresh) == 1 and bm.refcount(b0) == 2
    assert slots[0] == fresh * B + 4
    slots, cow = bm.append(1, 1)          # the original owner writes in place
    assert cow == [] and slots[0] == b1 * B + 4
    bm.fork(2, 3)
    bm.append(3, 11)                      # reply 3 copies reply 2's partial block
    bm.append(2, 11)                      # ... so reply 2's block is no longer shared
    assert bm.refcount(b0) == 3
    for s in (1, 2, 3):
        bm.free(s)
    assert bm.num_free == 8 and all(bm.refcount(b) == 0 for b in range(8))


def test_full_shared_block_needs_no_copy():
    bm = BlockManager(4, B)
    bm.add(1)
    bm.append(1, 16)
    bm.fork(1, 2)
    slots, cow = bm.append(2, 3)
    assert cow == [] and len(bm.block_table(2)) == 2


def test_beam_step_shares_prunes_and_copies_on_write():
    bm = BlockManager(16, B)
    bm.add(1)
    bm.append(1, 20)                                   # prompt: b0 full, b1 holds 4
    b0, b1 = bm.block_table(1)
    bm.beam_step([1], [0, 0, 0, 0], [10, 11, 12, 13])  # 4 beams from the prompt
    assert bm.num_tokens(1) == -1 and bm.refcount(b0) == 4 and bm.refcount(b1) == 4
    assert bm.num_free == 14
    cows = [bm.append(beam, 1)[1] for beam in (10, 11, 12, 13)]
    # the first three writers copy the shared partial block (4 filled slots),
    # the last one finds it unshared and writes in place
    assert [len(c) for c in cows] == [1, 1, 1, 0]
    assert all(c[0][0] == b1 and c[0][2] == 4 for c in cows[:3])
    assert bm.block_table(13)[1] == b1 and bm.num_free == 11
    own = {beam: int(bm.block_table(beam)[1]) for beam in (10, 11, 12, 13)}
    # beam 11 leaves no child; beam 10 has two
    bm.beam_step([10, 11, 12, 13], [0, 0, 2, 3], [20, 21, 22, 23])
    assert bm.refcount(own[11]) == 0 and bm.refcount(own[10]) == 2 and bm.num_free == 12
    assert bm.refcount(b0) == 4
    # ids may be reused across steps
    bm.beam_step([20, 21, 22, 23], [3, 2, 1, 0], [20, 21, 22, 23])
    assert bm.refcount(own[10]) == 2 and bm.num_free == 12
    for beam in (20, 21, 22, 23):
        bm.free(beam)
    assert bm.num_free == 16 and all(bm.refcount(b) == 0 for b in range(16))


def test_beam_step_rejects_and_changes_nothing():
    bm = BlockManager(8, B)
    for sq in (1, 2):
        bm.add(sq)
        bm.append(sq, 17)
    bm.add(9)
    before = (bm.num_free, [bm.refcount(b) for b in range(8)])
    for old, par, new in (([1, 2], [0, 2], [5, 6]),     # parent index out of range
                          ([1, 2], [0, 1], [5, 5]),     # repeated new id
                          ([1, 7], [0, 1], [5, 6]),     # unknown old id
                          ([1, 1], [0, 1], [5, 6]),     # repeated old id
                          ([1, 2], [0, 1], [9, 6])):    # new id held by a live sequence
        with pytest.raises(abi.PagedAttentionError):
            bm.beam_step(old, par, new)
        assert (bm.num_free, [bm.refcount(b) for b in range(8)]) == before
    assert bm.num_tokens(1) == 17 and bm.num_tokens(2) == 17


def test_out_of_space_changes_nothing():
    bm = BlockManager(2, B)
    bm.add(1)
    with pytest.raises(abi.PagedAttentionError) as e:
        bm.append(1, 40)
    assert e.value.status == PA_ENOSPACE
    assert bm.num_tokens(1) == 0 and bm.num_free == 2
    bm.append(1, 32)
    assert bm.num_free == 0


def test_bad_ids_rejected():
    bm = BlockManager(4, B)
    bm.add(7)
    with pytest.raises(abi.PagedAttentionError):
        bm.add(7)
    with pytest.raises(abi.PagedAttentionError):
        bm.append(8, 1)
    with pytest.raises(abi.PagedAttentionError):
        bm.fork(8, 9)
    with pytest.raises(abi.PagedAttentionError):
        bm.free(8)


def run_schedule(num_blocks, budget, chunk, max_running, reqs, max_ctx=4096):
    bm = BlockManager(num_blocks, B)
    sched = Scheduler(bm, budget, chunk, max_running)
    for rid, (prompt, new) in enumerate(reqs):
        sched.submit(rid, prompt, new)
    plan = StepPlan(max_running, budget, (max_ctx + B - 1) // B)
    steps = []
    while True:
        p = sched.step(plan)
        if p.num_seqs == 0:
            break
        S, T = p.num_seqs, p.num_tokens
        cu = p.cu_q_lens[:S + 1].copy()
        ql = np.diff(cu)
        assert 0 < T <= budget and cu[-1] == T
        assert np.all(ql[:p.num_decode] == 1)          # decode tokens first
        assert np.all(ql[p.num_decode:] <= chunk)      # prefill chunks
        assert p.table_stride == max((int(c) + B - 1) // B for c in p.context_lens[:S])
        for j in range(S):
            ctx = int(p.context_lens[j])
            nb = (ctx + B - 1) // B
            row = p.tables[j]
            assert np.all(row[:nb] >= 0) and np.all(row[nb:] == -1)
            assert nb * B - ctx <= B - 1                   # paging waste bound
            for i in range(int(ql[j])):
                pos = ctx - int(ql[j]) + i
                assert p.slot_mapping[cu[j] + i] == int(row[pos // B]) * B + pos % B
        steps.append((S, T, p.num_decode))
        sched.commit()
    return bm, sched, steps


def test_scheduler_runs_every_request_to_completion():
    rng = np.random.default_rng(0)
    reqs = [(int(rng.integers(1, 900)), int(rng.integers(1, 60))) for _ in range(40)]
    bm, sched, steps = run_schedule(600, 256, 96, 16, reqs)
    st = sched.stats()
    assert st["finished"] == len(reqs) and st["waiting"] == 0 and st["running"] == 0
    assert st["prefill_tokens"] == sum(p for p, _ in reqs)
    assert st["decode_tokens"] == sum(n - 1 for _, n in reqs)
    assert bm.num_free == 600                          # every block returned
    # while prompts are waiting to be prefilled the budget is used in full
    assert max(t for _, t, _ in steps) == 256


def test_scheduler_admission_respects_pool():
    # each request can reach 8 blocks; a pool of 20 blocks runs at most 2 at once
    reqs = [(100, 28)] * 6
    bm, sched, steps = run_schedule(20, 512, 512, 8, reqs)
    assert max(s for s, _, _ in steps) <= 2
    assert sched.stats()["finished"] == 6 and bm.num_free == 20


def test_scheduler_rejects_impossible_request():
    bm = BlockManager(4, B)
    sched = Scheduler(bm, 64, 32, 4)
    with pytest.raises(abi.PagedAttentionError) as e:
        sched.submit(1, 100, 10)
    assert e.value.status == PA_ENOSPACE
    with pytest.raises(abi.PagedAttentionError):
        sched.submit(2, 0, 1)


def test_sibling_shared_tokens():
    from paged_kv_cache_176_gb300.serving import sibling_shared_tokens as shared
    t = np.array([[5, 6, 7, 8, 9], [5, 6, 7, 3, 4], [5, 6, 7, 8, 2]])
    assert shared(t, [80, 70, 75]) == 48            # 3 equal leading blocks
    assert shared(t, [80, 40, 75]) == 32            # only whole pages within every context
    assert shared(t[:1], [70]) == 64                # one member: its whole pages
    assert shared(t, [15, 70, 75]) == 0             # a member inside its first page
    assert shared(np.array([[1, 2], [9, 2]]), [32, 32]) == 0
    assert shared(np.zeros((0, 4), dtype=np.int32), []) == 0


def test_sibling_shared_tokens_on_beams():
    """Beams forked from one prompt share its full pages and, after a fork,
    every page their parent had filled; the helper finds exactly the pages
    the block manager shares (refcount equal to the number of beams)."""
    from paged_kv_cache_176_gb300.serving import sibling_shared_tokens as shared
    bm = BlockManager(64)
    bm.add(0)
    bm.append(0, 70)                                 # 4 full pages + 6 tokens
    bm.beam_step([0], [0, 0, 0], [1, 2, 3])
    for b in (1, 2, 3):
        bm.append(b, 1)                              # copy-on-write of the partial page
    rows = [bm.block_table(b) for b in (1, 2, 3)]
    ctx = [bm.num_tokens(b) for b in (1, 2, 3)]
    n = shared(np.stack([r[:5] for r in rows]), ctx)
    assert n == 64
    assert all(bm.refcount(int(rows[0][j])) == 3 for j in range(n // 16))
    assert bm.refcount(int(rows[0][4])) == 1
    # the native block manager gives the same count
    assert bm.shared_prefix([1, 2, 3]) == 64 == bm.shared_prefix([3, 1])
    assert bm.shared_prefix([2]) == 64                 # one member: its whole pages (71 tokens)
    for b in (1, 2):
        bm.append(b, 60)                             # 131 tokens: pages 4..7 private
    assert bm.shared_prefix([1, 2, 3]) == 64
    assert bm.shared_prefix([1]) == 128
    with pytest.raises(abi.PagedAttentionError):
        bm.shared_prefix([1, 99])                    # unknown sequence
    with pytest.raises(abi.PagedAttentionError):
        bm.shared_prefix([])
