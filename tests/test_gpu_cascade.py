"""Shared-prefix (cascade) decode against the oracle: the prefix pass on the
tensor cores plus the suffix decode must give the attention over each
sequence's whole context, for every group shape, split and edge case."""
import numpy as np
import pytest
import torch

import paged_kv_cache_176_gb300 as pa
from paged_kv_cache_176_gb300 import workloads as W
from parity import compare, oracle_out, run_decode, to_device

pytestmark = pytest.mark.gpu


def run_cascade(w, cu_groups, prefix_lens, db=None, ctas=0):
    db = db or to_device(w)
    if db.slot_mapping is not None:
        pa.pa_reshape_and_cache(db.k_pool, db.v_pool, db.k_new, db.v_new, db.slot_mapping,
                                d_status=db.status)
    out = torch.empty_like(db.q)
    cu = torch.tensor(cu_groups, dtype=torch.int32, device="cuda")
    pl = torch.tensor(prefix_lens, dtype=torch.int32, device="cuda")
    pa.pa_decode_cascade_with_ctas(out, db.q, db.k_pool, db.v_pool, db.block_tables,
                                   db.context_lens, cu, pl, w.scale, ctas, d_status=db.status)
    torch.cuda.synchronize()
    return out, db


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (16, 4), (32, 4), (64, 8)])
@pytest.mark.parametrize("ctas", [0, 7])
def test_cascade_groups_and_edges(hq, hkv, ctas):
    # 75 sequences: [0,70) share 400 tokens (25 blocks: a partial last key
    # tile; 70 members: several 128-row tiles and a ragged tail), [70,71) is
    # a one-member group, [71,72) a group without a prefix, [72,74) share 400
    # tokens and member 72's whole context is the prefix (empty suffix), and
    # sequence 74 is in no group. ctas=7 makes sequences straddle CTAs.
    rng = np.random.default_rng(5)
    ctx = rng.integers(420, 700, size=75)
    ctx[72] = 400
    w = W.paged_workload("cascade", 9, ctx.tolist(), [1] * 75, hq, hkv, 128, 4000,
                         torch.bfloat16, write_new=False)
    cu, pl = [0, 70, 71, 72, 74], [400, 208, 0, 400]
    w = W.share_prefix(w, cu, pl)
    out, db = run_cascade(w, cu, pl, ctas=ctas)
    assert int(db.status.item()) == 0
    compare(out, oracle_out(w), torch.bfloat16)


def test_cascade_single_block_prefix_and_f32_unsupported():
    w = W.paged_workload("cascade1", 3, [16, 17, 40, 300], [1] * 4, 16, 4, 128, 64,
                         torch.bfloat16, write_new=False)
    cu, pl = [0, 4], [16]
    w = W.share_prefix(w, cu, pl)
    out, db = run_cascade(w, cu, pl)
    assert int(db.status.item()) == 0
    compare(out, oracle_out(w), torch.bfloat16)
    wf = W.paged_workload("cascade_f32", 3, [40, 40], [1, 1], 8, 2, 128, 16, torch.float32,
                          write_new=False)
    with pytest.raises(pa.abi.PagedAttentionError):
        run_cascade(wf, [0, 2], [16])


def test_cascade_bad_prefix_flagged_and_zeroed():
    w = W.paged_workload("cascade_bad", 4, [100, 120, 90, 200, 64], [1] * 5, 16, 4, 128, 64,
                         torch.bfloat16, write_new=False)
    cu = [0, 2, 4]                         # sequence 4 is in no group
    w = W.share_prefix(w, cu, [32, 80])
    ref = oracle_out(w)
    out, db = run_cascade(w, cu, [32, 80])
    assert int(db.status.item()) == 0
    compare(out, ref, torch.bfloat16)
    out, db = run_cascade(w, cu, [40, 80])  # group 0: not whole blocks
    assert int(db.status.item()) & pa.abi.PA_STATUS_BAD_LENGTH
    assert torch.count_nonzero(out[0:2]) == 0
    compare(out[2:], ref[2:], torch.bfloat16)
    out, db = run_cascade(w, cu, [32, 208])  # group 1: longer than both contexts
    assert int(db.status.item()) & pa.abi.PA_STATUS_BAD_LENGTH
    assert torch.count_nonzero(out[2:4]) == 0
    compare(out[:2], ref[:2], torch.bfloat16)
    compare(out[4:], ref[4:], torch.bfloat16)


def test_cascade_shared_prefix_full():
    w = W.shared_prefix_decode()
    S = w.num_seqs
    plen = w.info["shared_pages"] * 16
    out, db = run_cascade(w, [0, S], [plen])
    assert int(db.status.item()) == 0
    ref = oracle_out(w)
    compare(out, ref, torch.bfloat16)
    plain, _ = run_decode(w)
    compare(plain, ref, torch.bfloat16)
    # per-request groups over the whole prompt pages as well
    R, rep = w.info["num_requests"], w.info["replies"]
    prompt_full = (1100 // 16) * 16
    cu = [r * rep for r in range(R + 1)]
    out2, db2 = run_cascade(w, cu, [prompt_full] * R)
    assert int(db2.status.item()) == 0
    compare(out2, ref, torch.bfloat16)


# ------------------------------------------------------------- two levels


def run_nested(w, cu_groups, prefix_lens, cu_sib, sib_lens, db=None, ctas=0):
    db = db or to_device(w)
    if db.slot_mapping is not None:
        pa.pa_reshape_and_cache(db.k_pool, db.v_pool, db.k_new, db.v_new, db.slot_mapping,
                                d_status=db.status)
    out = torch.empty_like(db.q)

    def t(x):
        return torch.tensor(list(x), dtype=torch.int32, device="cuda")

    pa.pa_decode_cascade_nested(out, db.q, db.k_pool, db.v_pool, db.block_tables, db.context_lens,
                                t(cu_groups), t(prefix_lens), t(cu_sib), t(sib_lens), w.scale,
                                ctas, d_status=db.status)
    torch.cuda.synchronize()
    return out, db


@pytest.mark.parametrize("ctas", [0, 7])
@pytest.mark.parametrize("first_level", [True, False])
def test_nested_cascade_shared_prefix_full(ctas, first_level):
    """The shared-prefix batch (256 requests x 3 replies): the 62 pages of the
    system prompt once per batch (first level, or inside every entry without
    it) and each request's 68 full prompt pages once per entry of 4 replies
    (32/8 heads: 16 / 4 members per tile)."""
    w = W.shared_prefix_decode()
    S = w.num_seqs
    R, rep = w.info["num_requests"], w.info["replies"]
    plen = w.info["shared_pages"] * 16
    prompt_full = (w.info["prompt_len"] // 16) * 16
    assert prompt_full == 1088
    cu_sib = [r * rep for r in range(R + 1)]
    groups = ([0, S], [plen]) if first_level else ([0], [])
    out, db = run_nested(w, *groups, cu_sib, [prompt_full] * R, ctas=ctas)
    assert int(db.status.item()) == 0
    compare(out, oracle_out(w), torch.bfloat16)


# 48 sequences. First level: [0, 30) share 160 tokens, [30, 36) a group
# without a prefix, 36.. in none. Sibling groups (cu_sib / lengths below):
# 3 members; 6 (entries of 4 + 2 at 4 query heads per KV head); 1; 5 whose
# shared length is just the first-level prefix (no second-level blocks); 15
# (entries 4 + 4 + 4 + 3); 3 without a first-level prefix; 3 sharing nothing
# (entries of own blocks only); 5 outside the first level; 41.. in none.
NESTED_CU_GROUPS, NESTED_PREFIX = [0, 30, 36], [160, 0]
NESTED_CU_SIB = [0, 3, 9, 10, 15, 30, 33, 36, 41]
NESTED_SIB_LENS = [288, 320, 208, 160, 400, 96, 0, 256]


def nested_workload(hq, hkv, seed=11):
    rng = np.random.default_rng(seed)
    ctx = rng.integers(300, 700, size=48)
    ctx[15:30] = rng.integers(400, 700, size=15)
    ctx[3:9] = rng.integers(320, 700, size=6)
    ctx[3] = 320    # an entry's first member whose whole context is shared
    ctx[5] = 320    # a later member, likewise (no own blocks)
    ctx[16] = 400
    w = W.paged_workload("nested", seed, ctx.tolist(), [1] * 48, hq, hkv, 128, 2000,
                         torch.bfloat16, write_new=False)
    w = W.share_prefix(w, NESTED_CU_SIB, NESTED_SIB_LENS)
    return W.share_prefix(w, NESTED_CU_GROUPS, NESTED_PREFIX)


@pytest.mark.parametrize("hq,hkv", [(32, 8), (64, 8), (16, 8), (8, 8), (16, 4)])
@pytest.mark.parametrize("ctas", [0, 7, 40])
def test_nested_cascade_groups_and_edges(hq, hkv, ctas):
    """Every entry size the tile allows (16 / G members: 4, 2, 8, 16; hkv 4 runs
    the CUDA-core decode, which walks each member on its own), ragged last
    entries, members without own blocks, sibling groups with and without a
    first-level prefix and without second-level blocks; ctas 7 and 40 cut
    entries across CTAs (40: most entries span several)."""
    w = nested_workload(hq, hkv)
    ref = oracle_out(w)
    out, db = run_nested(w, NESTED_CU_GROUPS, NESTED_PREFIX, NESTED_CU_SIB, NESTED_SIB_LENS,
                         ctas=ctas)
    assert int(db.status.item()) == 0
    compare(out, ref, torch.bfloat16)
    # the second level alone
    out, db = run_nested(w, [0], [], NESTED_CU_SIB, NESTED_SIB_LENS, ctas=ctas)
    assert int(db.status.item()) == 0
    compare(out, ref, torch.bfloat16)


def test_nested_cascade_bad_lengths_zeroed():
    """A bad sibling length zeroes its group's members; a member whose context
    is shorter than the shared length is zeroed alone, unless it is the first
    member of its entry, whose table holds the shared blocks for all of them;
    a length below the first-level prefix is bad. The other rows stay exact."""
    w = nested_workload(32, 8)
    ref = oracle_out(w)
    G = 4

    def check(lens, ctx_edit, zero_rows):
        d = to_device(w)
        for s, c in ctx_edit.items():
            d.context_lens[s] = c
        out, d = run_nested(w, NESTED_CU_GROUPS, NESTED_PREFIX, NESTED_CU_SIB, lens, db=d)
        assert int(d.status.item()) & pa.abi.PA_STATUS_BAD_LENGTH
        zero = sorted(zero_rows)
        keep = [s for s in range(48) if s not in zero_rows and s not in ctx_edit]
        assert torch.count_nonzero(out[zero]) == 0
        compare(out, ref, torch.bfloat16, rows=keep)

    lens = list(NESTED_SIB_LENS)
    lens[1] = 328                      # group [3, 9): not whole blocks
    check(lens, {}, set(range(3, 9)))
    lens = list(NESTED_SIB_LENS)
    lens[0] = 144                      # group [0, 3): below the first-level prefix (160)
    check(lens, {}, {0, 1, 2})
    # group [15, 30) shares 400 tokens: member 17 (not first of its entry
    # [15, 19)) gets a context of 390, and member 23 (first of entry [23, 27))
    # one of 395: 17 alone is bad, 23..26 all are
    first = 15 + G * ((23 - 15) // G)
    assert first == 23
    check(list(NESTED_SIB_LENS), {17: 390, 23: 395}, {17, 23, 24, 25, 26})


@pytest.mark.parametrize("ctas", [0, 7])
def test_nested_cascade_bad_block_zeroed(ctas):
    """A bad block ID among an entry's shared blocks (read through its first
    member's table) zeroes every member of that entry; one among a member's
    own blocks zeroes that member alone. Both are flagged, the rest exact."""
    w = nested_workload(32, 8)
    ref = oracle_out(w)
    db = to_device(w)
    # entry [15, 19) of the sibling group [15, 30): shared blocks 10 .. 24
    # (160-token first-level prefix, 400 shared tokens), read through 15
    db.block_tables[15, 12] = w.num_blocks + 5
    # entry [19, 23): member 20 (470 tokens) has own blocks 25 .. 29
    assert int(w.context_lens[20]) == 470
    db.block_tables[20, 27] = w.num_blocks + 7
    out, db = run_nested(w, NESTED_CU_GROUPS, NESTED_PREFIX, NESTED_CU_SIB, NESTED_SIB_LENS,
                         db=db, ctas=ctas)
    assert int(db.status.item()) & pa.abi.PA_STATUS_BAD_BLOCK
    zero = [15, 16, 17, 18, 20]
    assert torch.count_nonzero(out[zero]) == 0
    compare(out, ref, torch.bfloat16, rows=[s for s in range(48) if s not in zero])
