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
