"""pa_decode_static_ws: the decode entry point that allocates nothing.

Some callers cannot allocate device memory around a library call (a host
framework that owns every device buffer, or a loop where cudaMalloc's
possible device synchronization or failure is not acceptable). For them,
pa_decode_static_ws takes its split-K scratch from a static device array in
libpa instead of a caller workspace. This file checks, through the C ABI,
that it returns what pa_decode returns, bit for bit, on two calls in a row,
each right after another batch has filled the array with its own values (the
array keeps the previous call's contents, which must not matter), and that
sizes beyond the array are rejected. It is named to be collected last.
"""
import pytest
import torch

import paged_kv_cache_176_gb300 as pa
from paged_kv_cache_176_gb300 import abi
from paged_kv_cache_176_gb300 import workloads as W
from parity import to_device

pytestmark = pytest.mark.gpu

CASES = {
    "tiny_f32": W.tiny_decode_f32,
    "decode_bf16": lambda: W.decode_b64(num_seqs=24, num_blocks=2000, ctx_range=(100, 1500)),
    "wide_gqa_bf16": lambda: W.wide_gqa_decode(num_seqs=6, ctx=700, num_blocks=400),
}
# a different batch of the same dtype run first, so that the array holds
# another call's partials when the checked call starts
OTHER = {
    "tiny_f32": lambda: W.paged_workload("other_f32", 7, [300, 5, 1000, 64, 17, 900], [1] * 6, 8, 2,
                                         64, 200, torch.float32, write_new=False),
    "decode_bf16": lambda: W.decode_b64(seed=3, num_seqs=40, num_blocks=3000, ctx_range=(30, 2500)),
    "wide_gqa_bf16": lambda: W.wide_gqa_decode(seed=4, num_seqs=9, ctx=1500, num_blocks=1000),
}


def _static(w, db):
    out = torch.full_like(db.q, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    abi.pa_decode_static_ws(out, db.q, db.k_pool, db.v_pool, db.block_tables, db.context_lens,
                            w.scale, d_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out


@pytest.mark.parametrize("name", sorted(CASES))
def test_static_workspace_matches_pa_decode(name):
    """pa_decode_static_ws returns exactly what pa_decode returns: both run the
    same kernels with the same split, so the outputs are bit-identical. The
    checked batch runs twice, each time right after another batch has left
    its own partials in the shared array."""
    w = CASES[name]()
    db = to_device(w)
    if db.slot_mapping is not None:
        pa.pa_reshape_and_cache(db.k_pool, db.v_pool, db.k_new, db.v_new, db.slot_mapping)
    ref = torch.empty_like(db.q)
    pa.pa_decode(ref, db.q, db.k_pool, db.v_pool, db.block_tables, db.context_lens, w.scale)
    wo = OTHER[name]()
    dbo = to_device(wo)
    for _ in range(2):
        _static(wo, dbo)  # leaves other partial values in the array
        out = _static(w, db)
        assert torch.equal(out, ref)


def test_static_workspace_rejects_oversized_batch():
    # enough sequences that the split-K scratch would exceed the static array
    S, hq, d = 4096, 64, 256
    need = abi.pa_decode_workspace_size(S, hq, d, 8)
    assert need > abi.PA_DECODE_STATIC_WS_BYTES
    q = torch.zeros(S, hq, d, device="cuda")
    kp = torch.zeros(4, 16, 8, d, device="cuda")
    bt = torch.zeros(S, 8, dtype=torch.int32, device="cuda")
    cl = torch.ones(S, dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PagedAttentionError) as e:
        abi.pa_decode_static_ws(torch.empty_like(q), q, kp, kp, bt, cl, 0.1)
    assert e.value.status == abi.PA_EWORKSPACE
