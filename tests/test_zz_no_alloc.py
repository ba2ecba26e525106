"""pa_decode_static_ws: the decode entry point that allocates nothing.

Some callers cannot allocate device memory around a library call (a host
framework that owns every device buffer, or a loop where cudaMalloc's
possible device synchronization or failure is not acceptable). For them,
pa_decode_static_ws takes its split-K scratch from a static device array in
libpa instead of a caller workspace. This file checks, through the C ABI,
that it returns what pa_decode returns, on two calls in a row (the array keeps
the previous call's contents, which must not matter), and that sizes beyond
the array are rejected. It is named to be collected last.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_176_gb300 as pa
from paged_kv_cache_176_gb300 import abi
from paged_kv_cache_176_gb300 import workloads as W
from parity import BF16_ATOL, BF16_RTOL, F32_ATOL, to_device

pytestmark = pytest.mark.gpu


def _close(a: torch.Tensor, b: torch.Tensor, dtype) -> None:
    x = a.double().cpu().numpy()
    y = b.double().cpu().numpy()
    assert np.all(np.isfinite(x)) and np.all(np.isfinite(y))
    err = np.abs(x - y)
    if dtype == torch.float32:
        assert err.max() <= F32_ATOL
    else:
        assert np.all(err <= np.maximum(BF16_ATOL, BF16_RTOL * np.abs(y)))


@pytest.mark.parametrize("make", [
    W.tiny_decode_f32,
    lambda: W.decode_b64(num_seqs=24, num_blocks=2000, ctx_range=(100, 1500)),
    lambda: W.wide_gqa_decode(num_seqs=6, ctx=700, num_blocks=400),
], ids=["tiny_f32", "decode_bf16", "wide_gqa_bf16"])
def test_static_workspace_matches_pa_decode(make):
    w = make()
    db = to_device(w)
    if db.slot_mapping is not None:
        pa.pa_reshape_and_cache(db.k_pool, db.v_pool, db.k_new, db.v_new, db.slot_mapping)
    ref = torch.empty_like(db.q)
    pa.pa_decode(ref, db.q, db.k_pool, db.v_pool, db.block_tables, db.context_lens, w.scale)
    for _ in range(2):  # the second call starts from the first call's scratch contents
        out = torch.full_like(db.q, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        abi.pa_decode_static_ws(out, db.q, db.k_pool, db.v_pool, db.block_tables,
                                db.context_lens, w.scale, d_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        _close(out, ref, w.dtype)


def test_static_workspace_rejects_oversized_batch():
    w = W.tiny_decode_f32()
    db = to_device(w)
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
