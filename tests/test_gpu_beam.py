"""Beam search over the paged pool: beams share their prefix blocks, the
fused KV write copies the filled slots of a shared partial block and writes
the step's tokens in one launch, and decode over the beams matches the
oracle while the device pools stay byte-identical to a host mirror."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_176_gb300 as pa
from paged_kv_cache_176_gb300.serving import (BlockManager, pa_reshape_and_cache_cow,
                                              sibling_shared_tokens)
from parity import compare

pytestmark = pytest.mark.gpu


def _bytes(t):
    t = t.contiguous().cpu()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.numpy().view(np.uint8)


def _host_apply(hk, hv, kn, vn, slots, cows):
    """The oracle's fused copy-on-write write on the host mirror."""
    src, dst, ntok = (torch.tensor([c[i] for c in cows], dtype=torch.int32) for i in range(3))
    oracle.cow_write(hk, hv, kn, vn, torch.tensor(slots, dtype=torch.int64), src, dst, ntok)


def _i32(x):
    return torch.tensor(x, dtype=torch.int32, device="cuda")


def test_fused_cow_write_bit_exact_and_bad_pairs():
    g = torch.Generator().manual_seed(6)
    nb, hkv, d = 64, 4, 128
    hk = torch.randn(nb, 16, hkv, d, generator=g).bfloat16()
    hv = torch.randn(nb, 16, hkv, d, generator=g).bfloat16()
    hk[3, 9:] = float("nan")  # unfilled slots of a shared block must not be copied
    cows = [(3, 40, 9), (3, 41, 9), (10, 42, 16), (20, 43, 0)]
    slots = [40 * 16 + 9, 40 * 16 + 10, 41 * 16 + 9, 43 * 16, 43 * 16 + 1, 50 * 16 + 7, -1]
    kn = torch.randn(len(slots), hkv, d, generator=g).bfloat16()
    vn = torch.randn(len(slots), hkv, d, generator=g).bfloat16()
    dk, dv = hk.cuda(), hv.cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    src, dst, ntok = (_i32([c[i] for c in cows]) for i in range(3))
    pa_reshape_and_cache_cow(dk, dv, kn.cuda(), vn.cuda(), torch.tensor(slots, device="cuda"),
                             src, dst, ntok, d_status=st)
    torch.cuda.synchronize()
    _host_apply(hk, hv, kn, vn, slots, cows)
    assert int(st.item()) == 0
    assert np.array_equal(_bytes(dk), _bytes(hk)) and np.array_equal(_bytes(dv), _bytes(hv))
    # pairs with a block outside the pool or too many slots are flagged and skipped
    before_k, before_v = _bytes(dk).copy(), _bytes(dv).copy()
    pa_reshape_and_cache_cow(dk, dv, None, None, None, _i32([1, 2]), _i32([nb, 5]), _i32([4, 17]),
                             d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & pa.abi.PA_STATUS_BAD_BLOCK
    assert np.array_equal(_bytes(dk), before_k) and np.array_equal(_bytes(dv), before_v)


@pytest.mark.parametrize("dtype,hq,hkv,d", [(torch.bfloat16, 16, 4, 128), (torch.float32, 8, 2, 64)])
def test_beam_search_decode_matches_oracle(dtype, hq, hkv, d):
    B, steps, prompt, nb = 4, 40, 37, 96
    g = torch.Generator().manual_seed(8)
    rng = np.random.default_rng(9)
    hk = torch.full((nb, 16, hkv, d), float("nan"), dtype=dtype)
    hv = hk.clone()
    dk, dv = hk.cuda(), hv.cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = d ** -0.5
    bm = BlockManager(nb)
    bm.add(0)
    slots, _ = bm.append(0, prompt)
    kn = torch.randn(prompt, hkv, d, generator=g).to(dtype)
    vn = torch.randn(prompt, hkv, d, generator=g).to(dtype)
    pa_reshape_and_cache_cow(dk, dv, kn.cuda(), vn.cuda(), torch.from_numpy(slots).cuda(), None,
                             None, None, d_status=st)
    _host_apply(hk, hv, kn, vn, slots.tolist(), [])
    beams, next_id, n_cow = [0], 1, 0
    for step in range(steps):
        parents = rng.integers(0, len(beams), size=B)
        new = list(range(next_id, next_id + B))
        next_id += B
        bm.beam_step(beams, parents, new)
        beams = new
        slots, cows = [], []
        for b in beams:
            s, c = bm.append(b, 1)
            slots.append(int(s[0]))
            cows += c
        n_cow += len(cows)
        kn = torch.randn(B, hkv, d, generator=g).to(dtype)
        vn = torch.randn(B, hkv, d, generator=g).to(dtype)
        src, dst, ntok = (_i32([c[i] for c in cows]) if cows else None for i in range(3))
        pa_reshape_and_cache_cow(dk, dv, kn.cuda(), vn.cuda(), torch.tensor(slots, device="cuda"),
                                 src, dst, ntok, d_status=st)
        _host_apply(hk, hv, kn, vn, slots, cows)
        ctx = [bm.num_tokens(b) for b in beams]
        mb = max((c + 15) // 16 for c in ctx)
        tables = torch.full((B, mb), -1, dtype=torch.int32)
        for i, b in enumerate(beams):
            t = bm.block_table(b)
            tables[i, :len(t)] = torch.from_numpy(t)
        q = torch.randn(B, hq, d, generator=g).to(dtype)
        out = torch.empty(B, hq, d, dtype=dtype, device="cuda")
        pa.pa_decode(out, q.cuda(), dk, dv, tables.cuda(), _i32(ctx), scale, d_status=st)
        torch.cuda.synchronize()
        ref = oracle.paged_attention(q, hk, hv, torch.arange(B + 1, dtype=torch.int32),
                                     torch.tensor(ctx, dtype=torch.int32), tables, scale)
        compare(out, ref, dtype)
        # beams share their common prefix: far fewer blocks than private copies
        assert nb - bm.num_free <= sum((c + 15) // 16 for c in ctx)
    assert int(st.item()) == 0 and n_cow > 0
    assert np.array_equal(_bytes(dk), _bytes(hk)) and np.array_equal(_bytes(dv), _bytes(hv))
    for b in beams:
        bm.free(b)
    assert bm.num_free == nb


@pytest.mark.parametrize("B", [4, 6])
def test_beam_search_nested_cascade_decode(B):
    """Beam search decoded with pa_decode_cascade_nested, each request's beams
    one sibling group whose shared length is the pages their block tables
    have in common: the shared pages are read once per entry of 4 beams (bf16,
    32/8 heads: 16/4 rows per tile; 6 beams make entries of 4 and 2), and
    the result matches the oracle and pa_decode. Two requests, so the groups
    sit side by side in one batch."""
    dtype, hq, hkv, d = torch.bfloat16, 32, 8, 128
    R, steps, prompt, nb = 2, 24, 300, 256
    g = torch.Generator().manual_seed(11)
    rng = np.random.default_rng(12)
    hk = torch.full((nb, 16, hkv, d), float("nan"), dtype=dtype)
    hv = hk.clone()
    dk, dv = hk.cuda(), hv.cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = d ** -0.5
    bm = BlockManager(nb)
    beams, next_id = [], 0
    for r in range(R):
        bm.add(next_id)
        slots, _ = bm.append(next_id, prompt + 7 * r)
        kn = torch.randn(len(slots), hkv, d, generator=g).to(dtype)
        vn = torch.randn(len(slots), hkv, d, generator=g).to(dtype)
        pa_reshape_and_cache_cow(dk, dv, kn.cuda(), vn.cuda(), torch.from_numpy(slots).cuda(), None,
                                 None, None, d_status=st)
        _host_apply(hk, hv, kn, vn, slots.tolist(), [])
        beams.append([next_id])
        next_id += 1
    shared_seen = 0
    for step in range(steps):
        slots, cows, order = [], [], []
        for r in range(R):
            parents = rng.integers(0, len(beams[r]), size=B)
            new = list(range(next_id, next_id + B))
            next_id += B
            bm.beam_step(beams[r], parents, new)
            beams[r] = new
            for b in new:
                s_, c_ = bm.append(b, 1)
                slots.append(int(s_[0]))
                cows += c_
                order.append(b)
        S = len(order)
        kn = torch.randn(S, hkv, d, generator=g).to(dtype)
        vn = torch.randn(S, hkv, d, generator=g).to(dtype)
        src, dst, ntok = (_i32([c[i] for c in cows]) if cows else None for i in range(3))
        pa_reshape_and_cache_cow(dk, dv, kn.cuda(), vn.cuda(), torch.tensor(slots, device="cuda"),
                                 src, dst, ntok, d_status=st)
        _host_apply(hk, hv, kn, vn, slots, cows)
        ctx = [bm.num_tokens(b) for b in order]
        mb = max((c + 15) // 16 for c in ctx)
        tables = torch.full((S, mb), -1, dtype=torch.int32)
        for i, b in enumerate(order):
            t = bm.block_table(b)
            tables[i, :len(t)] = torch.from_numpy(t)
        lens = [sibling_shared_tokens(tables[r * B:(r + 1) * B].numpy(), ctx[r * B:(r + 1) * B])
                for r in range(R)]
        # the native block manager's answer from its own tables
        assert lens == [bm.shared_prefix(order[r * B:(r + 1) * B]) for r in range(R)]
        shared_seen += sum(lens)
        q = torch.randn(S, hq, d, generator=g).to(dtype)
        out = torch.empty(S, hq, d, dtype=dtype, device="cuda")
        pa.pa_decode_cascade_nested(out, q.cuda(), dk, dv, tables.cuda(), _i32(ctx), _i32([0]),
                                    _i32([]), _i32([r * B for r in range(R + 1)]), _i32(lens),
                                    scale, d_status=st)
        plain = torch.empty_like(out)
        pa.pa_decode(plain, q.cuda(), dk, dv, tables.cuda(), _i32(ctx), scale, d_status=st)
        torch.cuda.synchronize()
        ref = oracle.paged_attention(q, hk, hv, torch.arange(S + 1, dtype=torch.int32),
                                     torch.tensor(ctx, dtype=torch.int32), tables, scale)
        compare(out, ref, dtype)
        compare(plain, ref, dtype)
    assert int(st.item()) == 0
    assert shared_seen >= steps * R * (prompt // 16) * 16  # the prompt pages at least
