"""Pins of the fp64 oracle to what the pages and the mathematics fix.

Each ``pin_*`` function takes a loaded oracle library (the real build, or a
copy with a planted mistake) and raises ``AssertionError`` when the oracle
disagrees with the pinned fact. ``test_oracle_pins.py`` runs them on the real
oracle; ``test_oracle_mutants.py`` checks that every planted mistake trips at
least one of them.

What pins what:

* brute force (``oracle/brute.py``, separate code) on tiny inputs, including
  the toy sizes of the C13-L2 gather figure (N_blk = 6, b = 2, D = 4, n_b = 3);
* a library routine: ``torch.nn.functional.scaled_dot_product_attention`` in
  fp64 on the explicitly gathered contiguous cache (paged == contiguous after
  the gather, C13-L2 page);
* the "Chunked Prefill" page's experiment: seed 0, 1000 tokens in chunks of
  256/256/256/232, 8 heads of 64, equal to one-pass causal prefill within
  1e-5, and equal to the library's causal SDPA;
* invariance under any permutation of physical block IDs (C13-L2 page: new
  blocks' physical IDs are scattered yet logically contiguous);
* copy-on-write sharing equals private copies (C13-L2 page, parallel
  sampling; Inference-engine guide section 1.5);
* the copy-on-write copy itself, on the worked parallel-sampling case: after
  the copies and writes every reply's gathered cache is its logical token
  sequence, and nothing else changed;
* closed forms of softmax attention (one key, equal keys, constant values,
  zero query, a dominant logit, two keys);
* the worked page table of the Inference-engine guide, section 1.2
  (logical 0 -> 5, 1 -> 12, 2 -> 3 for tokens 0-15, 16-31, 32-47).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch
import torch.nn.functional as F

import oracle
from oracle import brute
from paged_kv_cache_176_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name: str) -> dict:
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _raw(t: torch.Tensor) -> np.ndarray:
    t = t.contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def _after_write(w: W.Workload, lib):
    kp, vp = w.k_pool.clone(), w.v_pool.clone()
    if w.slot_mapping is not None:
        oracle.reshape_and_cache(kp, vp, w.k_new, w.v_new, w.slot_mapping, lib=lib)
    return kp, vp


def sdpa_reference(w: W.Workload, kp: torch.Tensor, vp: torch.Tensor) -> np.ndarray:
    """Library reference: gather each sequence's cache into a contiguous
    [ctx, Hkv, d] tensor with the block table, then fp64 SDPA with the mask
    ones(q_len, ctx).tril(diagonal=ctx - q_len) and KV heads repeated in
    contiguous groups of G = Hq / Hkv."""
    b = w.block_size
    G = w.num_q_heads // w.num_kv_heads
    q = w.q.to(torch.float64)
    K = kp.to(torch.float64)
    V = vp.to(torch.float64)
    cu = w.cu_q_lens.tolist()
    out = torch.empty(q.shape, dtype=torch.float64)
    for s, ctx in enumerate(w.context_lens.tolist()):
        table = w.block_tables[s].to(torch.int64)
        pos = torch.arange(ctx)
        Kc = K[table[pos // b], pos % b]  # [ctx, Hkv, d]
        Vc = V[table[pos // b], pos % b]
        ql = cu[s + 1] - cu[s]
        qs = q[cu[s]:cu[s + 1]].transpose(0, 1).unsqueeze(0)  # [1, Hq, ql, d]
        ks = Kc.transpose(0, 1).repeat_interleave(G, dim=0).unsqueeze(0)
        vs = Vc.transpose(0, 1).repeat_interleave(G, dim=0).unsqueeze(0)
        mask = torch.ones(ql, ctx, dtype=torch.bool).tril(diagonal=ctx - ql)
        o = F.scaled_dot_product_attention(qs, ks, vs, attn_mask=mask, scale=w.scale)
        out[cu[s]:cu[s + 1]] = o[0].transpose(0, 1)
    return out.numpy()


def _mixed_small(seed: int, dtype=torch.bfloat16, hq=8, hkv=2, d=16, write_new=True,
                 num_blocks=64):
    """Small mixed batch: decode rows, a prefill chunk at an offset, a whole
    prompt, a single-token context; ragged last blocks."""
    ctx = [37, 70, 45, 1, 16, 33]
    ql = [1, 21, 45, 1, 3, 1]
    return W.paged_workload("mixed_small", seed, ctx, ql, hq, hkv, d, num_blocks, dtype,
                            write_new=write_new)


# --------------------------------------------------------------------- pins


def pin_brute_tiny(lib) -> None:
    """oracle == brute force on the tiny fp32 decode config, the gather
    figure's toy sizes (b = 2, D = 2 heads x 2), and a small mixed bf16 batch."""
    cases = [W.tiny_decode_f32()]
    cases.append(W.paged_workload("toy_gather", 1, [6, 4], [3, 1], 4, 2, 2, 6,
                                  torch.bfloat16, write_new=True, block_size=2))
    cases.append(_mixed_small(2, hq=4, hkv=2, d=8))
    for w in cases:
        kp, vp = w.k_pool.clone(), w.v_pool.clone()
        kb, vb = _raw(kp), _raw(vp)
        if w.slot_mapping is not None:
            oracle.reshape_and_cache(kp, vp, w.k_new, w.v_new, w.slot_mapping, lib=lib)
            brute.reshape_and_cache(kb, vb, _raw(w.k_new), _raw(w.v_new), w.slot_mapping.tolist())
            assert np.array_equal(_raw(kp).view(np.uint8), kb.view(np.uint8)), w.name
            assert np.array_equal(_raw(vp).view(np.uint8), vb.view(np.uint8)), w.name
        got = oracle.paged_attention(w.q, kp, vp, w.cu_q_lens, w.context_lens, w.block_tables,
                                     w.scale, lib=lib)
        ref = brute.paged_attention(_raw(w.q), kb, vb, w.cu_q_lens.tolist(),
                                    w.context_lens.tolist(), w.block_tables.tolist(), w.scale)
        assert np.all(np.isfinite(got)), w.name
        err = float(np.max(np.abs(got - ref)))
        assert err < 1e-12, (w.name, err)


def pin_sdpa(lib) -> None:
    """oracle == fp64 SDPA on the gathered contiguous cache (GQA groups 1, 2,
    4; fp32 and bf16; decode rows and prefill chunks)."""
    cases = [
        _mixed_small(3, torch.bfloat16, hq=8, hkv=2, d=16),
        _mixed_small(4, torch.float32, hq=4, hkv=4, d=32),
        _mixed_small(5, torch.bfloat16, hq=6, hkv=3, d=8, write_new=False),
        W.tiny_decode_f32(),
    ]
    for w in cases:
        kp, vp = _after_write(w, lib)
        got = oracle.paged_attention(w.q, kp, vp, w.cu_q_lens, w.context_lens, w.block_tables,
                                     w.scale, lib=lib)
        ref = sdpa_reference(w, kp, vp)
        err = float(np.max(np.abs(got - ref)))
        assert err < 1e-10, (w.name, err)


def chunked_prefill_example(lib):
    """The glossary page's experiment run through the oracle on a paged pool:
    the prompt's K/V grows chunk by chunk through the KV write, each chunk
    attends to everything cached so far plus itself."""
    g = _golden("chunked_prefill_example.json")
    torch.manual_seed(g["seed"])
    q, k, v = torch.randn(*g["randn_shape"]).unbind(0)  # [1, 8, L, 64] each
    L, chunk, H, d = g["prompt_len"], g["chunk"], g["heads"], g["head_dim"]
    b = W.BLOCK_SIZE
    nblk = (L + b - 1) // b
    num_blocks = nblk + 17
    perm = np.random.default_rng(0).permutation(num_blocks)[:nblk].astype(np.int32)
    table = torch.from_numpy(perm).reshape(1, nblk)
    qt = q[0].transpose(0, 1).contiguous()  # [L, H, d]
    kt = k[0].transpose(0, 1).contiguous()
    vt = v[0].transpose(0, 1).contiguous()
    pos = np.arange(L)
    slots = torch.from_numpy(perm[pos // b].astype(np.int64) * b + pos % b)
    scale = 1.0 / math.sqrt(d)

    def run(start: int, end: int, kp, vp):
        oracle.reshape_and_cache(kp, vp, kt[start:end], vt[start:end], slots[start:end], lib=lib)
        cu = torch.tensor([0, end - start], dtype=torch.int32)
        ctx = torch.tensor([end], dtype=torch.int32)
        return oracle.paged_attention(qt[start:end], kp, vp, cu, ctx, table, scale, lib=lib)

    def fresh():
        return (torch.full((num_blocks, b, H, d), float("nan")),
                torch.full((num_blocks, b, H, d), float("nan")))

    kp, vp = fresh()
    outs, sizes = [], []
    for start in range(0, L, chunk):
        end = min(start + chunk, L)
        sizes.append(end - start)
        outs.append(run(start, end, kp, vp))
    chunked = np.concatenate(outs, axis=0)
    kp1, vp1 = fresh()
    one_pass = run(0, L, kp1, vp1)
    lib_fp64 = F.scaled_dot_product_attention(q.double(), k.double(), v.double(), is_causal=True)
    lib_fp32 = F.scaled_dot_product_attention(q, k, v, is_causal=True)
    return {
        "golden": g,
        "sizes": sizes,
        "chunked": chunked,
        "one_pass": one_pass,
        "sdpa_fp64": lib_fp64[0].transpose(0, 1).numpy(),
        "sdpa_fp32": lib_fp32[0].transpose(0, 1).double().numpy(),
    }


def pin_chunked_prefill(lib) -> None:
    r = chunked_prefill_example(lib)
    g = r["golden"]
    assert len(r["sizes"]) == g["printed_num_chunks"]
    assert r["sizes"] == g["printed_chunk_sizes"]
    # the page prints: same result as one pass (allclose, atol 1e-5) -> True
    assert np.allclose(r["one_pass"], r["chunked"], atol=g["atol"], rtol=0) == g["printed_same_as_one_pass"]
    # and the oracle is the library's causal attention
    assert float(np.max(np.abs(r["one_pass"] - r["sdpa_fp64"]))) < 1e-12
    assert float(np.max(np.abs(r["chunked"] - r["sdpa_fp64"]))) < 1e-12
    assert float(np.max(np.abs(r["chunked"] - r["sdpa_fp32"]))) < g["atol"]


def permute_pool(w: W.Workload, seed: int) -> W.Workload:
    """Relabel physical block IDs by a random permutation pi:
    pool'[pi(i)] = pool[i], table' = pi(table), slot' = pi(block)*b + offset."""
    nb, b = w.num_blocks, w.block_size
    pi = torch.from_numpy(np.random.default_rng(seed).permutation(nb).astype(np.int64))
    kp = torch.empty_like(w.k_pool)
    vp = torch.empty_like(w.v_pool)
    kp[pi] = w.k_pool
    vp[pi] = w.v_pool
    bt = w.block_tables.to(torch.int64)
    bt2 = torch.where(bt >= 0, pi[bt.clamp(min=0)], bt).to(torch.int32)
    sm = None
    if w.slot_mapping is not None:
        s = w.slot_mapping
        sm = torch.where(s >= 0, pi[(s // b).clamp(min=0)] * b + s % b, s)
    return W.Workload(w.name + "_perm", w.dtype, w.num_q_heads, w.num_kv_heads, w.head_dim, b,
                      kp, vp, w.q, w.cu_q_lens, w.context_lens, bt2, w.k_new, w.v_new, sm,
                      w.scale, w.token_budget, dict(w.info))


def pin_permutation(lib) -> None:
    for w in (_mixed_small(6), W.tiny_decode_f32()):
        a = oracle.workload_attention(w, lib=lib)
        for seed in (1, 2):
            bperm = oracle.workload_attention(permute_pool(w, seed), lib=lib)
            assert np.array_equal(a, bperm), w.name


def pin_cow(lib) -> None:
    shared = W.shared_prefix_decode(seed=1, num_requests=3, prefix_len=70, unique_len=13,
                                    reply_range=(5, 40), num_q_heads=4, num_kv_heads=2,
                                    head_dim=8)
    private = W.shared_prefix_decode(seed=1, num_requests=3, prefix_len=70, unique_len=13,
                                     reply_range=(5, 40), num_q_heads=4, num_kv_heads=2,
                                     head_dim=8, private=True)
    assert shared.num_blocks < private.num_blocks
    bt = shared.block_tables
    assert torch.equal(bt[0, :4], bt[-1, :4])  # prefix pages shared across requests
    a = oracle.workload_attention(shared, lib=lib)
    b = oracle.workload_attention(private, lib=lib)
    assert np.array_equal(a, b)
    kp, vp = _after_write(private, lib)
    ref = sdpa_reference(private, kp, vp)
    assert float(np.max(np.abs(b - ref))) < 1e-10


def pin_closed_forms(lib) -> None:
    g = torch.Generator().manual_seed(7)
    d, hq, hkv = 16, 4, 2

    def run(ctx, k, v, q, scale=0.25):
        b = W.BLOCK_SIZE
        nblk = (ctx + b - 1) // b
        kp = torch.full((nblk + 2, b, hkv, d), float("nan"))
        vp = torch.full((nblk + 2, b, hkv, d), float("nan"))
        table = torch.arange(nblk + 1, 1, -1, dtype=torch.int32)[:nblk].reshape(1, nblk)
        for p in range(ctx):
            kp[table[0, p // b], p % b] = k[p]
            vp[table[0, p // b], p % b] = v[p]
        return oracle.paged_attention(q, kp, vp, torch.tensor([0, 1], dtype=torch.int32),
                                      torch.tensor([ctx], dtype=torch.int32), table, scale,
                                      lib=lib)[0]

    q = torch.randn(1, hq, d, generator=g)
    # one key: output is that key's value
    k1, v1 = torch.randn(1, hkv, d, generator=g), torch.randn(1, hkv, d, generator=g)
    o = run(1, k1, v1, q)
    for h in range(hq):
        assert np.array_equal(o[h], v1[0, h // (hq // hkv)].double().numpy())
    ctx = 37
    v = torch.randn(ctx, hkv, d, generator=g)
    # all keys equal: output is the mean of the values
    k_eq = torch.randn(1, hkv, d, generator=g).expand(ctx, hkv, d).contiguous()
    o = run(ctx, k_eq, v, q)
    mean = v.double().mean(0).numpy()
    for h in range(hq):
        assert np.max(np.abs(o[h] - mean[h // (hq // hkv)])) < 1e-13
    # constant values: output is that constant
    k = torch.randn(ctx, hkv, d, generator=g)
    c = torch.randn(1, hkv, d, generator=g).expand(ctx, hkv, d).contiguous()
    o = run(ctx, k, c, q)
    for h in range(hq):
        assert np.max(np.abs(o[h] - c[0, h // (hq // hkv)].double().numpy())) < 1e-13
    # zero query: uniform weights
    o = run(ctx, k, v, torch.zeros(1, hq, d))
    for h in range(hq):
        assert np.max(np.abs(o[h] - mean[h // (hq // hkv)])) < 1e-13
    # a dominant logit (|x| ~ 1e4): the output is that key's value exactly
    kd = torch.zeros(ctx, hkv, d)
    kd[11, :, 0] = 1.0
    qd = torch.zeros(1, hq, d)
    qd[0, :, 0] = 4.0e4
    o = run(ctx, kd, v, qd, scale=1.0)
    for h in range(hq):
        assert np.array_equal(o[h], v[11, h // (hq // hkv)].double().numpy())
    # two keys: o = sigma(x0 - x1) v0 + sigma(x1 - x0) v1
    k2, v2 = torch.randn(2, hkv, d, generator=g), torch.randn(2, hkv, d, generator=g)
    o = run(2, k2, v2, q, scale=0.3)
    for h in range(hq):
        gh = h // (hq // hkv)
        x0 = 0.3 * float((q[0, h].double() * k2[0, gh].double()).sum())
        x1 = 0.3 * float((q[0, h].double() * k2[1, gh].double()).sum())
        w0 = 1.0 / (1.0 + math.exp(x1 - x0))
        ref = w0 * v2[0, gh].double().numpy() + (1.0 - w0) * v2[1, gh].double().numpy()
        assert np.max(np.abs(o[h] - ref)) < 1e-13


def pin_page_table_example(lib) -> None:
    g = _golden("page_table_example.json")
    b = g["block_size"]
    table = g["logical_to_physical"]
    n_tok = g["token_ranges"][-1][1] + 1
    hkv, d, hq = 2, 8, 4
    num_blocks = max(table) + 2
    gen = torch.Generator().manual_seed(3)
    K = torch.randn(n_tok, hkv, d, generator=gen)
    V = torch.randn(n_tok, hkv, d, generator=gen)
    # the page's mapping, token by token: token t lives in logical block t // b
    slots = []
    for t in range(n_tok):
        for j, (lo, hi) in enumerate(g["token_ranges"]):
            if lo <= t <= hi:
                slots.append(table[j] * b + (t - lo))
    kp = torch.full((num_blocks, b, hkv, d), float("nan"))
    vp = torch.full((num_blocks, b, hkv, d), float("nan"))
    oracle.reshape_and_cache(kp, vp, K, V, torch.tensor(slots, dtype=torch.int64), lib=lib)
    # physical page 5 holds tokens 0-15 (A.0), page 12 tokens 16-31, page 3 tokens 32-47 (A.2)
    for j, (lo, hi) in enumerate(g["token_ranges"]):
        assert torch.equal(kp[table[j]], K[lo:hi + 1])
        assert torch.equal(vp[table[j]], V[lo:hi + 1])
    for page, label in g["physical_pool_labels"].items():
        j = int(label.split(".")[1])
        assert table[j] == int(page)
    used = set(table)
    for i in range(num_blocks):
        if i not in used:
            assert torch.isnan(kp[i]).all()
    # attention through the table equals attention over tokens 0..47 in order
    q = torch.randn(n_tok, hq, d, generator=gen)
    bt = torch.tensor([table], dtype=torch.int32)
    cu = torch.tensor([0, n_tok], dtype=torch.int32)
    ctx = torch.tensor([n_tok], dtype=torch.int32)
    got = oracle.paged_attention(q, kp, vp, cu, ctx, bt, 0.35, lib=lib)
    qs = q.double().transpose(0, 1)[None]
    ks = K.double().transpose(0, 1).repeat_interleave(hq // hkv, 0)[None]
    vs = V.double().transpose(0, 1).repeat_interleave(hq // hkv, 0)[None]
    ref = F.scaled_dot_product_attention(qs, ks, vs, is_causal=True, scale=0.35)[0].transpose(0, 1)
    assert float(np.max(np.abs(got - ref.numpy()))) < 1e-12


def pin_kv_write(lib) -> None:
    """KV write: byte-exact against the brute scatter, slot -1 skipped,
    every untouched slot unchanged."""
    w = _mixed_small(8, torch.bfloat16)
    sm = w.slot_mapping.clone()
    sm[::5] = -1
    kp, vp = w.k_pool.clone(), w.v_pool.clone()
    kb, vb = _raw(kp), _raw(vp)
    before = _raw(kp).copy()
    oracle.reshape_and_cache(kp, vp, w.k_new, w.v_new, sm, lib=lib)
    brute.reshape_and_cache(kb, vb, _raw(w.k_new), _raw(w.v_new), sm.tolist())
    assert np.array_equal(_raw(kp), kb) and np.array_equal(_raw(vp), vb)
    touched = np.zeros(before.shape[:2], dtype=bool)
    for s in sm.tolist():
        if s >= 0:
            touched[s // w.block_size, s % w.block_size] = True
    after = _raw(kp)
    assert np.array_equal(after[~touched].view(np.uint16), before[~touched].view(np.uint16))


def pin_copy_on_write(lib) -> None:
    """The copy-on-write copy, on the worked case of parallel sampling: a
    request's 3 replies share its prompt's blocks ("C13 L2 serving", parallel
    sampling; "Inference engine core techniques" 1.5). The 37-token prompt
    fills blocks 0 and 1 and 5 slots of block 2. Each reply writes its first
    token at position 37, i.e. into the shared partial block: replies 0 and 1
    copy its 5 filled slots onto fresh blocks 7 and 9 and write there; reply 2,
    the last holder, writes in place. Afterwards each reply's cache, gathered
    through its table, is exactly its logical token sequence (built without a
    pool), and every slot outside the copies and writes is unchanged."""
    g = torch.Generator().manual_seed(11)
    b, hkv, d, nb = 16, 2, 8, 12
    prompt_k = torch.randn(37, hkv, d, generator=g).bfloat16()
    prompt_v = torch.randn(37, hkv, d, generator=g).bfloat16()
    new_k = torch.randn(3, hkv, d, generator=g).bfloat16()
    new_v = torch.randn(3, hkv, d, generator=g).bfloat16()
    # free blocks hold stale values of an earlier occupant; the prompt's
    # partial block holds NaN past its 5 filled slots
    kp = torch.randn(nb, b, hkv, d, generator=g).bfloat16()
    vp = torch.randn(nb, b, hkv, d, generator=g).bfloat16()
    kp[2], vp[2] = float("nan"), float("nan")
    prompt_blocks = [4, 0, 2]  # physical blocks of logical blocks 0, 1, 2
    for pos in range(37):
        kp[prompt_blocks[pos // b], pos % b] = prompt_k[pos]
        vp[prompt_blocks[pos // b], pos % b] = prompt_v[pos]
    before = _raw(kp).copy()
    tables = [[4, 0, 7], [4, 0, 9], [4, 0, 2]]
    src, dst, ntok = [2, 2], [7, 9], [5, 5]
    slots = [t[2] * b + 5 for t in tables]
    rc = oracle.cow_write(kp, vp, new_k, new_v, torch.tensor(slots), torch.tensor(src, dtype=torch.int32),
                          torch.tensor(dst, dtype=torch.int32), torch.tensor(ntok, dtype=torch.int32),
                          lib=lib)
    assert rc == 0
    for r, table in enumerate(tables):
        want_k = torch.cat([prompt_k, new_k[r:r + 1]])
        want_v = torch.cat([prompt_v, new_v[r:r + 1]])
        pos = torch.arange(38)
        got_k = kp[torch.tensor(table)[pos // b], pos % b]
        got_v = vp[torch.tensor(table)[pos // b], pos % b]
        assert np.array_equal(_raw(got_k), _raw(want_k)) and np.array_equal(_raw(got_v), _raw(want_v)), r
    touched = np.zeros((nb, b), dtype=bool)
    for blk in dst:
        touched[blk, :6] = True
    touched[2, 5] = True
    after = _raw(kp)
    assert np.array_equal(after[~touched], before[~touched])
    # whole-block copies: a table pointing at the copy sees the source's tokens
    kp2, vp2 = kp.clone(), vp.clone()
    assert oracle.copy_blocks(kp2, vp2, torch.tensor([0, 4], dtype=torch.int32),
                              torch.tensor([11, 10], dtype=torch.int32), lib=lib) == 0
    pos = torch.arange(37)
    for tab in ([4, 0, 2], [10, 11, 2]):
        got = kp2[torch.tensor(tab)[pos // b], pos % b]
        assert np.array_equal(_raw(got), _raw(prompt_k))
    # a pair outside the pool, or with more slots than a block holds, is skipped
    kp3, vp3 = kp.clone(), vp.clone()
    rc = oracle.copy_blocks(kp3, vp3, torch.tensor([1, 3], dtype=torch.int32),
                            torch.tensor([nb, 5], dtype=torch.int32),
                            torch.tensor([4, b + 1], dtype=torch.int32), lib=lib)
    assert rc == 2 and np.array_equal(_raw(kp3), _raw(kp)) and np.array_equal(_raw(vp3), _raw(vp))


ALL_PINS = [
    pin_kv_write,
    pin_page_table_example,
    pin_closed_forms,
    pin_brute_tiny,
    pin_sdpa,
    pin_chunked_prefill,
    pin_permutation,
    pin_cow,
    pin_copy_on_write,
]
