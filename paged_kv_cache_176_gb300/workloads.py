"""Seeded synthetic inputs for attention over a paged KV cache.

This module only *draws* inputs: context lengths, a permutation of physical
block IDs, block tables, pool contents, queries, the new tokens' K/V and the
slot each new token is written to. It holds none of the attention arithmetic.
Both the CUDA path and the CPU oracle are fed from the tensors built here, so
they see identical bytes.

Layouts (all row-major, contiguous):

* ``k_pool``, ``v_pool``: ``[num_blocks, block_size, num_kv_heads, head_dim]``.
  This is the per-layer block pool ``[N_blk, b, D]`` of the C13-L2 course page
  ("gather K by block table" figure), with ``D = num_kv_heads * head_dim``.
* ``block_tables``: int32 ``[S, max_blocks]``; row ``s`` maps logical block
  ``j`` of sequence ``s`` to a physical block ID (the page table of the
  "Inference engine core techniques" guide, section 1.2). Entries past the
  blocks a sequence uses are -1.
* ``q``: ``[T, num_q_heads, head_dim]``; ``cu_q_lens`` int32 ``[S + 1]``.
* ``context_lens``: int32 ``[S]``, the number of cached tokens each sequence
  attends to *including* the tokens written in this step.
* ``k_new``, ``v_new``: ``[T, num_kv_heads, head_dim]``; ``slot_mapping`` int64
  ``[T]`` with ``slot = physical_block * block_size + offset`` or -1 (skip).

Value recipe: every value is an N(0, 1) draw from numpy's PCG64 generator,
rounded to bf16 with round-to-nearest-even where the workload is bf16. Pool
slots that no table references, and slots at or past a sequence's filled
length, hold NaN so that any stray read poisons the result. Each stage draws
from its own child stream of the seed (context lengths, pool permutation, pool
K/V, q, new K/V), so the values drawn at one stage do not depend on the sizes
chosen at another (e.g. a shared and a private pool hold the same tokens).
"""
from __future__ import annotations

import concurrent.futures as _fut
import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

BLOCK_SIZE = 16  # tokens per physical block (vLLM default, quoted on all pages)

_CHUNK = 1 << 22


def _normal(rng: np.random.Generator, n: int) -> np.ndarray:
    """``n`` float32 N(0,1) draws. Large draws are split over child generators
    (spawned from ``rng``) and filled by a thread pool; the result depends only
    on the seed, not on the thread count."""
    if n <= 4 * _CHUNK:
        return rng.standard_normal(n, dtype=np.float32)
    nchunks = (n + _CHUNK - 1) // _CHUNK
    children = rng.spawn(nchunks)
    out = np.empty(n, dtype=np.float32)

    def fill(i: int) -> None:
        lo = i * _CHUNK
        hi = min(n, lo + _CHUNK)
        children[i].standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])

    with _fut.ThreadPoolExecutor(max_workers=min(16, nchunks)) as ex:
        list(ex.map(fill, range(nchunks)))
    return out


def _streams(seed: int) -> List[np.random.Generator]:
    """Five independent generators: context lengths, pool permutation, pool
    K/V, queries, new K/V."""
    return [np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(5)]


def _to_dtype(x: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    t = torch.from_numpy(x)
    return t.to(dtype) if dtype != torch.float32 else t


@dataclass
class Workload:
    """One call's worth of inputs (host tensors)."""

    name: str
    dtype: torch.dtype
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    q: torch.Tensor
    cu_q_lens: torch.Tensor
    context_lens: torch.Tensor
    block_tables: torch.Tensor
    k_new: Optional[torch.Tensor]
    v_new: Optional[torch.Tensor]
    slot_mapping: Optional[torch.Tensor]
    scale: float
    token_budget: int
    info: Dict[str, object] = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.numel())

    @property
    def num_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.k_pool.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def q_lens(self) -> List[int]:
        c = self.cu_q_lens.tolist()
        return [c[i + 1] - c[i] for i in range(len(c) - 1)]

    def kv_bytes_read(self) -> int:
        """Bytes of cached K and V that attention must read once (every token
        of every context, all KV heads)."""
        elt = self.k_pool.element_size()
        per_tok = 2 * self.num_kv_heads * self.head_dim * elt
        return int(self.context_lens.to(torch.int64).sum().item()) * per_tok


def _blocks_for(n_tokens: int, b: int) -> int:
    return (n_tokens + b - 1) // b


def _new_pool(num_blocks: int, b: int, hkv: int, d: int, dtype: torch.dtype) -> torch.Tensor:
    return torch.full((num_blocks, b, hkv, d), float("nan"), dtype=dtype)


def paged_workload(
    name: str,
    seed: int,
    context_lens: Sequence[int] | None,
    q_lens: Sequence[int],
    num_q_heads: int,
    num_kv_heads: int,
    head_dim: int,
    num_blocks: int,
    dtype: torch.dtype,
    write_new: bool,
    ctx_range: tuple[int, int] | None = None,
    num_seqs: int | None = None,
    block_size: int = BLOCK_SIZE,
    token_budget: int | None = None,
    scale: float | None = None,
    table_pad: int = 0,
) -> Workload:
    """General builder: ``S`` sequences, sequence ``s`` has ``q_lens[s]`` query
    tokens and ``context_lens[s]`` cached tokens (drawn from ``ctx_range`` when
    ``context_lens`` is None). Physical block IDs are a seeded permutation of
    the pool. With ``write_new`` the last ``q_len`` tokens of each context are
    the step's new tokens: their pool slots hold NaN and ``k_new``/``v_new`` +
    ``slot_mapping`` carry their values; otherwise the pool already holds every
    context token and no write is requested.
    """
    g_ctx, g_perm, g_kv, g_q, g_new = _streams(seed)
    b = block_size
    # 1. context lengths
    if context_lens is None:
        assert ctx_range is not None and num_seqs is not None
        lo, hi = ctx_range
        context_lens = g_ctx.integers(lo, hi + 1, size=num_seqs).tolist()
    context_lens = [int(c) for c in context_lens]
    S = len(context_lens)
    q_lens = [int(x) for x in q_lens]
    assert len(q_lens) == S
    for c, ql in zip(context_lens, q_lens):
        assert 1 <= ql <= c
    nblk = [_blocks_for(c, b) for c in context_lens]
    total = sum(nblk)
    if total > num_blocks:
        raise ValueError(f"pool of {num_blocks} blocks cannot hold {total}")
    # 2. pool permutation: logical blocks are handed physical IDs in order
    perm = g_perm.permutation(num_blocks).astype(np.int64)
    max_blocks = max(nblk) + table_pad
    tables = np.full((S, max_blocks), -1, dtype=np.int32)
    used = perm[:total]
    pos = 0
    for s in range(S):
        tables[s, : nblk[s]] = used[pos : pos + nblk[s]]
        pos += nblk[s]
    # 3. pool K/V (drawn in logical order, scattered to physical IDs)
    per_blk = b * num_kv_heads * head_dim
    k_vals = _normal(g_kv, total * per_blk).reshape(total, b, num_kv_heads, head_dim)
    v_vals = _normal(g_kv, total * per_blk).reshape(total, b, num_kv_heads, head_dim)
    filled = [c - ql if write_new else c for c, ql in zip(context_lens, q_lens)]
    pos = 0
    for s in range(S):
        # slots at or past the filled length of the last blocks become NaN
        first_empty = filled[s]
        for j in range(first_empty // b, nblk[s]):
            lo = max(0, first_empty - j * b)
            k_vals[pos + j, lo:] = np.nan
            v_vals[pos + j, lo:] = np.nan
        pos += nblk[s]
    kp = _new_pool(num_blocks, b, num_kv_heads, head_dim, dtype)
    vp = _new_pool(num_blocks, b, num_kv_heads, head_dim, dtype)
    idx = torch.from_numpy(used)
    kp.index_copy_(0, idx, _to_dtype(k_vals, dtype))
    vp.index_copy_(0, idx, _to_dtype(v_vals, dtype))
    del k_vals, v_vals
    # 4. queries
    T = sum(q_lens)
    q = _normal(g_q, T * num_q_heads * head_dim).reshape(T, num_q_heads, head_dim)
    # 5. new tokens
    k_new = v_new = slots = None
    if write_new:
        k_new = _normal(g_new, T * num_kv_heads * head_dim).reshape(T, num_kv_heads, head_dim)
        v_new = _normal(g_new, T * num_kv_heads * head_dim).reshape(T, num_kv_heads, head_dim)
        slots = np.empty(T, dtype=np.int64)
        t = 0
        for s in range(S):
            for i in range(q_lens[s]):
                p = context_lens[s] - q_lens[s] + i
                slots[t] = int(tables[s, p // b]) * b + p % b
                t += 1
    cu = np.zeros(S + 1, dtype=np.int32)
    cu[1:] = np.cumsum(q_lens)
    return Workload(
        name=name,
        dtype=dtype,
        num_q_heads=num_q_heads,
        num_kv_heads=num_kv_heads,
        head_dim=head_dim,
        block_size=b,
        k_pool=kp,
        v_pool=vp,
        q=_to_dtype(np.ascontiguousarray(q), dtype),
        cu_q_lens=torch.from_numpy(cu),
        context_lens=torch.tensor(context_lens, dtype=torch.int32),
        block_tables=torch.from_numpy(tables),
        k_new=None if k_new is None else _to_dtype(np.ascontiguousarray(k_new), dtype),
        v_new=None if v_new is None else _to_dtype(np.ascontiguousarray(v_new), dtype),
        slot_mapping=None if slots is None else torch.from_numpy(slots),
        scale=(1.0 / math.sqrt(head_dim)) if scale is None else float(scale),
        token_budget=T if token_budget is None else int(token_budget),
        info={"seed": seed, "blocks_used": total},
    )


# ---------------------------------------------------------------------------
# The five workloads. Sizes follow the pages: the tiny fp32 decode, the decode batch,
# the wide-head GQA batch of the anchor model, the budgeted mixed step and
# shared-prefix sampling.
# ---------------------------------------------------------------------------


def tiny_decode_f32(seed: int = 0) -> Workload:
    """4 sequences with contexts {17, 40, 64, 100}, 8 query / 2 KV heads,
    head_dim 64, a pool of 32 blocks with permuted IDs, fp32."""
    return paged_workload(
        "tiny_decode_f32", seed, [17, 40, 64, 100], [1, 1, 1, 1], 8, 2, 64, 32,
        torch.float32, write_new=False,
    )


def decode_b64(seed: int = 0, num_seqs: int = 64, num_blocks: int = 20000,
               ctx_range=(512, 4096)) -> Workload:
    """64 decode sequences, contexts U[512, 4096], 32 query / 8 KV heads,
    head_dim 128, bf16, tables drawn from a shuffled pool of 20,000 blocks; the
    step first writes each sequence's new token (position ctx - 1)."""
    return paged_workload(
        "decode_b64_bf16", seed, None, [1] * num_seqs, 32, 8, 128, num_blocks,
        torch.bfloat16, write_new=True, ctx_range=ctx_range, num_seqs=num_seqs,
    )


def wide_gqa_decode(seed: int = 0, num_seqs: int = 58, ctx: int = 4096,
                    num_blocks: int = 23305) -> Workload:
    """58 requests at context 4096 (256 blocks each), 4 KV heads x head_dim 256
    (1,024 values per token per layer), 16 query heads, bf16, in a pool of
    23,305 blocks (the anchor model's pool on an 80 GB H100)."""
    return paged_workload(
        "wide_gqa_decode_bf16", seed, [ctx] * num_seqs, [1] * num_seqs, 16, 4, 256,
        num_blocks, torch.bfloat16, write_new=False,
    )


def mixed_step(seed: int = 0, num_decode: int = 128, decode_ctx=(1024, 8192),
               chunks=(512, 512, 512, 384), prompt_len: int = 32768,
               num_q_heads: int = 64, num_kv_heads: int = 8, head_dim: int = 128,
               token_budget: int = 2048, spare: float = 0.25) -> Workload:
    """A budgeted mixed step: ``num_decode`` decode tokens (contexts uniform in
    ``decode_ctx``) followed by one prefill chunk from each of ``len(chunks)``
    prompts of ``prompt_len`` tokens, each chunk starting at a 512-aligned
    random offset. Every token of the step (decode and prefill) is written to
    the pool by the step itself. The pool holds the blocks needed plus
    ``spare`` extra, IDs permuted. 64 query / 8 KV heads, head_dim 128, bf16."""
    rng = np.random.default_rng(seed)
    lo, hi = decode_ctx
    dctx = rng.integers(lo, hi + 1, size=num_decode).tolist()
    chunk_unit = 512
    offs = []
    for c in chunks:
        max_u = (prompt_len - c) // chunk_unit
        offs.append(int(rng.integers(0, max_u + 1)) * chunk_unit)
    ctx = dctx + [o + c for o, c in zip(offs, chunks)]
    ql = [1] * num_decode + list(chunks)
    assert sum(ql) <= token_budget
    need = sum(_blocks_for(c, BLOCK_SIZE) for c in ctx)
    nb = int(math.ceil(need * (1.0 + spare)))
    w = paged_workload(
        "mixed_step_bf16", int(rng.integers(0, 2**31 - 1)), ctx, ql, num_q_heads,
        num_kv_heads, head_dim, nb, torch.bfloat16, write_new=True,
        token_budget=token_budget,
    )
    w.info.update({"chunk_offsets": offs, "chunks": list(chunks), "num_decode": num_decode,
                   "prompt_len": prompt_len})
    return w


def shared_prefix_decode(seed: int = 0, num_requests: int = 256, replies: int = 3,
                         prefix_len: int = 1000, unique_len: int = 100,
                         reply_range=(22, 356), num_q_heads: int = 32,
                         num_kv_heads: int = 8, head_dim: int = 128,
                         private: bool = False, spare: float = 0.25) -> Workload:
    """Parallel sampling over a shared prompt prefix.

    ``num_requests`` requests share a ``prefix_len``-token system prompt and
    add ``unique_len`` tokens each. Full pages of identical prefix tokens are
    stored once and shared by every request (prefix-cache hit, refcounted);
    the page that mixes prefix and unique tokens is per request. Each request
    samples ``replies`` replies that share all of its prompt pages. The prompt's
    last page is partial, so the first write of each reply copies it while it
    is still shared (copy-on-write); the last writer finds it unshared and
    writes in place. Reply ``r`` has generated ``L ~ U[reply_range]`` tokens,
    the last of which is written by this step, so its decode context is
    ``prefix_len + unique_len + L``.

    With ``private=True`` every reply instead gets private copies of all its
    pages, holding the same values (the reference point of the CoW pin).
    """
    g_ctx, g_perm, g_kv, g_q, g_new = _streams(seed)
    b = BLOCK_SIZE
    S = num_requests * replies
    prompt = prefix_len + unique_len
    # 1. context lengths (reply lengths)
    L = g_ctx.integers(reply_range[0], reply_range[1] + 1, size=S)
    ctx = (prompt + L).astype(np.int64)
    n_shared = prefix_len // b               # full pages of pure prefix
    n_prompt = _blocks_for(prompt, b)        # pages of the prompt
    prompt_partial = prompt % b != 0
    # logical page lists per sequence, each entry a key naming its content
    # ("P", j) shared prefix page j; ("R", r, j) request r's prompt page j;
    # ("Y", s, j) sequence s's own page j.
    lists: List[List[tuple]] = []
    for r in range(num_requests):
        for k in range(replies):
            s = r * replies + k
            pages: List[tuple] = []
            for j in range(_blocks_for(int(ctx[s]), b)):
                if j < n_shared:
                    pages.append(("P", j) if not private else ("Y", s, j))
                elif j < n_prompt - (1 if prompt_partial else 0):
                    pages.append(("R", r, j) if not private else ("Y", s, j))
                elif j == n_prompt - 1 and prompt_partial:
                    # copy-on-write of the partial prompt page: the first
                    # replies - 1 writers copy it, the last keeps the original
                    if not private and k == replies - 1:
                        pages.append(("R", r, j))
                    else:
                        pages.append(("Y", s, j))
                else:
                    pages.append(("Y", s, j))
            lists.append(pages)
    keys: Dict[tuple, int] = {}
    order: List[tuple] = []
    for pages in lists:
        for key in pages:
            if key not in keys:
                keys[key] = len(order)
                order.append(key)
    n_phys = len(order)
    num_blocks = int(math.ceil(n_phys * (1.0 + spare)))
    # 2. pool permutation
    perm = g_perm.permutation(num_blocks).astype(np.int64)
    phys = {key: int(perm[i]) for i, key in enumerate(order)}
    max_blocks = max(len(p) for p in lists)
    tables = np.full((S, max_blocks), -1, dtype=np.int32)
    for s, pages in enumerate(lists):
        tables[s, : len(pages)] = [phys[k] for k in pages]
    # 3. token values: prefix tokens are common to every request, prompt
    #    tokens common to a request's replies, reply tokens per sequence.
    per_tok = num_kv_heads * head_dim
    pre_k = _normal(g_kv, prefix_len * per_tok).reshape(prefix_len, num_kv_heads, head_dim)
    pre_v = _normal(g_kv, prefix_len * per_tok).reshape(prefix_len, num_kv_heads, head_dim)
    uq_k = _normal(g_kv, num_requests * unique_len * per_tok).reshape(
        num_requests, unique_len, num_kv_heads, head_dim)
    uq_v = _normal(g_kv, num_requests * unique_len * per_tok).reshape(
        num_requests, unique_len, num_kv_heads, head_dim)
    rep_tot = int(L.sum())
    rp_k = _normal(g_kv, rep_tot * per_tok).reshape(rep_tot, num_kv_heads, head_dim)
    rp_v = _normal(g_kv, rep_tot * per_tok).reshape(rep_tot, num_kv_heads, head_dim)
    rep_off = np.zeros(S + 1, dtype=np.int64)
    rep_off[1:] = np.cumsum(L)
    kp = np.full((num_blocks, b, num_kv_heads, head_dim), np.nan, dtype=np.float32)
    vp = np.full((num_blocks, b, num_kv_heads, head_dim), np.nan, dtype=np.float32)

    def fill(s: int, p0: int, p1: int, pb: int) -> None:
        """Copy the values of sequence ``s``'s positions [p0, p1) into page
        ``pb`` starting at offset 0."""
        r = s // replies
        for lo, hi, ks, vs, base in (
            (0, prefix_len, pre_k, pre_v, 0),
            (prefix_len, prompt, uq_k[r], uq_v[r], prefix_len),
            (prompt, int(ctx[s]), rp_k[rep_off[s]:rep_off[s + 1]],
             rp_v[rep_off[s]:rep_off[s + 1]], prompt),
        ):
            a, c = max(p0, lo), min(p1, hi)
            if a < c:
                kp[pb, a - p0:c - p0] = ks[a - base:c - base]
                vp[pb, a - p0:c - p0] = vs[a - base:c - base]

    # Each physical page is filled once, from the first sequence that maps
    # it. Where several sequences share a page its positions hold identical
    # values for all of them (common prefix / common prompt); a page that
    # holds reply tokens is mapped by exactly one sequence. The newest token
    # of every sequence is written by the step itself, so it stays NaN here.
    first_map: Dict[tuple, tuple] = {}
    for s, pages in enumerate(lists):
        for j, key in enumerate(pages):
            first_map.setdefault(key, (s, j))
    for key, (s, j) in first_map.items():
        p0 = j * b
        p1 = min(p0 + b, int(ctx[s]) - 1)
        if p1 > p0:
            fill(s, p0, p1, phys[key])
    q = _normal(g_q, S * num_q_heads * head_dim).reshape(S, num_q_heads, head_dim)
    k_new = _normal(g_new, S * per_tok).reshape(S, num_kv_heads, head_dim)
    v_new = _normal(g_new, S * per_tok).reshape(S, num_kv_heads, head_dim)
    slots = np.empty(S, dtype=np.int64)
    for s in range(S):
        p = int(ctx[s]) - 1
        slots[s] = int(tables[s, p // b]) * b + p % b
    cu = np.arange(S + 1, dtype=np.int32)
    return Workload(
        name="shared_prefix_decode_bf16" + ("_private" if private else ""),
        dtype=torch.bfloat16,
        num_q_heads=num_q_heads,
        num_kv_heads=num_kv_heads,
        head_dim=head_dim,
        block_size=b,
        k_pool=_to_dtype(kp, torch.bfloat16),
        v_pool=_to_dtype(vp, torch.bfloat16),
        q=_to_dtype(np.ascontiguousarray(q), torch.bfloat16),
        cu_q_lens=torch.from_numpy(cu),
        context_lens=torch.from_numpy(ctx.astype(np.int32)),
        block_tables=torch.from_numpy(tables),
        k_new=_to_dtype(np.ascontiguousarray(k_new), torch.bfloat16),
        v_new=_to_dtype(np.ascontiguousarray(v_new), torch.bfloat16),
        slot_mapping=torch.from_numpy(slots),
        scale=1.0 / math.sqrt(head_dim),
        token_budget=S,
        info={"seed": seed, "blocks_used": n_phys, "num_requests": num_requests,
              "replies": replies, "shared_pages": n_shared, "prompt_len": prompt},
    )



def share_prefix(w: Workload, cu_groups: Sequence[int], prefix_lens: Sequence[int]) -> Workload:
    """The same workload with shared prompt prefixes: the members
    ``cu_groups[g] .. cu_groups[g+1]-1`` of group ``g`` point the first
    ``prefix_lens[g] // 16`` entries of their block tables at the first
    member's blocks (the blocks they gave up stay in the pool, unreferenced).
    Each prefix must fit every member's context. Structure only: the values
    in the pool are untouched."""
    b = w.block_size
    bt = w.block_tables.clone()
    ctx = w.context_lens
    for g in range(len(prefix_lens)):
        a, e, plen = int(cu_groups[g]), int(cu_groups[g + 1]), int(prefix_lens[g])
        nb = plen // b
        for s in range(a + 1, e):
            assert plen <= int(ctx[s]) and plen <= int(ctx[a])
            bt[s, :nb] = bt[a, :nb]
    info = dict(w.info)
    info.update(cu_groups=[int(x) for x in cu_groups], prefix_lens=[int(x) for x in prefix_lens])
    return Workload(w.name + "+shared", w.dtype, w.num_q_heads, w.num_kv_heads, w.head_dim, b,
                    w.k_pool, w.v_pool, w.q, w.cu_q_lens, w.context_lens, bt, w.k_new, w.v_new,
                    w.slot_mapping, w.scale, w.token_budget, info)

CONFIGS = {
    "tiny_decode_f32": tiny_decode_f32,
    "decode_b64_bf16": decode_b64,
    "wide_gqa_decode_bf16": wide_gqa_decode,
    "mixed_step_bf16": mixed_step,
    "shared_prefix_decode_bf16": shared_prefix_decode,
}
