"""Independent brute force for tiny inputs (pure Python loops over NumPy scalars).

TEST INFRASTRUCTURE ONLY. It restates the same definition as ``oracle.c``
without sharing any of its code: the KV write walks each token's slot into
(physical block, offset); attention gathers the sequence's keys position by
position through the block table ("C13 L2 serving" page, K_r = gather(K_pool,
table_r)) and applies softmax over keys 0..P, P the row's absolute position
("Chunked Prefill" glossary page, causal over absolute positions).
"""
from __future__ import annotations

import math

import numpy as np


def widen(a: np.ndarray) -> np.ndarray:
    """float32 arrays pass through; uint16 arrays are bf16 bit patterns."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def reshape_and_cache(k_pool: np.ndarray, v_pool: np.ndarray, k_new: np.ndarray,
                      v_new: np.ndarray, slot_mapping) -> None:
    b = k_pool.shape[1]
    for t, slot in enumerate(slot_mapping):
        slot = int(slot)
        if slot < 0:
            continue
        blk, off = divmod(slot, b)
        k_pool[blk, off] = k_new[t]
        v_pool[blk, off] = v_new[t]


def paged_attention(q, k_pool, v_pool, cu_q_lens, context_lens, block_tables, scale):
    q = widen(np.asarray(q))
    K = widen(np.asarray(k_pool))
    V = widen(np.asarray(v_pool))
    T, Hq, d = q.shape
    b, Hkv = K.shape[1], K.shape[2]
    G = Hq // Hkv
    out = np.zeros((T, Hq, d))
    cu = [int(x) for x in cu_q_lens]
    for s in range(len(context_lens)):
        ctx = int(context_lens[s])
        q_len = cu[s + 1] - cu[s]
        for i in range(q_len):
            t = cu[s] + i
            P = ctx - q_len + i
            for h in range(Hq):
                g = h // G
                keys = []
                vals = []
                for p in range(P + 1):
                    blk = int(block_tables[s][p // b])
                    keys.append(K[blk, p % b, g])
                    vals.append(V[blk, p % b, g])
                xs = [scale * sum(q[t, h, k] * key[k] for k in range(d)) for key in keys]
                m = max(xs)
                ws = [math.exp(x - m) for x in xs]
                tot = sum(ws)
                for k in range(d):
                    out[t, h, k] = sum(w * v[k] for w, v in zip(ws, vals)) / tot
    return out
