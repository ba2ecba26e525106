"""The two-level cascade's work partition and partial-slot scheme, checked on
the host over many random batches (no GPU).

The decode kernel walks the blocks of all sequences in order, cut into equal
contiguous CTA ranges; a sibling group is walked in entries of up to M = 16/G
consecutive members, an entry's blocks being its shared blocks (through its
first member) and then each member's own. Member m of entry (first member a)
writes its partial of CTA c to slot a + c_f M + m n_c + (c - c_f), where the
entry's blocks lie in CTAs c_f .. c_f + n_c - 1; without sibling groups this
is c + s. This model restates that scheme and checks the properties the
kernel relies on: every block is walked exactly once by one CTA, every
partial has a slot of its own below num_seqs + M x CTAs (the workspace size),
and the merge's slot for (member, CTA) is the one the walk wrote.
"""
import numpy as np
import pytest


def upper_index(prefix, n, x):
    lo, hi = 0, n - 1
    while lo < hi:
        mid = (lo + hi + 1) >> 1
        if prefix[mid] <= x:
            lo = mid
        else:
            hi = mid - 1
    return lo


def cta_of_block(b, B, grid):
    return ((b + 1) * grid - 1) // B


def walk(blocks, cu_sib, M, grid):
    """blocks[s]: the blocks the kernel reads for s (its own, plus the shared
    ones when s is an entry's first member). Returns {slot: (cta, seq)} and
    the walked blocks."""
    S = len(blocks)
    prefix = np.concatenate([[0], np.cumsum(blocks)]).tolist()
    B = prefix[-1]
    entry = {}
    for j in range(len(cu_sib) - 1):
        for a in range(cu_sib[j], cu_sib[j + 1], M):
            k = min(M, cu_sib[j + 1] - a)
            for m in range(k):
                entry[a + m] = (a, k)
    written, seen = {}, []
    for c in range(grid):
        lo, hi = c * B // grid, (c + 1) * B // grid
        u, s = 0, upper_index(prefix, S, lo)
        while u < hi - lo:
            while prefix[s + 1] <= lo + u:
                s += 1
            a, k = entry.get(s, (s, 1))
            e_lo, e_hi = prefix[a], prefix[a + k]
            n = min(hi, e_hi) - lo - u
            assert n >= 1 and e_lo <= lo + u < e_hi
            seen += range(lo + u, lo + u + n)
            u += n
            c_f = cta_of_block(e_lo, B, grid)
            n_c = cta_of_block(e_hi - 1, B, grid) - c_f + 1
            for m in range(k):
                slot = a + c_f * M + m * n_c + (c - c_f)
                assert 0 <= slot < S + M * grid
                assert slot not in written, (slot, written[slot], (c, a + m))
                written[slot] = (c, a + m)
    return written, seen, prefix, entry


def merge_slots(s, prefix, entry, M, grid):
    a, k = entry.get(s, (s, 1))
    B = prefix[-1]
    a0, a1 = prefix[a], prefix[a + k]
    if a1 <= a0:
        return {}
    cf, cl = cta_of_block(a0, B, grid), cta_of_block(a1 - 1, B, grid)
    slot0 = a + cf * M + (s - a) * (cl - cf + 1) - cf
    return {c: slot0 + c for c in range(cf, cl + 1) if c * B // grid != (c + 1) * B // grid}


@pytest.mark.parametrize("seed", range(40))
def test_partition_and_slots(seed):
    rng = np.random.default_rng(seed)
    G = int(rng.choice([1, 2, 4, 8]))
    M = 16 // G
    S = int(rng.integers(1, 120))
    # sibling groups of random sizes over a random prefix of the batch
    cut = sorted(set(rng.integers(0, S + 1, size=int(rng.integers(0, 12))).tolist()) | {0})
    cu_sib = cut if len(cut) > 1 else []
    blocks = rng.integers(0, 9, size=S)  # own blocks (0: all shared, or a bad member)
    entry_first = set()
    for j in range(len(cu_sib) - 1):
        entry_first.update(range(cu_sib[j], cu_sib[j + 1], M))
    for a in entry_first:
        blocks[a] += int(rng.integers(0, 7))  # the entry's shared blocks
    if blocks.sum() == 0:
        blocks[0] = 1
    grid = int(rng.choice([1, 2, 7, 40, 152, 500]))
    written, seen, prefix, entry = walk(blocks.tolist(), cu_sib, M if cu_sib else 1, grid)
    assert sorted(seen) == list(range(prefix[-1]))
    Mw = M if cu_sib else 1
    for s in range(S):
        for c, slot in merge_slots(s, prefix, entry, Mw, grid).items():
            assert written[slot] == (c, s)


def test_plain_slots_are_cta_plus_sequence():
    blocks = [3, 0, 5, 2, 9, 1]
    written, _, _, _ = walk(blocks, [], 1, 7)
    assert all(slot == c + s for slot, (c, s) in written.items())
