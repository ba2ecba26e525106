"""Plain reference of prefix caching by page (test infrastructure only).

TEST INFRASTRUCTURE ONLY: imported by the tests, never by the library path,
and sharing no code with it.

"Inference engine core techniques", section 3.2 (prefix cache): a prompt is
split into pages, each page's tokens are hashed, a hash found in the table
means the page's KV is already in the pool, so the physical page is shared
(its reference count grows) and only the pages that miss are prefilled.

Two pieces, written from their definitions:

* ``fnv1a64`` -- the 64-bit FNV-1a hash (offset basis 14695981039346656037,
  prime 1099511628211; for each byte: xor, then multiply modulo 2**64), and
  ``page_key``, the chain key of one page: FNV-1a over the 8 little-endian
  bytes of the previous page's key and the page's token ids as 4-byte
  little-endian integers (key 0 before the first page). A chain key names the
  whole prefix, which is the plainest reading of "hash the prompt's prefix,
  page by page".
* ``ExactPrefixCache`` -- the hit rule on exact token prefixes, with no
  hashing at all: page j of a prompt hits when the exact token prefix
  ``prompt[: 16 * (j + 1)]`` was cached before and pages 0 .. j-1 hit too.
  At most ``(n - 1) // 16`` pages hit, so one token is always left to
  compute. Nothing is evicted (the tests that use it give the pool room).
"""
from __future__ import annotations

from typing import Dict, Sequence, Tuple

PAGE = 16
_FNV_OFFSET = 14695981039346656037
_FNV_PRIME = 1099511628211
_MASK = (1 << 64) - 1


def fnv1a64(data: bytes) -> int:
    h = _FNV_OFFSET
    for byte in data:
        h ^= byte
        h = (h * _FNV_PRIME) & _MASK
    return h


def page_key(parent: int, tokens: Sequence[int]) -> int:
    data = int(parent).to_bytes(8, "little")
    for t in tokens:
        data += (int(t) & 0xFFFFFFFF).to_bytes(4, "little")
    return fnv1a64(data)


def chain_keys(tokens: Sequence[int]) -> list:
    """Keys of every full page of ``tokens``."""
    keys, parent = [], 0
    for j in range(len(tokens) // PAGE):
        parent = page_key(parent, tokens[PAGE * j: PAGE * (j + 1)])
        keys.append(parent)
    return keys


class ExactPrefixCache:
    """Which pages of a prompt a prefix cache shares, by exact prefixes."""

    def __init__(self) -> None:
        self.prefixes: Dict[Tuple[int, ...], bool] = {}

    def hit_tokens(self, prompt: Sequence[int]) -> int:
        n = len(prompt)
        pages = 0
        for j in range((n - 1) // PAGE if n > 0 else 0):
            if tuple(prompt[: PAGE * (j + 1)]) not in self.prefixes:
                break
            pages = j + 1
        return pages * PAGE

    def add(self, tokens: Sequence[int]) -> None:
        """Cache every full page of ``tokens`` (all written to the pool)."""
        for j in range(len(tokens) // PAGE):
            self.prefixes[tuple(tokens[: PAGE * (j + 1)])] = True
