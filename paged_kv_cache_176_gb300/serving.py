"""Block manager, scheduler and a serving loop over libpa (include/pa_serving.h).

``BlockManager`` and ``Scheduler`` are ctypes bindings of the native C++
objects (argument marshalling only). ``ServingLoop`` drives them: every step
it asks the scheduler for a batch (decode tokens first, then prefill chunks
under the token budget), copies the plan to the device, runs the step's KV
write (fused with its copy-on-write copies when the step has any) and one
``pa_mixed_step`` over the paged pool, then commits the step. There is no model: the
new tokens' q/k/v are seeded random values, which is all the attention path
needs.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import numpy as np
import torch

from . import abi

PA_ENOSPACE = -6


class _Plan(ctypes.Structure):
    _fields_ = [
        ("max_seqs", ctypes.c_int), ("max_tokens", ctypes.c_int),
        ("max_blocks_per_seq", ctypes.c_int), ("max_cow", ctypes.c_int),
        ("num_seqs", ctypes.c_int), ("num_tokens", ctypes.c_int),
        ("num_decode", ctypes.c_int), ("num_cow", ctypes.c_int),
        ("table_stride", ctypes.c_int),
        ("seq_ids", ctypes.c_void_p), ("cu_q_lens", ctypes.c_void_p),
        ("context_lens", ctypes.c_void_p), ("block_tables", ctypes.c_void_p),
        ("slot_mapping", ctypes.c_void_p), ("cow_src", ctypes.c_void_p),
        ("cow_dst", ctypes.c_void_p), ("cow_ntok", ctypes.c_void_p),
        ("token_ids", ctypes.c_void_p),
    ]


_ready = False


def _lib() -> ctypes.CDLL:
    global _ready
    lib = abi.load()
    if not _ready:
        P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        lib.pa_bm_create.restype = P
        lib.pa_bm_create.argtypes = [I64, I]
        lib.pa_bm_destroy.restype = None
        lib.pa_bm_destroy.argtypes = [P]
        lib.pa_bm_num_free.restype = I64
        lib.pa_bm_num_free.argtypes = [P]
        lib.pa_bm_add.restype = I
        lib.pa_bm_add.argtypes = [P, I64]
        lib.pa_bm_fork.restype = I
        lib.pa_bm_fork.argtypes = [P, I64, I64]
        lib.pa_bm_append.restype = I
        lib.pa_bm_append.argtypes = [P, I64, I, P, P, P, P, P]
        lib.pa_bm_beam_step.restype = I
        lib.pa_bm_beam_step.argtypes = [P, I, P, I, P, P]
        lib.pa_page_hash.restype = ctypes.c_uint64
        lib.pa_page_hash.argtypes = [ctypes.c_uint64, P, I]
        lib.pa_bm_set_prefix_cache.restype = I
        lib.pa_bm_set_prefix_cache.argtypes = [P, I]
        lib.pa_bm_num_cached.restype = I64
        lib.pa_bm_num_cached.argtypes = [P]
        lib.pa_bm_add_cached.restype = I
        lib.pa_bm_add_cached.argtypes = [P, I64, P, I64, P]
        lib.pa_bm_cache_pages.restype = I
        lib.pa_bm_cache_pages.argtypes = [P, I64, P, I64]
        lib.pa_sched_submit_tokens.restype = I
        lib.pa_sched_submit_tokens.argtypes = [P, I64, P, I, I]
        lib.pa_sched_commit_tokens.restype = I
        lib.pa_sched_commit_tokens.argtypes = [P, P]
        lib.pa_sched_cached_tokens.restype = I64
        lib.pa_sched_cached_tokens.argtypes = [P]
        lib.pa_bm_free.restype = I
        lib.pa_bm_free.argtypes = [P, I64]
        lib.pa_bm_num_tokens.restype = I64
        lib.pa_bm_num_tokens.argtypes = [P, I64]
        lib.pa_bm_block_table.restype = I
        lib.pa_bm_block_table.argtypes = [P, I64, P, I]
        lib.pa_bm_refcount.restype = I
        lib.pa_bm_refcount.argtypes = [P, ctypes.c_int32]
        lib.pa_bm_shared_prefix.restype = ctypes.c_int64
        lib.pa_bm_shared_prefix.argtypes = [P, P, I]
        lib.pa_sched_create.restype = P
        lib.pa_sched_create.argtypes = [P, I, I, I]
        lib.pa_sched_destroy.restype = None
        lib.pa_sched_destroy.argtypes = [P]
        lib.pa_sched_submit.restype = I
        lib.pa_sched_submit.argtypes = [P, I64, I, I]
        lib.pa_sched_step.restype = I
        lib.pa_sched_step.argtypes = [P, ctypes.POINTER(_Plan)]
        lib.pa_sched_commit.restype = I
        lib.pa_sched_commit.argtypes = [P]
        lib.pa_sched_stats.restype = I
        lib.pa_sched_stats.argtypes = [P, P, P, P, P, P]
        lib.pa_copy_blocks.restype = I
        lib.pa_copy_blocks.argtypes = [ctypes.POINTER(abi.pa_kv_pool), P, P, I, P, P]
        lib.pa_reshape_and_cache_cow.restype = I
        lib.pa_reshape_and_cache_cow.argtypes = [ctypes.POINTER(abi.pa_kv_pool), P, P, P, I, P, P,
                                                 P, I, P, P]
        _ready = True
    return lib


def _np_ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def pa_page_hash(parent_key: int, tokens) -> int:
    """Chain key of one page (see include/pa_serving.h)."""
    t = _i32(tokens)
    return int(_lib().pa_page_hash(parent_key, _np_ptr(t), t.size))


class BlockManager:
    """Pool of ``num_blocks`` blocks of ``block_size`` tokens (native)."""

    def __init__(self, num_blocks: int, block_size: int = 16):
        self._lib = _lib()
        self.block_size = block_size
        self.num_blocks = num_blocks
        self._h = self._lib.pa_bm_create(num_blocks, block_size)
        if not self._h:
            raise ValueError("bad block manager sizes")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._lib.pa_bm_destroy(h)
            self._h = None

    @property
    def num_free(self) -> int:
        return int(self._lib.pa_bm_num_free(self._h))

    def add(self, seq: int) -> None:
        abi._check("pa_bm_add", self._lib.pa_bm_add(self._h, seq))

    def fork(self, parent: int, child: int) -> None:
        abi._check("pa_bm_fork", self._lib.pa_bm_fork(self._h, parent, child))

    def append(self, seq: int, n: int):
        """Slots of n new tokens and the copy-on-write pairs
        [(src, dst, filled slots to copy)]."""
        slots = np.empty(max(n, 1), dtype=np.int64)
        src = np.empty(1, dtype=np.int32)
        dst = np.empty(1, dtype=np.int32)
        ntok = np.empty(1, dtype=np.int32)
        n_cow = ctypes.c_int(0)
        rc = self._lib.pa_bm_append(self._h, seq, n, _np_ptr(slots), _np_ptr(src), _np_ptr(dst),
                                    _np_ptr(ntok), ctypes.byref(n_cow))
        abi._check("pa_bm_append", rc)
        cow = [(int(src[0]), int(dst[0]), int(ntok[0]))] if n_cow.value else []
        return slots[:n], cow

    def beam_step(self, old_ids, parents, new_ids) -> None:
        """New beam i continues old beam old_ids[parents[i]] (shared blocks);
        the old beams are released."""
        old = np.ascontiguousarray(old_ids, dtype=np.int64)
        par = np.ascontiguousarray(parents, dtype=np.int32)
        new = np.ascontiguousarray(new_ids, dtype=np.int64)
        if par.size != new.size:
            raise ValueError("one parent per new beam")
        abi._check("pa_bm_beam_step", self._lib.pa_bm_beam_step(
            self._h, old.size, _np_ptr(old), new.size, _np_ptr(par), _np_ptr(new)))

    def free(self, seq: int) -> None:
        abi._check("pa_bm_free", self._lib.pa_bm_free(self._h, seq))

    def num_tokens(self, seq: int) -> int:
        return int(self._lib.pa_bm_num_tokens(self._h, seq))

    def block_table(self, seq: int, max_blocks: int = 1 << 16) -> np.ndarray:
        out = np.empty(max_blocks, dtype=np.int32)
        n = self._lib.pa_bm_block_table(self._h, seq, _np_ptr(out), max_blocks)
        if n < 0:
            raise abi.PagedAttentionError("pa_bm_block_table", n)
        return out[:n].copy()

    def shared_prefix(self, seqs) -> int:
        """Tokens the sequences share as a sibling group (whole pages that are
        the same physical blocks in every table, within every context)."""
        ids = np.ascontiguousarray(np.asarray(seqs, dtype=np.int64))
        n = int(self._lib.pa_bm_shared_prefix(self._h, _np_ptr(ids), int(ids.size)))
        if n < 0:
            abi._check("pa_bm_shared_prefix", n)
        return n

    def refcount(self, block: int) -> int:
        return int(self._lib.pa_bm_refcount(self._h, block))

    def set_prefix_cache(self, enable: bool) -> None:
        abi._check("pa_bm_set_prefix_cache", self._lib.pa_bm_set_prefix_cache(self._h, int(enable)))

    @property
    def num_cached(self) -> int:
        return int(self._lib.pa_bm_num_cached(self._h))

    def add_cached(self, seq: int, tokens) -> int:
        """Register seq with prompt ``tokens``; returns the tokens shared from
        the prefix cache."""
        t = _i32(tokens)
        hit = ctypes.c_int64(0)
        abi._check("pa_bm_add_cached", self._lib.pa_bm_add_cached(self._h, seq, _np_ptr(t), t.size,
                                                                   ctypes.byref(hit)))
        return int(hit.value)

    def cache_pages(self, seq: int, tokens) -> None:
        t = _i32(tokens)
        abi._check("pa_bm_cache_pages", self._lib.pa_bm_cache_pages(self._h, seq, _np_ptr(t), t.size))


class StepPlan:
    """Host buffers of one scheduler step (see pa_step_plan)."""

    def __init__(self, max_seqs: int, max_tokens: int, max_blocks_per_seq: int, max_cow: int = 64):
        self.seq_ids = np.zeros(max_seqs, dtype=np.int64)
        self.cu_q_lens = np.zeros(max_seqs + 1, dtype=np.int32)
        self.context_lens = np.zeros(max_seqs, dtype=np.int32)
        self.block_tables = np.full(max_seqs * max_blocks_per_seq, -1, dtype=np.int32)
        self.slot_mapping = np.zeros(max_tokens, dtype=np.int64)
        self.cow_src = np.zeros(max_cow, dtype=np.int32)
        self.cow_dst = np.zeros(max_cow, dtype=np.int32)
        self.cow_ntok = np.zeros(max_cow, dtype=np.int32)
        self.token_ids = np.full(max_tokens, -1, dtype=np.int32)
        self.c = _Plan(max_seqs, max_tokens, max_blocks_per_seq, max_cow, 0, 0, 0, 0, 0,
                       _np_ptr(self.seq_ids).value, _np_ptr(self.cu_q_lens).value,
                       _np_ptr(self.context_lens).value, _np_ptr(self.block_tables).value,
                       _np_ptr(self.slot_mapping).value, _np_ptr(self.cow_src).value,
                       _np_ptr(self.cow_dst).value, _np_ptr(self.cow_ntok).value,
                       _np_ptr(self.token_ids).value)

    @property
    def num_seqs(self) -> int:
        return self.c.num_seqs

    @property
    def num_tokens(self) -> int:
        return self.c.num_tokens

    @property
    def num_decode(self) -> int:
        return self.c.num_decode

    @property
    def num_cow(self) -> int:
        return self.c.num_cow

    @property
    def table_stride(self) -> int:
        return self.c.table_stride

    @property
    def tables(self) -> np.ndarray:
        """This step's block tables, [num_seqs, table_stride] (-1 padded)."""
        S, W = self.num_seqs, self.table_stride
        return self.block_tables[:S * W].reshape(S, W)


class Scheduler:
    """Iteration-level scheduler with chunked prefill (native)."""

    def __init__(self, bm: BlockManager, token_budget: int, chunk_size: int, max_running: int):
        self._lib = _lib()
        self.bm = bm  # keep the block manager alive
        self.token_budget = token_budget
        self._h = self._lib.pa_sched_create(bm._h, token_budget, chunk_size, max_running)
        if not self._h:
            raise ValueError("bad scheduler arguments")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._lib.pa_sched_destroy(h)
            self._h = None

    def submit(self, req_id: int, prompt_len: int, max_new_tokens: int, tokens=None) -> None:
        """Queue a request; with ``tokens`` (the prompt's ids) it goes
        through the prefix cache and its generated tokens must be committed."""
        if tokens is None:
            rc = self._lib.pa_sched_submit(self._h, req_id, prompt_len, max_new_tokens)
        else:
            t = _i32(tokens)
            if t.size != prompt_len:
                raise ValueError("tokens must hold prompt_len ids")
            rc = self._lib.pa_sched_submit_tokens(self._h, req_id, _np_ptr(t), prompt_len,
                                                  max_new_tokens)
        abi._check("pa_sched_submit", rc)

    def step(self, plan: StepPlan) -> StepPlan:
        abi._check("pa_sched_step", self._lib.pa_sched_step(self._h, ctypes.byref(plan.c)))
        return plan

    def commit(self, next_tokens=None) -> None:
        """Commit the planned step; ``next_tokens[j]`` is the token plan row j
        generated (needed when the step holds token-mode requests)."""
        if next_tokens is None:
            rc = self._lib.pa_sched_commit(self._h)
        else:
            t = _i32(next_tokens)
            rc = self._lib.pa_sched_commit_tokens(self._h, _np_ptr(t))
        abi._check("pa_sched_commit", rc)

    @property
    def cached_tokens(self) -> int:
        return int(self._lib.pa_sched_cached_tokens(self._h))

    def stats(self) -> dict:
        v = [ctypes.c_int64(0) for _ in range(5)]
        abi._check("pa_sched_stats", self._lib.pa_sched_stats(self._h, *[ctypes.byref(x) for x in v]))
        keys = ("waiting", "running", "finished", "prefill_tokens", "decode_tokens")
        return {k: int(x.value) for k, x in zip(keys, v)}


def sibling_shared_tokens(tables, context_lens, block_size: int = 16) -> int:
    """Tokens a group of sequences (a request's beams or sampled replies) can
    share in pa_decode_cascade_nested: the leading block-table entries equal
    in every row (the same physical blocks, so the same cache contents),
    whole pages only, each within every member's context."""
    t = np.asarray(tables)
    c = np.asarray(context_lens)
    if t.shape[0] == 0:
        return 0
    lim = min(int(c.min()) // block_size, t.shape[1])
    eq = np.all(t[:, :lim] == t[0, :lim], axis=0)
    n = lim if bool(eq.all()) else int(np.argmin(eq))
    return n * block_size


def pa_reshape_and_cache_cow(k_pool, v_pool, k_new, v_new, slot_mapping, cow_src, cow_dst,
                             cow_ntok, d_status=None, stream=None) -> None:
    """KV write of the step's tokens with the copy-on-write copies (the filled
    slots of shared blocks) fused into the same launch."""
    lib = _lib()
    pool = abi.make_pool(k_pool, v_pool)
    T = 0 if slot_mapping is None else int(slot_mapping.numel())
    n = 0 if cow_src is None else int(cow_src.numel())
    abi._check("pa_reshape_and_cache_cow",
               lib.pa_reshape_and_cache_cow(ctypes.byref(pool), abi._ptr(k_new), abi._ptr(v_new),
                                            abi._ptr(slot_mapping), T, abi._ptr(cow_src),
                                            abi._ptr(cow_dst), abi._ptr(cow_ntok), n,
                                            abi._ptr(d_status), abi._stream(stream)))


def pa_copy_blocks(k_pool, v_pool, src: torch.Tensor, dst: torch.Tensor, d_status=None,
                   stream=None) -> None:
    """Device copy of whole K/V blocks src[i] -> dst[i] (copy-on-write)."""
    lib = _lib()
    pool = abi.make_pool(k_pool, v_pool)
    n = int(src.numel())
    abi._check("pa_copy_blocks", lib.pa_copy_blocks(ctypes.byref(pool), abi._ptr(src),
                                                    abi._ptr(dst), n, abi._ptr(d_status),
                                                    abi._stream(stream)))


def _align16(n: int) -> int:
    return (n + 15) & ~15


class ServingLoop:
    """Continuous batching with chunked prefill over one layer's paged pool.

    Each step's plan (slot mapping, cu_q_lens, context lengths, copy-on-write
    pairs and the packed block tables) is packed into one of two pinned host
    buffers and sent with a single asynchronous copy on ``stream``; the host
    then plans the next step while the device runs this one. A pinned buffer
    is refilled only after the copy that read it has finished.

    With ``fresh_inputs`` the step's q/k/v are redrawn on the device every
    step; otherwise the buffers keep the values drawn at construction (the
    kernels' work does not depend on the values).

    With ``vocab`` the loop runs on token ids: requests carry their prompt's
    ids, a token's q/k/v are rows of seeded per-token tables (so the same
    prefix always yields the same cache contents, which is what makes a
    shared cached page correct), each generated token is a fixed function of
    the sequence id and position, and ``prefix_cache`` turns on the block
    manager's prefix cache.
    """

    def __init__(self, num_blocks: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                 dtype=torch.bfloat16, token_budget: int = 2048, chunk_size: int = 512,
                 max_running: int = 256, max_context: int = 32768, device="cuda", seed: int = 0,
                 stream: Optional[torch.cuda.Stream] = None, fresh_inputs: bool = True,
                 max_cow: int = 64, vocab: Optional[int] = None, prefix_cache: bool = False):
        self.bm = BlockManager(num_blocks, 16)
        if prefix_cache:
            if vocab is None:
                raise ValueError("the prefix cache needs token ids (vocab)")
            self.bm.set_prefix_cache(True)
        self.sched = Scheduler(self.bm, token_budget, chunk_size, max_running)
        self.vocab = vocab
        self.hq, self.hkv, self.d, self.dtype = num_q_heads, num_kv_heads, head_dim, dtype
        self.budget = token_budget
        self.device = torch.device(device)
        self.stream = stream or torch.cuda.current_stream(self.device)
        self.fresh_inputs = fresh_inputs
        mb = (max_context + 15) // 16
        self.max_blocks = mb
        T, S = token_budget, max_running
        self.plan = StepPlan(S, T, mb, max_cow)
        self.k_pool = torch.full((num_blocks, 16, num_kv_heads, head_dim), float("nan"), dtype=dtype,
                                 device=self.device)
        self.v_pool = torch.full_like(self.k_pool, float("nan"))
        self.q = torch.empty(T, num_q_heads, head_dim, dtype=dtype, device=self.device)
        self.k_new = torch.empty(T, num_kv_heads, head_dim, dtype=dtype, device=self.device)
        self.v_new = torch.empty_like(self.k_new)
        self.out = torch.empty_like(self.q)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        # packed plan: slots (int64) | cu (S+1) | ctx (S) | cow src | dst | ntok |
        # token ids (T) | tables
        self._cap = (_align16(8 * T) + _align16(4 * (S + 1)) + _align16(4 * S) +
                     3 * _align16(4 * max_cow) + _align16(4 * T) + _align16(4 * S * mb))
        self._dev = torch.empty(self._cap, dtype=torch.uint8, device=self.device)
        self._host = [torch.empty(self._cap, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
        self._host_np = [h.numpy() for h in self._host]
        self._sent = [None, None]
        self._k = 0
        self.h2d_bytes = 0
        self.ws = torch.empty(abi.pa_mixed_workspace_size(S, T, num_q_heads, head_dim, mb),
                              dtype=torch.uint8, device=self.device)
        self.gen = torch.Generator(device=self.device)
        self.gen.manual_seed(seed)
        with torch.cuda.stream(self.stream):
            if vocab is None:
                self._draw(T)
            else:
                def table(h):
                    return torch.randn(vocab, h, head_dim, generator=self.gen, device=self.device,
                                       dtype=torch.float32).to(dtype)
                self.emb_q, self.emb_k, self.emb_v = table(num_q_heads), table(num_kv_heads), \
                    table(num_kv_heads)
        self.scale = head_dim ** -0.5
        self.steps = 0
        self.prompt_len = {}
        self.first_token_step = {}  # request id -> step that yielded its first token

    def _draw(self, T: int) -> None:
        for t in (self.q[:T], self.k_new[:T], self.v_new[:T]):
            t.copy_(torch.randn(t.shape, generator=self.gen, device=self.device, dtype=torch.float32))

    def submit(self, req_id: int, prompt_len: int, max_new_tokens: int, tokens=None) -> None:
        if (tokens is None) != (self.vocab is None):
            raise ValueError("token ids go with a loop built with vocab, and only with it")
        self.sched.submit(req_id, prompt_len, max_new_tokens, tokens)
        self.prompt_len[req_id] = prompt_len

    def next_tokens(self, p: StepPlan) -> np.ndarray:
        """The token each plan row generates: a fixed function of the
        sequence id and the new token's position (a stand-in sampler)."""
        S = p.num_seqs
        x = (p.seq_ids[:S].astype(np.uint64) * np.uint64(0x9E3779B97F4A7C15)
             + p.context_lens[:S].astype(np.uint64) * np.uint64(0xBF58476D1CE4E5B9))
        x ^= x >> np.uint64(31)
        return (x % np.uint64(self.vocab)).astype(np.int32)

    def _pack(self, p: StepPlan):
        """Pack the plan into the free pinned buffer; returns the byte offsets."""
        S, T, C, W = p.num_seqs, p.num_tokens, p.num_cow, p.table_stride
        k = self._k
        if self._sent[k] is not None:
            self._sent[k].synchronize()  # the copy that read this buffer is done
        buf = self._host_np[k]
        offs = {}
        o = 0
        for name, src, dt in (("slots", p.slot_mapping[:T], np.int64),
                              ("cu", p.cu_q_lens[:S + 1], np.int32),
                              ("ctx", p.context_lens[:S], np.int32),
                              ("src", p.cow_src[:C], np.int32),
                              ("dst", p.cow_dst[:C], np.int32),
                              ("ntok", p.cow_ntok[:C], np.int32),
                              ("ids", p.token_ids[:T] if self.vocab else p.token_ids[:0], np.int32),
                              ("bt", p.block_tables[:S * W], np.int32)):
            n = src.size * np.dtype(dt).itemsize
            buf[o:o + n].view(dt)[:] = src
            offs[name] = (o, src.size)
            o = _align16(o + n)
        return k, o, offs

    def _view(self, offs, name, dtype):
        o, n = offs[name]
        size = torch.tensor([], dtype=dtype).element_size()
        return self._dev[o:o + n * size].view(dtype)

    def step(self) -> Optional[StepPlan]:
        """Enqueue one step on ``stream``; returns its plan (host arrays), or
        None when every request has finished. The host does not wait for the
        device, except to reuse a pinned buffer."""
        p = self.sched.step(self.plan)
        S, T, C = p.num_seqs, p.num_tokens, p.num_cow
        if S == 0:
            return None
        k, nbytes, offs = self._pack(p)
        with torch.cuda.stream(self.stream):
            if self.vocab is None and self.fresh_inputs:
                self._draw(T)
            self._dev[:nbytes].copy_(self._host[k][:nbytes], non_blocking=True)
            if self.vocab is not None:
                ids = self._view(offs, "ids", torch.int32)
                torch.index_select(self.emb_q, 0, ids, out=self.q[:T])
                torch.index_select(self.emb_k, 0, ids, out=self.k_new[:T])
                torch.index_select(self.emb_v, 0, ids, out=self.v_new[:T])
            ev = torch.cuda.Event()
            ev.record(self.stream)
            self._sent[k] = ev
            self._k ^= 1
            self.h2d_bytes += nbytes
            slots = self._view(offs, "slots", torch.int64)
            bt = self._view(offs, "bt", torch.int32).view(S, p.table_stride)
            if C:
                # copy-on-write copies fused with the step's KV write
                pa_reshape_and_cache_cow(self.k_pool, self.v_pool, self.k_new[:T], self.v_new[:T],
                                         slots, self._view(offs, "src", torch.int32),
                                         self._view(offs, "dst", torch.int32),
                                         self._view(offs, "ntok", torch.int32),
                                         d_status=self.status, stream=self.stream)
            write = C == 0  # otherwise already written above
            abi.pa_mixed_step(self.out[:T], self.q[:T], self._view(offs, "cu", torch.int32),
                              self._view(offs, "ctx", torch.int32), bt, self.k_pool, self.v_pool,
                              self.scale, self.budget,
                              k_new=self.k_new[:T] if write else None,
                              v_new=self.v_new[:T] if write else None,
                              slot_mapping=slots if write else None,
                              workspace=self.ws, d_status=self.status, stream=self.stream)
        self.sched.commit(self.next_tokens(p) if self.vocab is not None else None)
        for j in range(p.num_decode, S):  # prefill chunks that finish their prompt
            sid = int(p.seq_ids[j])
            if int(p.context_lens[j]) == self.prompt_len.get(sid, -1):
                self.first_token_step[sid] = self.steps
        self.steps += 1
        return p
