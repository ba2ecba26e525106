"""fp64 CPU oracle for attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY. Only the tests, the package's smoke check and the
benchmark's CPU-baseline / reference leg may import this package. The library
path never does, and this package never imports the library's package: the two
share no code.

``oracle.c`` (built here into ``liboracle.so`` with gcc) is the oracle proper;
``brute.py`` is an independent pure-Python/NumPy brute force for tiny inputs.
See ``oracle.h`` for what each function computes and which passage it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32 = 0
BF16 = 1


def build(src: str = _SRC, out: str = _LIB_PATH, force: bool = False) -> str:
    """Compile ``src`` with gcc into the shared library ``out``."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)
            and os.path.getmtime(out) >= os.path.getmtime(os.path.join(os.path.dirname(src), "oracle.h"))):
        return out
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-fPIC", "-shared", "-pthread",
           "-I", os.path.dirname(src), "-o", out + ".tmp", src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def _setup(lib: ctypes.CDLL) -> ctypes.CDLL:
    P = ctypes.c_void_p
    lib.oracle_reshape_and_cache.restype = ctypes.c_int
    lib.oracle_reshape_and_cache.argtypes = [P, P, ctypes.c_int64, ctypes.c_int, ctypes.c_int64,
                                             P, P, P, ctypes.c_int]
    lib.oracle_copy_blocks.restype = ctypes.c_int
    lib.oracle_copy_blocks.argtypes = [P, P, ctypes.c_int64, ctypes.c_int, ctypes.c_int64, P, P, P,
                                       ctypes.c_int]
    lib.oracle_paged_attention.restype = ctypes.c_int
    lib.oracle_paged_attention.argtypes = [P, P, P, P, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           P, P, P, ctypes.c_int, ctypes.c_double, P, ctypes.c_int]
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library. A ``path`` loads a
    specific build, e.g. a copy with a planted mistake."""
    global _lib
    if path is not None:
        return _setup(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            build()
            _lib = _setup(ctypes.CDLL(_LIB_PATH))
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _raw(x) -> np.ndarray:
    """A contiguous numpy view of a host tensor/array. bf16 tensors become
    their uint16 bit patterns."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().contiguous().cpu()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16)
            return x.numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x)


def dtype_code(x) -> int:
    import torch
    if isinstance(x, torch.Tensor):
        if x.dtype == torch.bfloat16:
            return BF16
        if x.dtype == torch.float32:
            return F32
        raise TypeError(f"unsupported dtype {x.dtype}")
    if x.dtype == np.float32:
        return F32
    if x.dtype == np.uint16:
        return BF16
    raise TypeError(f"unsupported dtype {x.dtype}")


def reshape_and_cache(k_pool, v_pool, k_new, v_new, slot_mapping, lib=None) -> None:
    """In-place KV write into host pools ``[N_blk, b, Hkv, d]``."""
    lib = lib or load()
    kp, vp = _raw(k_pool), _raw(v_pool)
    kn, vn = _raw(k_new), _raw(v_new)
    sm = np.ascontiguousarray(_raw(slot_mapping), dtype=np.int64)
    nb, b = kp.shape[0], kp.shape[1]
    token_bytes = int(np.prod(kp.shape[2:])) * kp.itemsize
    rc = lib.oracle_reshape_and_cache(_ptr(kp), _ptr(vp), nb, b, token_bytes, _ptr(kn), _ptr(vn),
                                      _ptr(sm), int(sm.shape[0]))
    if rc != 0:
        raise ValueError(f"oracle_reshape_and_cache failed with code {rc}")
    # write back for torch inputs that were copied by _raw
    for dst, src in ((k_pool, kp), (v_pool, vp)):
        _writeback(dst, src)


def _writeback(dst, src: np.ndarray) -> None:
    try:
        import torch
        if isinstance(dst, torch.Tensor):
            if dst.dtype == torch.bfloat16:
                view = dst.view(torch.int16).numpy().view(np.uint16)
            else:
                view = dst.numpy()
            if view.ctypes.data != src.ctypes.data:
                view[...] = src
    except ImportError:  # pragma: no cover
        pass


def copy_blocks(k_pool, v_pool, src, dst, ntok=None, lib=None) -> int:
    """In-place copy-on-write copy on host pools ``[N_blk, b, Hkv, d]``: pair i
    copies the first ``ntok[i]`` slots (whole blocks when ``ntok`` is None) of
    block ``src[i]`` onto block ``dst[i]``. Returns 0, or ORACLE_ERANGE (2)
    when a bad pair was skipped."""
    lib = lib or load()
    kp, vp = _raw(k_pool), _raw(v_pool)
    s = np.ascontiguousarray(_raw(src), dtype=np.int32)
    d = np.ascontiguousarray(_raw(dst), dtype=np.int32)
    n = None if ntok is None else np.ascontiguousarray(_raw(ntok), dtype=np.int32)
    nb, b = kp.shape[0], kp.shape[1]
    token_bytes = int(np.prod(kp.shape[2:])) * kp.itemsize
    rc = lib.oracle_copy_blocks(_ptr(kp), _ptr(vp), nb, b, token_bytes, _ptr(s), _ptr(d), _ptr(n),
                                int(s.shape[0]))
    if rc not in (0, 2):
        raise ValueError(f"oracle_copy_blocks failed with code {rc}")
    for dst_t, src_a in ((k_pool, kp), (v_pool, vp)):
        _writeback(dst_t, src_a)
    return int(rc)


def cow_write(k_pool, v_pool, k_new, v_new, slot_mapping, src, dst, ntok, lib=None) -> int:
    """The fused copy-on-write KV write on host pools: the copies first (the
    filled slots of each shared block onto its fresh copy), then the step's
    KV write into the copies and other blocks. Returns copy_blocks' code."""
    rc = copy_blocks(k_pool, v_pool, src, dst, ntok, lib=lib)
    if slot_mapping is not None and len(slot_mapping):
        reshape_and_cache(k_pool, v_pool, k_new, v_new, slot_mapping, lib=lib)
    return rc


def paged_attention(q, k_pool, v_pool, cu_q_lens, context_lens, block_tables, scale: float,
                    row_mask=None, num_threads: int | None = None, lib=None) -> np.ndarray:
    """fp64 attention output ``[T, Hq, d]`` for every query row of a batch.

    q ``[T, Hq, d]``; pools ``[N_blk, b, Hkv, d]``; cu_q_lens ``[S+1]``;
    context_lens ``[S]``; block_tables ``[S, max_blocks]``. Rows whose
    ``row_mask`` entry is 0 come back as NaN.
    """
    lib = lib or load()
    qa, kp, vp = _raw(q), _raw(k_pool), _raw(v_pool)
    dt = dtype_code(qa)
    if dtype_code(kp) != dt or dtype_code(vp) != dt:
        raise TypeError("q and pools must share a dtype")
    cu = np.ascontiguousarray(_raw(cu_q_lens), dtype=np.int32)
    cl = np.ascontiguousarray(_raw(context_lens), dtype=np.int32)
    bt = np.ascontiguousarray(_raw(block_tables), dtype=np.int32)
    T, Hq, d = qa.shape
    nb, b, hkv, d2 = kp.shape
    assert d2 == d and int(cu[-1]) == T
    out = np.full((T, Hq, d), np.nan, dtype=np.float64)
    mask = None if row_mask is None else np.ascontiguousarray(_raw(row_mask), dtype=np.uint8)
    nt = num_threads or os.cpu_count() or 1
    rc = lib.oracle_paged_attention(_ptr(out), _ptr(qa), _ptr(kp), _ptr(vp), dt, nb, b, hkv, d, Hq,
                                    int(cl.shape[0]), _ptr(cu), _ptr(cl), _ptr(bt), int(bt.shape[1]),
                                    float(scale), _ptr(mask), int(nt))
    if rc != 0:
        raise ValueError(f"oracle_paged_attention failed with code {rc}")
    return out


def workload_attention(w, row_mask=None, num_threads=None, lib=None) -> np.ndarray:
    """Oracle output for a ``Workload``: the step's KV write (if any) is
    applied to copies of the pools first, then attention is computed."""
    kp, vp = w.k_pool.clone(), w.v_pool.clone()
    if w.slot_mapping is not None:
        reshape_and_cache(kp, vp, w.k_new, w.v_new, w.slot_mapping, lib=lib)
    return paged_attention(w.q, kp, vp, w.cu_q_lens, w.context_lens, w.block_tables, w.scale,
                           row_mask=row_mask, num_threads=num_threads, lib=lib)
