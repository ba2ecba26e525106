"""ctypes binding of libpa (include/pa.h). Argument marshalling only.

Every function here has the name of the C entry point it calls and passes
PyTorch tensors' device pointers, sizes and the current CUDA stream through.
All computation happens in libpa's CUDA kernels; there is no fallback: if the
library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa.so")
PROBE_LIB_PATH = os.path.join(_HERE, "libpa_probe.so")

PA_OK = 0
PA_EINVAL = -1
PA_EUNSUPPORTED = -2
PA_EWORKSPACE = -3
PA_EBUDGET = -4
PA_ECUDA = -5
PA_F32 = 0
PA_BF16 = 1
PA_STATUS_BAD_BLOCK = 1
PA_STATUS_BAD_LENGTH = 2
PA_STATUS_BAD_SLOT = 4
PA_STATUS_TIMEOUT = 8


class pa_kv_pool(ctypes.Structure):
    _fields_ = [
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("num_blocks", ctypes.c_int64),
        ("block_size", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
    ]


class PagedAttentionError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status} ({pa_strerror(status)})")
        self.status = status


_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libpa.so (built by ``paged_kv_cache_176_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m paged_kv_cache_176_gb300.build`")
        lib = ctypes.CDLL(path)
        P, I, I64, SZ, F = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t,
                            ctypes.c_float)
        PP = ctypes.POINTER(pa_kv_pool)
        lib.pa_strerror.restype = ctypes.c_char_p
        lib.pa_strerror.argtypes = [I]
        lib.pa_version.restype = I
        lib.pa_version.argtypes = []
        lib.pa_reshape_and_cache.restype = I
        lib.pa_reshape_and_cache.argtypes = [PP, P, P, P, I, P, P]
        lib.pa_decode_workspace_size.restype = SZ
        lib.pa_decode_workspace_size.argtypes = [I, I, I, I]
        lib.pa_decode.restype = I
        lib.pa_decode.argtypes = [PP, P, P, I, I, P, I, P, F, P, SZ, P, P]
        lib.pa_mixed_workspace_size.restype = SZ
        lib.pa_mixed_workspace_size.argtypes = [I, I, I, I, I]
        lib.pa_mixed_step.restype = I
        lib.pa_mixed_step.argtypes = [PP, P, P, P, I, I, I, P, P, I, F, I, P, P, P, P, SZ, P, P]
        lib.pa_mixed_step_with_units.restype = I
        lib.pa_mixed_step_with_units.argtypes = [PP, P, P, P, I, I, I, P, P, I, F, I, P, P, P, I, P,
                                                 SZ, P, P]
        lib.pa_decode_with_ctas.restype = I
        lib.pa_decode_with_ctas.argtypes = [PP, P, P, I, I, P, I, P, F, I, P, SZ, P, P]
        lib.pa_decode_static_ws.restype = I
        lib.pa_decode_static_ws.argtypes = [PP, P, P, I, I, P, I, P, F, P, P]
        lib.pa_decode_cascade_workspace_size.restype = SZ
        lib.pa_decode_cascade_workspace_size.argtypes = [I, I, I, I]
        lib.pa_decode_cascade.restype = I
        lib.pa_decode_cascade.argtypes = [PP, P, P, I, I, P, I, P, P, P, I, F, P, SZ, P, P]
        lib.pa_decode_cascade_with_ctas.restype = I
        lib.pa_decode_cascade_with_ctas.argtypes = [PP, P, P, I, I, P, I, P, P, P, I, F, I, P, SZ, P,
                                                    P]
        lib.pa_decode_cascade_nested_workspace_size.restype = SZ
        lib.pa_decode_cascade_nested_workspace_size.argtypes = [I, I, I, I, I, I]
        lib.pa_decode_cascade_nested.restype = I
        lib.pa_decode_cascade_nested.argtypes = [PP, P, P, I, I, P, I, P, P, P, I, P, P, I, F, I,
                                                 P, SZ, P, P]
        _lib = lib
        return lib


_probe_lib: Optional[ctypes.CDLL] = None


def load_probe(path: str = PROBE_LIB_PATH) -> ctypes.CDLL:
    """Load libpa_probe.so, the measurement and test aids of include/pa_probe.h
    (built beside libpa.so; not part of the attention path)."""
    global _probe_lib
    with _lock:
        if _probe_lib is not None:
            return _probe_lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m paged_kv_cache_176_gb300.build`")
        lib = ctypes.CDLL(path)
        P, I, U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_ulonglong
        lib.pa_gather_probe.restype = I
        lib.pa_gather_probe.argtypes = [ctypes.POINTER(pa_kv_pool), P, I, I, I, P, P]
        lib.pa_wait_probe.restype = I
        lib.pa_wait_probe.argtypes = [P, I, U64, P, P]
        _probe_lib = lib
        return lib


def pa_strerror(status: int) -> str:
    return load().pa_strerror(int(status)).decode()


def pa_version() -> int:
    return int(load().pa_version())


# ----------------------------------------------------------------- helpers


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return PA_BF16
    if t.dtype == torch.float32:
        return PA_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libpa takes device tensors")
    if not t.is_contiguous():
        raise ValueError("libpa takes contiguous tensors")
    return t.data_ptr()


def make_pool(k_pool: torch.Tensor, v_pool: torch.Tensor) -> pa_kv_pool:
    if k_pool.shape != v_pool.shape or k_pool.dtype != v_pool.dtype or k_pool.dim() != 4:
        raise ValueError("k_pool/v_pool must both be [num_blocks, block_size, Hkv, d]")
    nb, b, hkv, d = k_pool.shape
    return pa_kv_pool(_ptr(k_pool), _ptr(v_pool), nb, b, hkv, d, _dtype_code(k_pool))


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(fn: str, rc: int) -> None:
    if rc != PA_OK:
        raise PagedAttentionError(fn, rc)


# ----------------------------------------------------------------- entry points


def pa_reshape_and_cache(k_pool, v_pool, k_new, v_new, slot_mapping, d_status=None,
                         stream=None) -> None:
    """KV write: scatter k_new/v_new [T, Hkv, d] into the pools at slot_mapping."""
    lib = load()
    pool = make_pool(k_pool, v_pool)
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    T = int(slot_mapping.shape[0])
    if T and (k_new.shape[0] != T or v_new.shape[0] != T):
        raise ValueError("k_new/v_new/slot_mapping disagree on num_tokens")
    _check("pa_reshape_and_cache",
           lib.pa_reshape_and_cache(ctypes.byref(pool), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
                                    T, _ptr(d_status), _stream(stream)))


def pa_decode_workspace_size(num_seqs: int, num_q_heads: int, head_dim: int,
                             max_blocks_per_seq: int) -> int:
    return int(load().pa_decode_workspace_size(num_seqs, num_q_heads, head_dim, max_blocks_per_seq))


def pa_mixed_workspace_size(num_seqs: int, num_tokens: int, num_q_heads: int, head_dim: int,
                            max_blocks_per_seq: int) -> int:
    return int(load().pa_mixed_workspace_size(num_seqs, num_tokens, num_q_heads, head_dim,
                                              max_blocks_per_seq))


def _workspace(nbytes: int, device, workspace) -> torch.Tensor:
    if workspace is not None:
        return workspace
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)


def pa_decode(out, q, k_pool, v_pool, block_tables, context_lens, scale: float, workspace=None,
              d_status=None, stream=None):
    """Decode attention, q/out [S, Hq, d]. Returns out."""
    lib = load()
    pool = make_pool(k_pool, v_pool)
    S, hq, d = q.shape
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    mb = int(block_tables.shape[1])
    ws = _workspace(pa_decode_workspace_size(S, hq, d, mb), q.device, workspace)
    _check("pa_decode",
           lib.pa_decode(ctypes.byref(pool), _ptr(out), _ptr(q), S, hq, _ptr(block_tables), mb,
                         _ptr(context_lens), float(scale), _ptr(ws), ws.numel() * ws.element_size(),
                         _ptr(d_status), _stream(stream)))
    return out


def pa_decode_with_ctas(out, q, k_pool, v_pool, block_tables, context_lens, scale: float,
                        num_ctas: int, workspace=None, d_status=None, stream=None):
    """pa_decode on ``num_ctas`` persistent CTAs (0: one per SM). Returns out."""
    lib = load()
    pool = make_pool(k_pool, v_pool)
    S, hq, d = q.shape
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    mb = int(block_tables.shape[1])
    ws = _workspace(pa_decode_workspace_size(S, hq, d, mb), q.device, workspace)
    _check("pa_decode_with_ctas",
           lib.pa_decode_with_ctas(ctypes.byref(pool), _ptr(out), _ptr(q), S, hq, _ptr(block_tables),
                                   mb, _ptr(context_lens), float(scale), int(num_ctas), _ptr(ws),
                                   ws.numel() * ws.element_size(), _ptr(d_status), _stream(stream)))
    return out


def pa_decode_cascade_workspace_size(num_seqs: int, num_q_heads: int, head_dim: int,
                                    max_blocks_per_seq: int) -> int:
    return int(load().pa_decode_cascade_workspace_size(num_seqs, num_q_heads, head_dim,
                                                       max_blocks_per_seq))


def pa_decode_cascade(out, q, k_pool, v_pool, block_tables, context_lens, cu_groups, prefix_lens,
                      scale: float, workspace=None, d_status=None, stream=None):
    """Decode attention over groups of sequences sharing a prefix of whole
    blocks: sequences cu_groups[g] .. cu_groups[g+1]-1 share their first
    prefix_lens[g] tokens (see include/pa.h). q/out [S, Hq, d]. Returns out."""
    return pa_decode_cascade_with_ctas(out, q, k_pool, v_pool, block_tables, context_lens,
                                       cu_groups, prefix_lens, scale, 0, workspace, d_status,
                                       stream, _name="pa_decode_cascade")


def pa_decode_cascade_with_ctas(out, q, k_pool, v_pool, block_tables, context_lens, cu_groups,
                                prefix_lens, scale: float, num_ctas: int, workspace=None,
                                d_status=None, stream=None, _name="pa_decode_cascade_with_ctas"):
    """pa_decode_cascade with ``num_ctas`` persistent decode CTAs (0: one per
    SM). Returns out."""
    lib = load()
    pool = make_pool(k_pool, v_pool)
    S, hq, d = q.shape
    for name, t in (("block_tables", block_tables), ("context_lens", context_lens),
                    ("cu_groups", cu_groups), ("prefix_lens", prefix_lens)):
        if t.dtype != torch.int32:
            raise TypeError(f"{name} must be int32")
    ng = int(prefix_lens.shape[0])
    if int(cu_groups.shape[0]) != ng + 1:
        raise ValueError("cu_groups must hold num_groups + 1 entries")
    mb = int(block_tables.shape[1])
    ws = _workspace(pa_decode_cascade_workspace_size(S, hq, d, mb), q.device, workspace)
    args = (ctypes.byref(pool), _ptr(out), _ptr(q), S, hq, _ptr(block_tables), mb,
            _ptr(context_lens), _ptr(cu_groups), _ptr(prefix_lens), ng, float(scale))
    tail = (_ptr(ws), ws.numel() * ws.element_size(), _ptr(d_status), _stream(stream))
    if _name == "pa_decode_cascade":
        rc = lib.pa_decode_cascade(*args, *tail)
    else:
        rc = lib.pa_decode_cascade_with_ctas(*args, int(num_ctas), *tail)
    _check(_name, rc)
    return out


def pa_decode_cascade_nested_workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                                           head_dim: int, max_blocks_per_seq: int,
                                           num_ctas: int = 0) -> int:
    return int(load().pa_decode_cascade_nested_workspace_size(
        num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, num_ctas))


def pa_decode_cascade_nested(out, q, k_pool, v_pool, block_tables, context_lens, cu_groups,
                             prefix_lens, cu_siblings, sibling_lens, scale: float,
                             num_ctas: int = 0, workspace=None, d_status=None, stream=None):
    """Two-level cascade decode (see include/pa.h): groups sharing a prefix
    (cu_groups / prefix_lens, may be empty) and sibling groups sharing a longer
    one (cu_siblings / sibling_lens), each sibling entry's shared blocks read
    once. q/out [S, Hq, d]. Returns out."""
    lib = load()
    pool = make_pool(k_pool, v_pool)
    S, hq, d = q.shape
    for name, t in (("block_tables", block_tables), ("context_lens", context_lens),
                    ("cu_groups", cu_groups), ("prefix_lens", prefix_lens),
                    ("cu_siblings", cu_siblings), ("sibling_lens", sibling_lens)):
        if t.dtype != torch.int32:
            raise TypeError(f"{name} must be int32")
    ng = int(prefix_lens.shape[0])
    nsib = int(sibling_lens.shape[0])
    if int(cu_groups.shape[0]) != ng + 1:
        raise ValueError("cu_groups must hold num_groups + 1 entries")
    if int(cu_siblings.shape[0]) != nsib + 1:
        raise ValueError("cu_siblings must hold num_sibling_groups + 1 entries")
    mb = int(block_tables.shape[1])
    hkv = int(k_pool.shape[2])
    ws = _workspace(pa_decode_cascade_nested_workspace_size(S, hq, hkv, d, mb, int(num_ctas)),
                    q.device, workspace)
    rc = lib.pa_decode_cascade_nested(
        ctypes.byref(pool), _ptr(out), _ptr(q), S, hq, _ptr(block_tables), mb,
        _ptr(context_lens), _ptr(cu_groups), _ptr(prefix_lens), ng, _ptr(cu_siblings),
        _ptr(sibling_lens), nsib, float(scale), int(num_ctas), _ptr(ws),
        ws.numel() * ws.element_size(), _ptr(d_status), _stream(stream))
    _check("pa_decode_cascade_nested", rc)
    return out


def pa_gather_probe(k_pool, v_pool, blocks, stages: int = 3, ctas: int = 0, d_status=None,
                    stream=None) -> None:
    """Measurement aid (include/pa_probe.h, libpa_probe.so): stream the listed
    K/V blocks into shared memory with the decode kernel's copies and compute
    nothing."""
    lib = load_probe()
    pool = make_pool(k_pool, v_pool)
    if blocks.dtype != torch.int32:
        raise TypeError("blocks must be int32")
    _check("pa_gather_probe", lib.pa_gather_probe(ctypes.byref(pool), _ptr(blocks),
                                                  int(blocks.numel()), stages, ctas,
                                                  _ptr(d_status), _stream(stream)))


def pa_wait_probe(src, starve: bool, limit_ns: int, d_status=None, stream=None) -> None:
    """Test aid (include/pa_probe.h, libpa_probe.so): one CTA through the
    kernels' bounded wait; with ``starve`` the copy is never started and the
    wait gives up after ``limit_ns``, setting PA_STATUS_TIMEOUT."""
    lib = load_probe()
    if src.numel() * src.element_size() < 1024:
        raise ValueError("src must hold at least 1,024 bytes")
    _check("pa_wait_probe", lib.pa_wait_probe(_ptr(src), int(bool(starve)), int(limit_ns),
                                              _ptr(d_status), _stream(stream)))


PA_DECODE_STATIC_WS_BYTES = 32 << 20


def pa_decode_static_ws(out, q, k_pool, v_pool, block_tables, context_lens, scale: float,
                        d_status=None, stream=None):
    """Decode attention that allocates nothing: the split-K scratch is a
    static device array inside libpa (see include/pa.h). For callers that
    cannot allocate device memory around the call. Returns out."""
    lib = load()
    pool = make_pool(k_pool, v_pool)
    S, hq, d = q.shape
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    mb = int(block_tables.shape[1])
    _check("pa_decode_static_ws",
           lib.pa_decode_static_ws(ctypes.byref(pool), _ptr(out), _ptr(q), S, hq,
                                   _ptr(block_tables), mb, _ptr(context_lens), float(scale),
                                   _ptr(d_status), _stream(stream)))
    return out


def pa_mixed_step(out, q, cu_q_lens, context_lens, block_tables, k_pool, v_pool, scale: float,
                  token_budget: int, k_new=None, v_new=None, slot_mapping=None, workspace=None,
                  d_status=None, stream=None):
    """Mixed decode + prefill-chunk step, q/out [T, Hq, d]. Returns out."""
    return _mixed(None, out, q, cu_q_lens, context_lens, block_tables, k_pool, v_pool, scale,
                  token_budget, k_new, v_new, slot_mapping, workspace, d_status, stream)


def pa_mixed_step_with_units(out, q, cu_q_lens, context_lens, block_tables, k_pool, v_pool,
                             scale: float, token_budget: int, prefill_q_tiles: int, k_new=None,
                             v_new=None, slot_mapping=None, workspace=None, d_status=None,
                             stream=None):
    """pa_mixed_step with 1 or 2 query tiles per tensor-core prefill unit (0: automatic)."""
    return _mixed(int(prefill_q_tiles), out, q, cu_q_lens, context_lens, block_tables, k_pool,
                  v_pool, scale, token_budget, k_new, v_new, slot_mapping, workspace, d_status,
                  stream)


def _mixed(q_tiles, out, q, cu_q_lens, context_lens, block_tables, k_pool, v_pool, scale,
           token_budget, k_new, v_new, slot_mapping, workspace, d_status, stream):
    lib = load()
    pool = make_pool(k_pool, v_pool)
    T, hq, d = q.shape
    S = int(context_lens.shape[0])
    if (cu_q_lens.dtype != torch.int32 or block_tables.dtype != torch.int32
            or context_lens.dtype != torch.int32):
        raise TypeError("cu_q_lens, block_tables and context_lens must be int32")
    mb = int(block_tables.shape[1])
    ws = _workspace(pa_mixed_workspace_size(S, T, hq, d, mb), q.device, workspace)
    common = (ctypes.byref(pool), _ptr(out), _ptr(q), _ptr(cu_q_lens), S, T, hq,
              _ptr(context_lens), _ptr(block_tables), mb, float(scale), int(token_budget),
              _ptr(k_new), _ptr(v_new), _ptr(slot_mapping))
    tail = (_ptr(ws), ws.numel() * ws.element_size(), _ptr(d_status), _stream(stream))
    if q_tiles is None:
        _check("pa_mixed_step", lib.pa_mixed_step(*common, *tail))
    else:
        _check("pa_mixed_step_with_units", lib.pa_mixed_step_with_units(*common, q_tiles, *tail))
    return out
