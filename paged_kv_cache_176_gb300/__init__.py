"""Attention over a paged KV cache on GB300 (sm_103a).

The compute path is libpa.so (CUDA kernels behind the C ABI in include/pa.h);
``abi`` is its ctypes binding and ``workloads`` draws seeded synthetic inputs.
"""
from .abi import (  # noqa: F401
    PagedAttentionError,
    pa_decode,
    pa_decode_cascade,
    pa_decode_cascade_workspace_size,
    pa_decode_workspace_size,
    pa_mixed_step,
    pa_mixed_workspace_size,
    pa_reshape_and_cache,
    pa_decode_with_ctas,
    pa_mixed_step_with_units,
    pa_decode_cascade_with_ctas,
    pa_decode_cascade_nested,
    pa_decode_cascade_nested_workspace_size,
    pa_strerror,
    pa_version,
)

__all__ = [
    "pa_reshape_and_cache",
    "pa_decode",
    "pa_decode_cascade",
    "pa_decode_cascade_workspace_size",
    "pa_decode_workspace_size",
    "pa_mixed_step",
    "pa_mixed_workspace_size",
    "pa_decode_with_ctas",
    "pa_mixed_step_with_units",
    "pa_decode_cascade_with_ctas",
    "pa_decode_cascade_nested",
    "pa_decode_cascade_nested_workspace_size",
    "pa_strerror",
    "pa_version",
    "PagedAttentionError",
]
