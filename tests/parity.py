"""Shared helpers for the GPU parity tests: move a workload to the device, run
the CUDA path through the C-ABI binding, compare with the oracle.

Tolerances (the output is compared element by element with the fp64 oracle
computed on the same stored input values):

* fp32 inputs: max |gpu - oracle| <= 1e-5;
* bf16 inputs: an element passes iff |gpu - oracle| <= max(1e-2, 2e-2 * |oracle|)
  (max-abs 1e-2 and max-rel 2e-2, the absolute bound governing small values).
  The GPU accumulates in fp32 and rounds its output to bf16, so for |o| >= 4
  half a bf16 ulp alone exceeds 1e-2; the relative bound covers those.
* KV writes: byte-exact.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

import oracle
import paged_kv_cache_176_gb300 as pa
from paged_kv_cache_176_gb300 import workloads as W

F32_ATOL = 1e-5
BF16_ATOL = 1e-2
BF16_RTOL = 2e-2


@dataclass
class DeviceBatch:
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    q: torch.Tensor
    cu_q_lens: torch.Tensor
    context_lens: torch.Tensor
    block_tables: torch.Tensor
    k_new: torch.Tensor | None
    v_new: torch.Tensor | None
    slot_mapping: torch.Tensor | None
    status: torch.Tensor


def to_device(w: W.Workload, device="cuda") -> DeviceBatch:
    def d(t):
        return None if t is None else t.to(device).contiguous()

    return DeviceBatch(d(w.k_pool), d(w.v_pool), d(w.q), d(w.cu_q_lens), d(w.context_lens),
                       d(w.block_tables), d(w.k_new), d(w.v_new), d(w.slot_mapping),
                       torch.zeros(1, dtype=torch.int32, device=device))


def run_decode(w: W.Workload, db: DeviceBatch | None = None) -> tuple[torch.Tensor, DeviceBatch]:
    """KV write (if the workload has one) then pa_decode, as one decode step."""
    db = db or to_device(w)
    if db.slot_mapping is not None:
        pa.pa_reshape_and_cache(db.k_pool, db.v_pool, db.k_new, db.v_new, db.slot_mapping,
                                d_status=db.status)
    out = torch.empty_like(db.q)
    pa.pa_decode(out, db.q, db.k_pool, db.v_pool, db.block_tables, db.context_lens, w.scale,
                 d_status=db.status)
    torch.cuda.synchronize()
    return out, db


def run_mixed(w: W.Workload, db: DeviceBatch | None = None, write: bool = True):
    db = db or to_device(w)
    out = torch.empty_like(db.q)
    pa.pa_mixed_step(out, db.q, db.cu_q_lens, db.context_lens, db.block_tables, db.k_pool,
                     db.v_pool, w.scale, w.token_budget,
                     k_new=db.k_new if write else None, v_new=db.v_new if write else None,
                     slot_mapping=db.slot_mapping if write else None, d_status=db.status)
    torch.cuda.synchronize()
    return out, db


def compare(got: torch.Tensor, ref: np.ndarray, dtype: torch.dtype, rows=None) -> dict:
    """Element-wise check against the oracle; returns the error summary and
    raises AssertionError on failure."""
    g = got.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        g = g[rows]
        ref = ref[rows]
    assert np.all(np.isfinite(ref)), "oracle output not finite"
    assert np.all(np.isfinite(g)), f"GPU output has {np.sum(~np.isfinite(g))} non-finite values"
    err = np.abs(g - ref)
    info = {"max_abs": float(err.max()) if err.size else 0.0}
    big = np.abs(ref) >= 0.5
    info["max_rel_big"] = float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0
    if dtype == torch.float32:
        assert info["max_abs"] <= F32_ATOL, info
    else:
        bound = np.maximum(BF16_ATOL, BF16_RTOL * np.abs(ref))
        bad = err > bound
        info["n_bad"] = int(bad.sum())
        assert not bad.any(), info
    return info


def oracle_out(w: W.Workload, row_mask=None) -> np.ndarray:
    return oracle.workload_attention(w, row_mask=row_mask)
