"""Shared helpers for the GPU parity tests: move a workload to the device, run
the CUDA path through the C-ABI binding, compare with the oracle.

Tolerances (the output is compared element by element with the fp64 oracle
computed on the same stored input values):

* fp32 inputs: |gpu - oracle| <= 1e-5 for every element.
* bf16 inputs, max-abs <= 1e-2 AND max-rel <= 2e-2, each asserted wherever
  bf16 arithmetic can meet it:
    - absolute: |gpu - oracle| <= 1e-2 for every element with |oracle| < 4.
      The GPU rounds its fp32 result to bf16, whose spacing is 2^(e-7) for
      |x| in [2^e, 2^(e+1)): at |x| >= 4 half a spacing is 1/64 > 1e-2, so
      the rounding alone can exceed the absolute bound there, while below 4
      it is at most 1/128 and leaves room for the fp32 accumulation error.
      Elements with |oracle| >= 4 are exempt from the absolute bound only,
      and their count is reported.
    - relative: |gpu - oracle| <= 2e-2 * |oracle| for every element with
      |oracle| >= 0.5, the magnitude at which the relative bound reaches the
      absolute one. Nearer zero a relative error measures the cancellation
      inside the weighted average, not the kernel (the bf16 rounding of the
      softmax weights gives an absolute error that does not shrink with |o|);
      max-rel over |oracle| >= 0.1 is reported, not asserted.
* KV writes and copies: byte-exact.

Each comparison's summary (max-abs, max-rel, exempt count) is appended as one
JSON line to the file named by the environment variable PA_PARITY_LOG, when it
is set, so a run can record the margins of every workload.
"""
from __future__ import annotations

import json
import os
from dataclasses import dataclass

import numpy as np
import torch

import oracle
import paged_kv_cache_176_gb300 as pa
from paged_kv_cache_176_gb300 import workloads as W

F32_ATOL = 1e-5
BF16_ATOL = 1e-2
BF16_RTOL = 2e-2
BF16_ABS_EXEMPT = 4.0   # |oracle| at and above which half a bf16 spacing exceeds 1e-2
BF16_REL_FLOOR = 0.5    # |oracle| at and above which the relative bound is asserted


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


def run_decode(w: W.Workload, db: DeviceBatch | None = None,
               ctas: int = 0) -> tuple[torch.Tensor, DeviceBatch]:
    """KV write (if the workload has one) then pa_decode, as one decode step;
    ``ctas`` > 0 runs the decode on that many persistent CTAs."""
    db = db or to_device(w)
    if db.slot_mapping is not None:
        pa.pa_reshape_and_cache(db.k_pool, db.v_pool, db.k_new, db.v_new, db.slot_mapping,
                                d_status=db.status)
    out = torch.empty_like(db.q)
    if ctas:
        pa.pa_decode_with_ctas(out, db.q, db.k_pool, db.v_pool, db.block_tables, db.context_lens,
                               w.scale, ctas, d_status=db.status)
    else:
        pa.pa_decode(out, db.q, db.k_pool, db.v_pool, db.block_tables, db.context_lens, w.scale,
                     d_status=db.status)
    torch.cuda.synchronize()
    return out, db


def run_mixed(w: W.Workload, db: DeviceBatch | None = None, write: bool = True, units: int = 0):
    """pa_mixed_step (units == 0) or pa_mixed_step_with_units with 1 or 2
    query tiles per tensor-core prefill unit."""
    db = db or to_device(w)
    out = torch.empty_like(db.q)
    kw = dict(k_new=db.k_new if write else None, v_new=db.v_new if write else None,
              slot_mapping=db.slot_mapping if write else None, d_status=db.status)
    if units:
        pa.pa_mixed_step_with_units(out, db.q, db.cu_q_lens, db.context_lens, db.block_tables,
                                    db.k_pool, db.v_pool, w.scale, w.token_budget, units, **kw)
    else:
        pa.pa_mixed_step(out, db.q, db.cu_q_lens, db.context_lens, db.block_tables, db.k_pool,
                         db.v_pool, w.scale, w.token_budget, **kw)
    torch.cuda.synchronize()
    return out, db


def bf16_errors(got: np.ndarray, ref: np.ndarray) -> dict:
    """Error summary of a bf16 result against the fp64 oracle (both fp64 arrays)."""
    err = np.abs(got - ref)
    mag = np.abs(ref)
    info = {"n": int(err.size), "max_abs": float(err.max()) if err.size else 0.0}
    in_abs = mag < BF16_ABS_EXEMPT
    info["max_abs_checked"] = float(err[in_abs].max()) if in_abs.any() else 0.0
    info["n_abs_exempt"] = int((~in_abs).sum())
    for floor, key in ((BF16_REL_FLOOR, "max_rel"), (0.1, "max_rel_ge_0.1")):
        sel = mag >= floor
        info[key] = float((err[sel] / mag[sel]).max()) if sel.any() else 0.0
    info["n_abs_bad"] = int((err[in_abs] > BF16_ATOL).sum())
    rel_sel = mag >= BF16_REL_FLOOR
    info["n_rel_bad"] = int((err[rel_sel] > BF16_RTOL * mag[rel_sel]).sum())
    return info


def _log(info: dict) -> None:
    path = os.environ.get("PA_PARITY_LOG")
    if not path:
        return
    rec = dict(info, test=os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0])
    with open(path, "a") as f:
        f.write(json.dumps(rec) + "\n")


def compare(got: torch.Tensor, ref: np.ndarray, dtype: torch.dtype, rows=None) -> dict:
    """Element-wise check against the oracle; returns the error summary and
    raises AssertionError on failure."""
    g = got.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        g = g[rows]
        ref = ref[rows]
    assert np.all(np.isfinite(ref)), "oracle output not finite"
    assert np.all(np.isfinite(g)), f"GPU output has {np.sum(~np.isfinite(g))} non-finite values"
    if dtype == torch.float32:
        err = np.abs(g - ref)
        info = {"dtype": "f32", "n": int(err.size), "max_abs": float(err.max()) if err.size else 0.0}
        _log(info)
        assert info["max_abs"] <= F32_ATOL, info
    else:
        info = dict(bf16_errors(g, ref), dtype="bf16")
        _log(info)
        assert info["n_abs_bad"] == 0 and info["n_rel_bad"] == 0, info
    return info


def oracle_out(w: W.Workload, row_mask=None) -> np.ndarray:
    return oracle.workload_attention(w, row_mask=row_mask)
