"""Failure detection on the GPU without a GPU fault: the kernels' bounded
wait gives up, reports PA_STATUS_TIMEOUT, releases its TMEM and returns, and
the context stays usable.

The wait runs out on a barrier armed for a copy that is never started
(pa_wait_probe in libpa_probe), so no copy is in flight when the CTA leaves.
"""
import time

import pytest
import torch

from paged_kv_cache_176_gb300 import abi
from paged_kv_cache_176_gb300 import workloads as W
from parity import compare, oracle_out, run_decode, run_mixed

pytestmark = pytest.mark.gpu


def _probe(src, starve, limit_ns):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    abi.pa_wait_probe(src, starve, limit_ns, d_status=st)
    torch.cuda.synchronize()
    return int(st.item()), time.perf_counter() - t0


def test_bounded_wait_times_out_and_context_stays_usable():
    src = torch.arange(256, dtype=torch.int32, device="cuda")  # 1,024 bytes
    # the copy completes: no status bit, the bytes arrived
    st, _ = _probe(src, False, 1_000_000)
    assert st == 0
    # the copy never starts: the 1 ms wait gives up and the kernel returns
    st, secs = _probe(src, True, 1_000_000)
    assert st == abi.PA_STATUS_TIMEOUT
    assert secs < 1.0, secs
    # a kernel that leaves without freeing TMEM would stall the next
    # allocation; run the TMEM-holding probe again, several times, then the
    # normal path and a real decode call
    for _ in range(3):
        st, secs = _probe(src, True, 200_000)
        assert st == abi.PA_STATUS_TIMEOUT and secs < 1.0
    st, _ = _probe(src, False, 1_000_000)
    assert st == 0
    w = W.decode_b64(num_seqs=4, num_blocks=100, ctx_range=(40, 300))
    out, db = run_decode(w)
    assert int(db.status.item()) == 0
    compare(out, oracle_out(w), torch.bfloat16)
    # the mixed step's tcgen05 kernel allocates TMEM too
    wm = W.paged_workload("after_timeout", 3, [200, 40], [1, 40], 16, 8, 128, 32, torch.bfloat16,
                          write_new=True)
    outm, dbm = run_mixed(wm)
    assert int(dbm.status.item()) == 0
    compare(outm, oracle_out(wm), torch.bfloat16)
