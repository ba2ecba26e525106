"""The bf16 acceptance rule of the parity tests, checked on planted errors
(CPU only): max-abs 1e-2 below |oracle| = 4, max-rel 2e-2 from |oracle| = 0.5."""
import numpy as np
import pytest
import torch

from parity import bf16_errors, compare


def _one(ref: float, err: float) -> dict:
    r = np.array([ref], dtype=np.float64)
    return bf16_errors(r + err, r)


@pytest.mark.parametrize("ref,err,ok", [
    (3.0, 0.009, True),      # inside the absolute bound
    (3.0, 0.02, False),      # 0.7 % relative, but above 1e-2 absolute below |o| = 4
    (0.6, 0.011, False),     # absolute bound governs here too
    (0.01, 0.009, True),     # near zero only the absolute bound is asserted
    (5.0, 0.03, True),       # |o| >= 4: exempt from the absolute bound, 0.6 % relative
    (5.0, 0.15, False),      # 3 % relative
    (-6.0, -0.2, False),     # sign does not matter
])
def test_bf16_rule(ref, err, ok):
    info = _one(ref, err)
    assert (info["n_abs_bad"] == 0 and info["n_rel_bad"] == 0) == ok, info


def test_bf16_exempt_count_and_compare_raises():
    ref = np.array([[0.1, 4.5], [2.0, -7.0]])
    got = ref + np.array([[0.001, 0.02], [0.001, 0.05]])
    info = compare(torch.tensor(got, dtype=torch.float32), ref, torch.bfloat16)
    assert info["n_abs_exempt"] == 2 and info["max_abs_checked"] <= 0.0011
    with pytest.raises(AssertionError):
        compare(torch.tensor(ref + 0.011, dtype=torch.float32), ref, torch.bfloat16)


def test_f32_rule():
    ref = np.zeros((3, 2))
    compare(torch.tensor(ref + 5e-6, dtype=torch.float32), ref, torch.float32)
    with pytest.raises(AssertionError):
        compare(torch.tensor(ref + 3e-5, dtype=torch.float32), ref, torch.float32)
