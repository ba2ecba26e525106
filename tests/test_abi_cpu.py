"""The C-ABI library loads, exports every declared symbol, and its host-side
validation rejects bad arguments before any CUDA call (runs without a GPU)."""
import ctypes
import os
import re

import pytest

from paged_kv_cache_176_gb300 import abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions(headers):
    names = []
    for fn in headers:
        text = open(os.path.join(ROOT, "include", fn)).read()
        names += re.findall(r"^PA_API\s+[\w\s\*]+?\b(pa_\w+)\s*\(", text, flags=re.M)
    return names


@pytest.fixture(scope="module")
def lib():
    return abi.load()


def test_exports_every_declared_symbol(lib):
    """libpa exports everything pa.h and pa_serving.h declare; libpa_probe
    everything pa_probe.h declares, and libpa none of the probes."""
    headers = sorted(f for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h"))
    assert "pa_probe.h" in headers
    names = declared_functions([h for h in headers if h != "pa_probe.h"])
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n
    probe = abi.load_probe()
    probes = declared_functions(["pa_probe.h"])
    assert set(probes) == {"pa_gather_probe", "pa_wait_probe"}
    for n in probes:
        assert hasattr(probe, n), n
        assert not hasattr(lib, n), n


def test_version_and_strerror(lib):
    assert abi.pa_version() >> 16 == 1
    for code in (0, -1, -2, -3, -4, -5):
        assert abi.pa_strerror(code)
    assert abi.pa_strerror(-99) == "unknown status"


FAKE = 0x10000  # aligned, never dereferenced by host validation


def pool(**kw):
    p = dict(k=FAKE, v=FAKE, num_blocks=32, block_size=16, num_kv_heads=2, head_dim=64, dtype=0)
    p.update(kw)
    return abi.pa_kv_pool(p["k"], p["v"], p["num_blocks"], p["block_size"], p["num_kv_heads"],
                          p["head_dim"], p["dtype"])


def decode(lib, pl, q=FAKE, out=FAKE, hq=8, S=4, mb=8, ws=FAKE, ws_bytes=1 << 40):
    return lib.pa_decode(ctypes.byref(pl), out, q, S, hq, FAKE, mb, FAKE, 0.125, ws, ws_bytes,
                         None, None)


def test_decode_validation(lib):
    assert decode(lib, pool(k=None)) == abi.PA_EINVAL
    assert decode(lib, pool(v=FAKE + 4)) == abi.PA_EINVAL          # misaligned
    assert decode(lib, pool(block_size=8)) == abi.PA_EUNSUPPORTED
    assert decode(lib, pool(head_dim=96)) == abi.PA_EUNSUPPORTED
    assert decode(lib, pool(dtype=7)) == abi.PA_EUNSUPPORTED
    assert decode(lib, pool(), hq=6) == abi.PA_EUNSUPPORTED        # group 3
    assert decode(lib, pool(), hq=7) == abi.PA_EINVAL              # not a multiple
    assert decode(lib, pool(num_kv_heads=16), hq=16) == abi.PA_EUNSUPPORTED
    assert decode(lib, pool(), q=None) == abi.PA_EINVAL
    assert decode(lib, pool(), out=FAKE + 8) == abi.PA_EINVAL
    assert decode(lib, pool(), ws=None) == abi.PA_EWORKSPACE
    assert decode(lib, pool(), ws_bytes=16) == abi.PA_EWORKSPACE
    assert decode(lib, pool(), S=-1) == abi.PA_EINVAL
    assert decode(lib, pool(), S=0) == abi.PA_OK                   # nothing to do


def test_workspace_queries(lib):
    assert abi.pa_decode_workspace_size(-1, 8, 64, 8) == 0
    a = abi.pa_decode_workspace_size(4, 8, 64, 8)
    b = abi.pa_decode_workspace_size(64, 32, 128, 256)
    assert 0 < a < b
    assert abi.pa_mixed_workspace_size(4, 10, 8, 64, 8) >= a


def test_mixed_and_write_validation(lib):
    pl = pool()
    rc = lib.pa_mixed_step(ctypes.byref(pl), FAKE, FAKE, FAKE, 2, 100, 8, FAKE, FAKE, 8, 0.1, 64,
                           None, None, None, FAKE, 1 << 40, None, None)
    assert rc == abi.PA_EBUDGET
    rc = lib.pa_mixed_step(ctypes.byref(pl), FAKE, FAKE, FAKE, 2, 10, 8, FAKE, FAKE, 8, 0.1, 64,
                           FAKE, None, FAKE, FAKE, 1 << 40, None, None)  # v_new missing
    assert rc == abi.PA_EINVAL
    rc = lib.pa_mixed_step(ctypes.byref(pl), FAKE, FAKE, None, 2, 10, 8, FAKE, FAKE, 8, 0.1, 64,
                           None, None, None, FAKE, 1 << 40, None, None)
    assert rc == abi.PA_EINVAL
    rc = lib.pa_mixed_step(ctypes.byref(pl), FAKE, FAKE, FAKE, 2, 10, 8, FAKE, FAKE, 8, 0.1, 64,
                           None, None, None, FAKE, 16, None, None)
    assert rc == abi.PA_EWORKSPACE
    assert lib.pa_reshape_and_cache(ctypes.byref(pl), FAKE, FAKE, FAKE, -1, None, None) == abi.PA_EINVAL
    assert lib.pa_reshape_and_cache(ctypes.byref(pl), None, FAKE, FAKE, 3, None, None) == abi.PA_EINVAL
    assert lib.pa_reshape_and_cache(ctypes.byref(pl), FAKE + 2, FAKE, FAKE, 3, None, None) == abi.PA_EINVAL
    assert lib.pa_reshape_and_cache(ctypes.byref(pl), FAKE, FAKE, FAKE, 0, None, None) == abi.PA_OK


def test_prefill_unit_size_is_an_argument(lib):
    """pa_mixed_step_with_units takes 0, 1 or 2 query tiles per prefill unit;
    anything else is rejected before any device work."""
    pl = pool()
    for bad in (-1, 3, 64):
        rc = lib.pa_mixed_step_with_units(ctypes.byref(pl), FAKE, FAKE, FAKE, 2, 10, 8, FAKE, FAKE,
                                          8, 0.1, 64, None, None, None, bad, FAKE, 1 << 40, None,
                                          None)
        assert rc == abi.PA_EINVAL
    for ok in (0, 1, 2):  # valid unit sizes reach the workspace check
        rc = lib.pa_mixed_step_with_units(ctypes.byref(pl), FAKE, FAKE, FAKE, 2, 10, 8, FAKE, FAKE,
                                          8, 0.1, 64, None, None, None, ok, FAKE, 16, None, None)
        assert rc == abi.PA_EWORKSPACE


def test_decode_cta_count_is_an_argument(lib):
    """The CTA count is passed per call; the library has no setter for it."""
    assert not hasattr(lib, "pa_set_decode_ctas")
    pl = pool()
    args = (ctypes.byref(pl), FAKE, FAKE, 4, 8, FAKE, 8, FAKE, 0.125)
    assert lib.pa_decode_with_ctas(*args, -1, FAKE, 1 << 40, None, None) == abi.PA_EINVAL
    assert lib.pa_decode_with_ctas(ctypes.byref(pool(head_dim=96)), FAKE, FAKE, 4, 8, FAKE, 8, FAKE,
                                   0.125, 3, FAKE, 1 << 40, None, None) == abi.PA_EUNSUPPORTED
    assert lib.pa_decode_with_ctas(*args, 3, FAKE, 16, None, None) == abi.PA_EWORKSPACE
    bf16 = pool(dtype=1, head_dim=128)
    assert lib.pa_decode_cascade_with_ctas(ctypes.byref(bf16), FAKE, FAKE, 4, 8, FAKE, 8, FAKE,
                                           FAKE, FAKE, 1, 0.125, -2, FAKE, 1 << 40, None,
                                           None) == abi.PA_EINVAL


def test_static_workspace_checks_arguments_before_size(lib):
    """pa_decode_static_ws returns pa_decode's status for a bad call even when
    the batch is too large for its array; only a valid call gets PA_EWORKSPACE."""
    S = 1 << 20
    big = dict(S=S, hq=64)
    f = lib.pa_decode_static_ws

    def call(pl, S=4, hq=8, q=FAKE):
        return f(ctypes.byref(pl), FAKE, q, S, hq, FAKE, 8, FAKE, 0.125, None, None)

    assert call(pool(num_kv_heads=8, head_dim=256), **big) == abi.PA_EWORKSPACE
    assert call(pool(num_kv_heads=8, head_dim=96), **big) == abi.PA_EUNSUPPORTED
    assert call(pool(num_kv_heads=8, head_dim=256), S=S, hq=60) == abi.PA_EINVAL
    assert call(pool(num_kv_heads=8, head_dim=256), q=None, **big) == abi.PA_EINVAL
    assert call(pool(), S=0) == abi.PA_OK


def test_wait_probe_validation():
    probe = abi.load_probe()
    assert probe.pa_wait_probe(None, 1, 1000000, None, None) == abi.PA_EINVAL
    assert probe.pa_wait_probe(FAKE + 8, 1, 1000000, None, None) == abi.PA_EINVAL
    assert probe.pa_wait_probe(FAKE, 1, 0, None, None) == abi.PA_EINVAL
    assert probe.pa_wait_probe(FAKE, 1, 3 * 10**9, None, None) == abi.PA_EINVAL


def test_binding_rejects_host_tensors():
    import torch
    k = torch.zeros(4, 16, 2, 64)
    with pytest.raises(ValueError):
        abi.make_pool(k, k)


def cascade(lib, pl, S=4, hq=8, mb=8, ng=1, cu=FAKE, plen=FAKE, ws=FAKE, ws_bytes=1 << 40):
    return lib.pa_decode_cascade(ctypes.byref(pl), FAKE, FAKE, S, hq, FAKE, mb, FAKE, cu, plen, ng,
                                 0.125, ws, ws_bytes, None, None)


def test_cascade_validation(lib):
    bf16 = dict(dtype=1, head_dim=128)
    assert cascade(lib, pool(k=None, **bf16)) == abi.PA_EINVAL
    assert cascade(lib, pool(**bf16), ng=-1) == abi.PA_EINVAL
    assert cascade(lib, pool(**bf16), mb=0) == abi.PA_EINVAL
    assert cascade(lib, pool(**bf16), hq=7) == abi.PA_EINVAL          # heads not a multiple
    # the shared-prefix pass runs on the bf16 head_dim-128 tensor-core kernel only
    assert cascade(lib, pool(dtype=0, head_dim=128)) == abi.PA_EUNSUPPORTED
    assert cascade(lib, pool(dtype=1, head_dim=64)) == abi.PA_EUNSUPPORTED
    sz = abi.pa_decode_cascade_workspace_size(768, 32, 128, 100)
    assert sz > abi.pa_decode_workspace_size(768, 32, 128, 100) + 768 * 32 * 128 * 4
    assert abi.pa_decode_cascade_workspace_size(-1, 32, 128, 100) == 0


def nested(lib, pl, S=4, hq=8, mb=8, ng=1, nsib=1, sib=FAKE, slen=FAKE, ctas=0, ws=FAKE,
           ws_bytes=1 << 40):
    return lib.pa_decode_cascade_nested(ctypes.byref(pl), FAKE, FAKE, S, hq, FAKE, mb, FAKE, FAKE,
                                        FAKE, ng, sib, slen, nsib, 0.125, ctas, ws, ws_bytes, None,
                                        None)


def test_nested_cascade_validation(lib):
    # (checks that come before the support test, which needs the CUDA driver)
    bf16 = dict(dtype=1, head_dim=128, num_kv_heads=2)
    assert nested(lib, pool(**bf16), nsib=-1) == abi.PA_EINVAL
    assert nested(lib, pool(**bf16), ng=-1) == abi.PA_EINVAL
    assert nested(lib, pool(**bf16), ctas=-1) == abi.PA_EINVAL
    assert nested(lib, pool(k=None, **bf16)) == abi.PA_EINVAL
    assert nested(lib, pool(dtype=0, head_dim=128)) == abi.PA_EUNSUPPORTED
    # an entry of up to 16 / G members that spans n CTAs leaves n partials per
    # member: the partial slots grow to num_seqs + (16 / G) x CTAs
    size = abi.pa_decode_cascade_nested_workspace_size
    plain = abi.pa_decode_cascade_workspace_size(768, 32, 128, 100)
    assert size(768, 32, 8, 128, 100, 0) > plain                      # G 4: 4 x 1024 slots
    per_slot = 32 * (128 * 4 + 8)
    assert size(768, 32, 8, 128, 100, 0) - size(768, 32, 8, 128, 100, 152) >= per_slot * 4 * (1024 - 152)
    assert size(768, 32, 8, 128, 100, 152) < size(768, 32, 8, 128, 100, 0)
    assert size(768, 64, 8, 128, 100, 152) > size(768, 32, 8, 128, 100, 152)
    assert size(-1, 32, 8, 128, 100, 0) == 0
    assert size(768, 30, 8, 128, 100, 0) == 0                          # heads not a multiple
    assert size(768, 32, 8, 128, 100, -1) == 0
