"""The oracle against its pins (CPU only)."""
import numpy as np
import pytest

import oracle
import oracle_pins as P


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, lib):
    pin(lib)


def test_chunked_prefill_matches_page_printout(lib):
    """The glossary page prints '4 chunks, same result as one pass: True'."""
    r = P.chunked_prefill_example(lib)
    same = bool(np.allclose(r["one_pass"], r["chunked"], atol=1e-5, rtol=0))
    line = f"{len(r['sizes'])} chunks, same result as one pass: {same}"
    assert line == "4 chunks, same result as one pass: True"


def test_oracle_rejects_bad_inputs(lib):
    import torch
    from paged_kv_cache_176_gb300 import workloads as W
    w = W.tiny_decode_f32()
    bad = w.block_tables.clone()
    bad[0, 0] = w.num_blocks  # out of the pool
    with pytest.raises(ValueError):
        oracle.paged_attention(w.q, w.k_pool, w.v_pool, w.cu_q_lens, w.context_lens, bad, w.scale,
                               lib=lib)
    ctx = w.context_lens.clone()
    ctx[0] = 0  # q_len 1 > ctx 0
    with pytest.raises(ValueError):
        oracle.paged_attention(w.q, w.k_pool, w.v_pool, w.cu_q_lens, ctx, w.block_tables, w.scale,
                               lib=lib)
    sm = torch.tensor([w.num_blocks * 16], dtype=torch.int64)
    with pytest.raises(ValueError):
        oracle.reshape_and_cache(w.k_pool.clone(), w.v_pool.clone(), w.k_pool[0, :1],
                                 w.v_pool[0, :1], sm, lib=lib)


def test_anchor_pool_sizes():
    """The C13-L2 anchor sizes behind the wide-head GQA workload."""
    g = P._golden("anchor_pool_sizes.json")
    assert g["kv_heads"] * g["head_dim"] == g["D"]
    assert g["context"] // g["b"] == g["n_b"]
    assert g["b"] * g["bytes_per_token_all_layers"] == g["block_bytes"] == 2 ** 20
    assert round(g["N_blk"] * g["block_bytes"] / 1e9, 2) == g["kv_gb"]
    from paged_kv_cache_176_gb300 import workloads as W
    import inspect
    sig = inspect.signature(W.wide_gqa_decode)
    assert sig.parameters["num_blocks"].default == g["N_blk"]
    assert sig.parameters["ctx"].default == g["context"]
