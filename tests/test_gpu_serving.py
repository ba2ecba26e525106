"""Continuous batching with chunked prefill driving the CUDA path, every step
checked against the oracle on a host mirror of the paged pool."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_176_gb300.serving import ServingLoop, pa_copy_blocks
from parity import compare

pytestmark = pytest.mark.gpu


def _bytes(t):
    t = t.contiguous().cpu()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.numpy().view(np.uint8)


def run_with_oracle(dtype, hq, hkv, d, reqs, num_blocks, budget, chunk, max_running, max_ctx):
    loop = ServingLoop(num_blocks, hq, hkv, d, dtype=dtype, token_budget=budget, chunk_size=chunk,
                       max_running=max_running, max_context=max_ctx, seed=3)
    for rid, (prompt, new) in enumerate(reqs):
        loop.submit(rid, prompt, new)
    hk, hv = loop.k_pool.cpu(), loop.v_pool.cpu()  # host mirror of the pool
    mixed_steps = 0
    while True:
        p = loop.step()
        if p is None:
            break
        torch.cuda.synchronize()
        S, T = p.num_seqs, p.num_tokens
        for i in range(p.num_cow):
            hk[int(p.cow_dst[i])] = hk[int(p.cow_src[i])]
            hv[int(p.cow_dst[i])] = hv[int(p.cow_src[i])]
        oracle.reshape_and_cache(hk, hv, loop.k_new[:T].cpu(), loop.v_new[:T].cpu(),
                                 torch.from_numpy(p.slot_mapping[:T].copy()))
        ref = oracle.paged_attention(loop.q[:T].cpu(), hk, hv,
                                     torch.from_numpy(p.cu_q_lens[:S + 1].copy()),
                                     torch.from_numpy(p.context_lens[:S].copy()),
                                     torch.from_numpy(p.tables.copy()), loop.scale)
        compare(loop.out[:T], ref, dtype)
        mixed_steps += int(0 < p.num_decode < S)
    assert int(loop.status.item()) == 0
    assert np.array_equal(_bytes(loop.k_pool), _bytes(hk))
    assert np.array_equal(_bytes(loop.v_pool), _bytes(hv))
    assert loop.bm.num_free == num_blocks
    st = loop.sched.stats()
    assert st["finished"] == len(reqs)
    return loop.steps, mixed_steps


def test_serving_loop_bf16_tensor_core_path():
    rng = np.random.default_rng(1)
    reqs = [(int(rng.integers(1, 400)), int(rng.integers(1, 20))) for _ in range(12)]
    steps, mixed = run_with_oracle(torch.bfloat16, 16, 4, 128, reqs, 320, 128, 64, 6, 512)
    assert steps > 10 and mixed > 0  # decode tokens and prefill chunks shared steps


def test_serving_loop_f32_cuda_core_path():
    rng = np.random.default_rng(2)
    reqs = [(int(rng.integers(1, 200)), int(rng.integers(1, 12))) for _ in range(8)]
    run_with_oracle(torch.float32, 8, 2, 64, reqs, 200, 96, 40, 5, 256)


def test_copy_blocks_bit_exact():
    g = torch.Generator().manual_seed(4)
    k = torch.randn(40, 16, 8, 128, generator=g).bfloat16()
    v = torch.randn(40, 16, 8, 128, generator=g).bfloat16()
    k[3] = float("nan")
    src = torch.tensor([1, 3, 7, 7], dtype=torch.int32)
    dst = torch.tensor([2, 30, 8, 39], dtype=torch.int32)
    dk, dv = k.cuda(), v.cuda()
    pa_copy_blocks(dk, dv, src.cuda(), dst.cuda())
    torch.cuda.synchronize()
    for s, d_ in zip(src.tolist(), dst.tolist()):
        k[d_] = k[s]
        v[d_] = v[s]
    assert np.array_equal(_bytes(dk), _bytes(k)) and np.array_equal(_bytes(dv), _bytes(v))
