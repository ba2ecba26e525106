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
    return drive_with_oracle(loop, num_blocks, len(reqs), dtype)


def drive_with_oracle(loop, num_blocks, num_reqs, dtype, on_step=None):
    """Run the loop to the end, checking every step against the oracle on a
    host mirror of the pool; ``on_step(plan)`` runs after each check."""
    hk, hv = loop.k_pool.cpu(), loop.v_pool.cpu()  # host mirror of the pool
    mixed_steps = 0
    while True:
        p = loop.step()
        if p is None:
            break
        torch.cuda.synchronize()
        S, T = p.num_seqs, p.num_tokens
        if p.num_cow:
            assert oracle.copy_blocks(hk, hv, torch.from_numpy(p.cow_src[:p.num_cow].copy()),
                                      torch.from_numpy(p.cow_dst[:p.num_cow].copy()),
                                      torch.from_numpy(p.cow_ntok[:p.num_cow].copy())) == 0
        oracle.reshape_and_cache(hk, hv, loop.k_new[:T].cpu(), loop.v_new[:T].cpu(),
                                 torch.from_numpy(p.slot_mapping[:T].copy()))
        ref = oracle.paged_attention(loop.q[:T].cpu(), hk, hv,
                                     torch.from_numpy(p.cu_q_lens[:S + 1].copy()),
                                     torch.from_numpy(p.context_lens[:S].copy()),
                                     torch.from_numpy(p.tables.copy()), loop.scale)
        compare(loop.out[:T], ref, dtype)
        mixed_steps += int(0 < p.num_decode < S)
        if on_step is not None:
            on_step(p, hk, hv)
    assert int(loop.status.item()) == 0
    assert np.array_equal(_bytes(loop.k_pool), _bytes(hk))
    assert np.array_equal(_bytes(loop.v_pool), _bytes(hv))
    assert loop.bm.num_free == num_blocks
    st = loop.sched.stats()
    assert st["finished"] == num_reqs
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


@pytest.mark.parametrize("cache", [True, False])
def test_serving_loop_prefix_cache(cache):
    # requests share a 100-token system prompt (6 full pages) and add a
    # question; with the cache on, later requests prefill only what misses
    rng = np.random.default_rng(4)
    vocab = 500
    system = rng.integers(0, vocab, size=100).tolist()
    reqs = [(system + rng.integers(0, vocab, size=int(rng.integers(1, 60))).tolist(),
             int(rng.integers(1, 12))) for _ in range(16)]
    loop = ServingLoop(200, 16, 4, 128, dtype=torch.bfloat16, token_budget=128, chunk_size=64,
                       max_running=4, max_context=256, seed=5, vocab=vocab, prefix_cache=cache)
    for rid, (p, n) in enumerate(reqs):
        loop.submit(rid, len(p), n, tokens=p)
    toks = {rid: list(p) for rid, (p, _) in enumerate(reqs)}
    emb_k = loop.emb_k.cpu()

    def check_pages(p, hk, hv):
        # every sequence's cache holds exactly its tokens' rows, shared or not
        S = p.num_seqs
        nxt = loop.next_tokens(p)
        for j in range(S):
            sid, ctx = int(p.seq_ids[j]), int(p.context_lens[j])
            table = p.tables[j]
            slots = [int(table[q // 16]) * 16 + q % 16 for q in range(ctx)]
            got = hk.view(-1, 4, 128)[slots]
            assert torch.equal(got, emb_k[toks[sid][:ctx]]), (sid, ctx)
            if j < p.num_decode or ctx == len(reqs[sid][0]):
                toks[sid].append(int(nxt[j]))

    drive_with_oracle(loop, 200, len(reqs), torch.bfloat16, on_step=check_pages)
    st = loop.sched.stats()
    prompts = sum(len(p) for p, _ in reqs)
    if cache:
        assert loop.sched.cached_tokens >= 96 * 8
        assert st["prefill_tokens"] == prompts - loop.sched.cached_tokens
    else:
        assert loop.sched.cached_tokens == 0 and st["prefill_tokens"] == prompts


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
    assert oracle.copy_blocks(k, v, src, dst) == 0
    assert np.array_equal(_bytes(dk), _bytes(k)) and np.array_equal(_bytes(dv), _bytes(v))
