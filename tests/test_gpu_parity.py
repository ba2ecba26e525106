"""GPU parity: the CUDA path, called through the C-ABI binding, against the
fp64 oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import oracle
import oracle_pins
import paged_kv_cache_176_gb300 as pa
from paged_kv_cache_176_gb300 import workloads as W
from parity import compare, oracle_out, run_decode, run_mixed, to_device

pytestmark = pytest.mark.gpu


def _bytes(t: torch.Tensor) -> np.ndarray:
    t = t.contiguous().cpu()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.numpy().view(np.uint8)


# ------------------------------------------------------------------ KV write


@pytest.mark.parametrize("make", [W.tiny_decode_f32, lambda: oracle_pins._mixed_small(8)],
                         ids=["f32", "bf16"])
def test_kv_write_bit_exact(make):
    w = make()
    if w.slot_mapping is None:  # give the fp32 case new tokens too
        w = W.paged_workload("w", 3, [17, 40, 64, 100], [5, 1, 16, 33], 8, 2, 64, 32,
                             torch.float32, write_new=True)
    sm = w.slot_mapping.clone()
    sm[::7] = -1  # padding tokens are skipped
    db = to_device(w)
    pa.pa_reshape_and_cache(db.k_pool, db.v_pool, db.k_new, db.v_new, sm.cuda(), d_status=db.status)
    torch.cuda.synchronize()
    kp, vp = w.k_pool.clone(), w.v_pool.clone()
    oracle.reshape_and_cache(kp, vp, w.k_new, w.v_new, sm)
    assert np.array_equal(_bytes(db.k_pool), _bytes(kp))
    assert np.array_equal(_bytes(db.v_pool), _bytes(vp))
    assert int(db.status.item()) == 0


def test_kv_write_full_config_bit_exact():
    w = W.decode_b64()
    db = to_device(w)
    pa.pa_reshape_and_cache(db.k_pool, db.v_pool, db.k_new, db.v_new, db.slot_mapping)
    torch.cuda.synchronize()
    kp, vp = w.k_pool.clone(), w.v_pool.clone()
    oracle.reshape_and_cache(kp, vp, w.k_new, w.v_new, w.slot_mapping)
    assert np.array_equal(_bytes(db.k_pool), _bytes(kp))
    assert np.array_equal(_bytes(db.v_pool), _bytes(vp))


def test_kv_write_bad_slot_flags_and_skips():
    w = oracle_pins._mixed_small(9)
    sm = w.slot_mapping.clone()
    sm[0] = w.num_blocks * 16  # one past the pool
    db = to_device(w)
    before = _bytes(db.k_pool).copy()
    pa.pa_reshape_and_cache(db.k_pool, db.v_pool, db.k_new, db.v_new, sm.cuda(), d_status=db.status)
    torch.cuda.synchronize()
    assert int(db.status.item()) & pa.abi.PA_STATUS_BAD_SLOT
    kp = w.k_pool.clone()
    sm_ok = sm.clone()
    sm_ok[0] = -1
    oracle.reshape_and_cache(kp, w.v_pool.clone(), w.k_new, w.v_new, sm_ok)
    assert np.array_equal(_bytes(db.k_pool), _bytes(kp))
    assert not np.array_equal(before, _bytes(db.k_pool))


# ------------------------------------------------------------------ decode


def test_decode_tiny_f32():
    w = W.tiny_decode_f32()
    out, db = run_decode(w)
    info = compare(out, oracle_out(w), torch.float32)
    assert int(db.status.item()) == 0, info


@pytest.mark.parametrize("hkv", [4, 8])
@pytest.mark.parametrize("ctas", [1, 3, 64, 1024])
def test_decode_split_counts(ctas, hkv):
    """Every CTA count gives the same result within tolerance, including a
    count far above the number of blocks (empty CTAs, many partials); 8 KV
    heads take the tensor-core products, 4 the CUDA-core ones."""
    w = W.paged_workload("split", 5, [1, 15, 16, 17, 33, 100, 257, 600], [1] * 8, 4 * hkv, hkv, 128,
                         200, torch.bfloat16, write_new=True)
    out, db = run_decode(w, ctas=ctas)
    compare(out, oracle_out(w), torch.bfloat16)
    assert int(db.status.item()) == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_cta_range_beyond_table_cache(dtype):
    """One CTA owning more blocks than it stages in shared memory (1,063 >
    1,024): the refills past the staged table read the block table directly;
    fp32 with 8 KV heads moves half blocks (two units per block)."""
    w = W.paged_workload("long", 13, [9000, 8000], [1, 1], 32, 8, 128, 1300, dtype,
                         write_new=True)
    out, db = run_decode(w, ctas=1)
    compare(out, oracle_out(w), dtype)
    assert int(db.status.item()) == 0


@pytest.mark.parametrize("d,hq,hkv,dtype", [
    (64, 8, 8, torch.bfloat16), (64, 16, 2, torch.float32), (128, 8, 1, torch.bfloat16),
    (128, 16, 4, torch.float32), (256, 16, 8, torch.bfloat16), (256, 8, 1, torch.float32),
    (128, 64, 8, torch.bfloat16), (256, 32, 4, torch.bfloat16),
    # tensor-core products (bf16, head_dim 64 / 128, 8 KV heads): every group size
    (128, 16, 8, torch.bfloat16), (64, 32, 8, torch.bfloat16), (64, 64, 8, torch.bfloat16),
])
def test_decode_shapes(d, hq, hkv, dtype):
    w = W.paged_workload("shape", 11, [3, 16, 31, 200, 513], [1] * 5, hq, hkv, d, 128, dtype,
                         write_new=True)
    for ctas in (0, 5):
        out, _ = run_decode(w, ctas=ctas)
        compare(out, oracle_out(w), dtype)


def test_decode_b64_full():
    w = W.decode_b64()
    out, db = run_decode(w)
    info = compare(out, oracle_out(w), torch.bfloat16)
    assert int(db.status.item()) == 0, info


def test_wide_gqa_full():
    w = W.wide_gqa_decode()
    out, db = run_decode(w)
    compare(out, oracle_out(w), torch.bfloat16)
    assert int(db.status.item()) == 0


def test_shared_prefix_full_and_cow_bit_identical():
    ws = W.shared_prefix_decode()
    out_s, _ = run_decode(ws)
    compare(out_s, oracle_out(ws), torch.bfloat16)
    wp = W.shared_prefix_decode(private=True)
    out_p, _ = run_decode(wp)
    assert torch.equal(out_s, out_p)  # copy-on-write sharing == private copies, bit for bit


def test_decode_permutation_bit_identical():
    w = W.decode_b64(num_seqs=16, num_blocks=1200, ctx_range=(100, 1000))
    out_a, _ = run_decode(w)
    out_b, _ = run_decode(oracle_pins.permute_pool(w, 4))
    assert torch.equal(out_a, out_b)


@pytest.mark.parametrize("hq,hkv,d,dtype", [(8, 2, 64, torch.float32), (32, 8, 128, torch.bfloat16)])
def test_decode_bad_block_and_length_zeroed(hq, hkv, d, dtype):
    w = W.paged_workload("bad", 2, [40, 40, 40], [1, 1, 1], hq, hkv, d, 32, dtype,
                         write_new=False)
    bt = w.block_tables.clone()
    bt[1, 1] = w.num_blocks + 5
    ctx = w.context_lens.clone()
    ctx[2] = bt.shape[1] * 16 + 1  # longer than the table
    w2 = W.Workload(w.name, w.dtype, w.num_q_heads, w.num_kv_heads, w.head_dim, 16, w.k_pool,
                    w.v_pool, w.q, w.cu_q_lens, ctx, bt, None, None, None, w.scale, 3)
    out, db = run_decode(w2)
    st = int(db.status.item())
    assert st & pa.abi.PA_STATUS_BAD_BLOCK and st & pa.abi.PA_STATUS_BAD_LENGTH
    assert torch.count_nonzero(out[1]) == 0 and torch.count_nonzero(out[2]) == 0
    good = oracle.paged_attention(w.q[:1], w.k_pool, w.v_pool, torch.tensor([0, 1], dtype=torch.int32),
                                  w.context_lens[:1], w.block_tables[:1], w.scale)
    compare(out[:1], good, dtype)


def test_decode_empty_batch():
    w = W.tiny_decode_f32()
    db = to_device(w)
    out = torch.zeros(0, w.num_q_heads, w.head_dim, device="cuda")
    pa.pa_decode(out, db.q[:0], db.k_pool, db.v_pool, db.block_tables[:0], db.context_lens[:0],
                 w.scale)


# ------------------------------------------------------------------ mixed step


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_mixed_small(dtype):
    w = oracle_pins._mixed_small(12, dtype, hq=8, hkv=2, d=64)
    out, db = run_mixed(w)
    compare(out, oracle_out(w), dtype)
    assert int(db.status.item()) == 0


def test_chunked_prefill_example_on_gpu():
    """The glossary page's experiment through pa_mixed_step: 1000 tokens in
    chunks of 256/256/256/232 equal one-pass causal prefill within 1e-5, and
    both equal the oracle."""
    r = oracle_pins.chunked_prefill_example(oracle.load())
    torch.manual_seed(0)
    q, k, v = torch.randn(3, 1, 8, 1000, 64).unbind(0)
    qt = q[0].transpose(0, 1).contiguous().cuda()
    kt = k[0].transpose(0, 1).contiguous().cuda()
    vt = v[0].transpose(0, 1).contiguous().cuda()
    nblk = 63
    perm = torch.randperm(80, generator=torch.Generator().manual_seed(1))[:nblk].to(torch.int32)
    table = perm.reshape(1, nblk).cuda()
    pos = torch.arange(1000)
    slots = (perm[pos // 16].to(torch.int64) * 16 + pos % 16).cuda()

    def run(chunk):
        kp = torch.full((80, 16, 8, 64), float("nan"), device="cuda")
        vp = torch.full_like(kp, float("nan"))
        outs = []
        for start in range(0, 1000, chunk):
            end = min(start + chunk, 1000)
            o = torch.empty(end - start, 8, 64, device="cuda")
            pa.pa_mixed_step(o, qt[start:end], torch.tensor([0, end - start], dtype=torch.int32).cuda(),
                             torch.tensor([end], dtype=torch.int32).cuda(), table, kp, vp, 0.125,
                             2048, k_new=kt[start:end], v_new=vt[start:end],
                             slot_mapping=slots[start:end])
            outs.append(o)
        return torch.cat(outs).cpu()

    chunked, one_pass = run(256), run(1000)
    assert torch.allclose(one_pass, chunked, atol=1e-5, rtol=0)
    compare(chunked, r["sdpa_fp64"], torch.float32)
    compare(one_pass, r["one_pass"], torch.float32)


@pytest.mark.parametrize("units", [0, 1])
def test_mixed_step_scaled_full(units):
    """Config-4 structure with 4,096-token prompts, every row checked: the
    library's choice (two query tiles per prefill unit at this size) and
    one-tile units."""
    w = W.mixed_step(num_decode=16, decode_ctx=(64, 2048), prompt_len=4096)
    out, db = run_mixed(w, units=units)
    compare(out, oracle_out(w), torch.bfloat16)
    assert int(db.status.item()) == 0


def test_mixed_step_full_sampled():
    """The full mixed step (budget 2048: 128 decode rows + chunks 512/512/512/384
    of 32,768-token prompts, 64/8 heads): every decode row and 64 sampled rows
    per prefill chunk (all heads) against the oracle."""
    w = W.mixed_step()
    out, db = run_mixed(w)
    assert int(db.status.item()) == 0
    nd = w.info["num_decode"]
    rng = np.random.default_rng(0)
    mask = np.zeros(w.num_tokens, dtype=np.uint8)
    mask[:nd] = 1
    cu = w.cu_q_lens.tolist()
    for s in range(nd, w.num_seqs):
        # 64 seeded rows of every chunk, plus its first and last rows (the
        # shortest and the longest key ranges)
        rows = rng.choice(np.arange(cu[s], cu[s + 1]), size=64, replace=False)
        mask[rows] = 1
        mask[cu[s]] = 1
        mask[cu[s + 1] - 1] = 1
    ref = oracle_out(w, row_mask=mask)
    compare(out, ref, torch.bfloat16, rows=np.nonzero(mask)[0])


def test_mixed_permutation_bit_identical():
    w = W.mixed_step(num_decode=8, decode_ctx=(64, 1024), prompt_len=2048)
    out_a, _ = run_mixed(w)
    out_b, _ = run_mixed(oracle_pins.permute_pool(w, 5))
    assert torch.equal(out_a, out_b)


def test_mixed_budget_rejected():
    w = oracle_pins._mixed_small(13, d=64)
    db = to_device(w)
    out = torch.empty_like(db.q)
    with pytest.raises(pa.PagedAttentionError) as e:
        pa.pa_mixed_step(out, db.q, db.cu_q_lens, db.context_lens, db.block_tables, db.k_pool,
                         db.v_pool, w.scale, w.num_tokens - 1)
    assert e.value.status == pa.abi.PA_EBUDGET


# ------------------------------------------------------------------ tensor-core prefill


@pytest.mark.parametrize("units", [1, 2])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (32, 8), (64, 8), (8, 2)])
def test_prefill_tc_groups_and_ragged_chunks(hq, hkv, units):
    """bf16, head_dim 128 (the tcgen05 path): every GQA group size, chunks at
    offset 0 and at ragged offsets, chunk lengths that are not multiples of the
    tile, 2-token chunks, contexts spanning several 128-key tiles and partial
    last blocks (slots past the context hold NaN); units of one query tile and
    of two (including two-tile units whose second tile is empty)."""
    ctx = [37, 300, 129, 1000, 2, 517, 64]
    ql = [37, 45, 2, 201, 2, 1, 17]
    w = W.paged_workload("tc", 21, ctx, ql, hq, hkv, 128, 300, torch.bfloat16, write_new=True)
    out, db = run_mixed(w, units=units)
    compare(out, oracle_out(w), torch.bfloat16)
    assert int(db.status.item()) == 0


@pytest.mark.parametrize("units", [1, 2])
def test_prefill_tc_without_kv_write(units):
    """The cache already holds every token (no KV write in the step)."""
    ctx = [700, 260, 96]
    ql = [300, 260, 40]
    w = W.paged_workload("tc_nowrite", 22, ctx, ql, 32, 8, 128, 200, torch.bfloat16, write_new=False)
    out, db = run_mixed(w, write=False, units=units)
    compare(out, oracle_out(w), torch.bfloat16)
    assert int(db.status.item()) == 0


@pytest.mark.parametrize("units", [1, 2])
def test_prefill_tc_chunked_equals_one_pass(units):
    """A 1000-token prompt prefilled in chunks of 256 through the tensor-core
    path equals one pass, within the bf16 tolerance, and both match the oracle."""
    L, H, G = 1000, 8, 4
    w1 = W.paged_workload("onepass", 23, [L], [L], H * G, H, 128, 80, torch.bfloat16, write_new=True)
    out1, _ = run_mixed(w1, units=units)
    ref = oracle_out(w1)
    compare(out1, ref, torch.bfloat16)
    db = to_device(w1)
    db.k_pool.fill_(float("nan"))
    db.v_pool.fill_(float("nan"))
    outs = []
    for start in range(0, L, 256):
        end = min(start + 256, L)
        o = torch.empty(end - start, H * G, 128, dtype=torch.bfloat16, device="cuda")
        pa.pa_mixed_step_with_units(o, db.q[start:end],
                                    torch.tensor([0, end - start], dtype=torch.int32).cuda(),
                                    torch.tensor([end], dtype=torch.int32).cuda(), db.block_tables,
                                    db.k_pool, db.v_pool, w1.scale, 2048, units,
                                    k_new=db.k_new[start:end], v_new=db.v_new[start:end],
                                    slot_mapping=db.slot_mapping[start:end])
        outs.append(o)
    chunked = torch.cat(outs)
    compare(chunked, ref, torch.bfloat16)


@pytest.mark.parametrize("units", [1, 2])
def test_prefill_tc_running_max_jumps(units):
    """Scores that jump far past the lazy-rescale threshold (8 in the log2
    domain) inside later key tiles, for one query head of a group only, so a
    warp holds rows whose running max moves and rows whose max stays: a jump
    in the second 64-key half of a tile (the first half's P is already in
    TMEM and is rescaled in place), a larger one in the first half of the
    next tile, and one among the chunk's own keys; both unit sizes."""
    hq, hkv, G = 32, 8, 4
    w = W.paged_workload("jumps", 31, [700, 420], [180, 64], hq, hkv, 128, 200, torch.bfloat16,
                         write_new=True)
    q, k_pool, k_new = w.q.clone(), w.k_pool.clone(), w.k_new.clone()
    cu = w.cu_q_lens.tolist()
    rng = np.random.default_rng(7)
    # (first, last + 1, scale) of planted cached keys per sequence: sequence 0
    # jumps in keys 192-255 of key tile 1, then again in keys 256-319 of
    # tile 2; sequence 1 in keys 128-191 of tile 1
    plants = {0: [(200, 205, 4.0), (300, 303, 6.0)], 1: [(150, 153, 3.0)]}
    for s_i, spans in plants.items():
        g = s_i  # KV head whose query head g * G sees the planted keys
        u = torch.from_numpy(rng.standard_normal(128)).to(torch.bfloat16)
        t0, t1 = cu[s_i], cu[s_i + 1]
        q[t0:t1, g * G] = u  # one query head of the group, every row of the chunk
        first_new = int(w.context_lens[s_i]) - (t1 - t0)
        for lo, hi, c in spans:
            for pos in range(lo, hi):
                assert pos < first_new  # a cached key, in the pool
                blk = int(w.block_tables[s_i, pos // 16])
                k_pool[blk, pos % 16, g] = (c * u.float()).to(torch.bfloat16)
        # one planted key among the chunk's own tokens, written by the step:
        # for sequence 1 it jumps again inside keys 320-383 of tile 2
        k_new[t0 + 5, g] = (5.0 * u.float()).to(torch.bfloat16)
    w.q, w.k_pool, w.k_new = q, k_pool, k_new
    out, db = run_mixed(w, units=units)
    compare(out, oracle_out(w), torch.bfloat16)
    assert int(db.status.item()) == 0


@pytest.mark.parametrize("hq,hkv,d,dtype,units", [(64, 8, 128, torch.bfloat16, 1),
                                                   (64, 8, 128, torch.bfloat16, 2),
                                                   (8, 2, 64, torch.float32, 0)])
def test_prefill_bad_block_and_length_zeroed(hq, hkv, d, dtype, units):
    """A prefill chunk whose first block-table entry is out of range (every
    unit of it reads that block) and a chunk longer than its context: both
    flagged in the status word, their rows zero; the decode rows and the
    other chunk of the step still match the oracle. Tensor-core prefill with
    one- and two-tile units, and the CUDA-core prefill."""
    ctx = [300, 700, 200, 90, 40]
    ql = [1, 150, 60, 1, 33]
    w = W.paged_workload("bad_pf", 41, ctx, ql, hq, hkv, d, 160, dtype, write_new=True)
    ref = oracle_out(w)  # with the valid tables and lengths
    db = to_device(w)
    db.block_tables[1, 0] = int(w.k_pool.shape[0]) + 5  # sequence 1: bad first block
    db.context_lens[4] = 20  # sequence 4: 33 rows over a context of 20
    out, db = run_mixed(w, db=db, units=units)
    st = int(db.status.item())
    assert st & pa.abi.PA_STATUS_BAD_BLOCK and st & pa.abi.PA_STATUS_BAD_LENGTH
    cu = w.cu_q_lens.tolist()
    bad = np.zeros(w.num_tokens, dtype=bool)
    for s in (1, 4):
        bad[cu[s]:cu[s + 1]] = True
    got = out.float().cpu()
    assert torch.count_nonzero(got[torch.from_numpy(bad)]) == 0
    good = np.nonzero(~bad)[0]
    compare(out, ref, dtype, rows=good)


def test_gather_probe_runs_and_flags_bad_blocks():
    # the measurement aid of include/pa_probe.h: no output, only a status
    k = torch.zeros(64, 16, 8, 128, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    blocks = torch.randperm(64, dtype=torch.int32).cuda()
    for stages, ctas in ((3, 0), (1, 5), (2, 200)):
        pa.abi.pa_gather_probe(k, v, blocks, stages=stages, ctas=ctas, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    pa.abi.pa_gather_probe(k, v, torch.tensor([3, 64, 5], dtype=torch.int32, device="cuda"),
                           d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == pa.abi.PA_STATUS_BAD_BLOCK
    with pytest.raises(pa.abi.PagedAttentionError):
        pa.abi.pa_gather_probe(k, v, blocks, stages=4)  # 4 x 64 KB exceeds shared memory
