"""Planted mistakes in the oracle must trip at least one pin.

Each case copies oracle.c, applies one plausible mistake (a dropped term, a
wrong sign or index, a transposed layout), builds the copy with gcc on the CPU
and runs the pin battery against it. The shipped oracle is never modified.
"""
import os
import shutil

import pytest

import oracle
import oracle_pins as P

HERE = os.path.dirname(os.path.abspath(__file__))
SRC_DIR = os.path.join(os.path.dirname(HERE), "oracle")

MUTANTS = {
    # causal rule drops the diagonal key
    "causal_excludes_diagonal": [("p <= P", "p < P")],
    # GQA: query head -> KV head by modulo instead of contiguous groups
    "gqa_modulo": [("const int g = h / group;", "const int g = h % j->num_kv_heads;")],
    # softmax scale dropped
    "scale_dropped": [("scores[p] = j->scale * dot;", "scores[p] = dot;")],
    # chunk-local instead of absolute positions
    "relative_positions": [("row_pos[cu_q_lens[s] + i] = ctx - q_len + i;",
                            "row_pos[cu_q_lens[s] + i] = i;")],
    # pool read as [N_blk, Hkv, b, d]
    "pool_layout_transposed": [("((block * b + p % b) * j->num_kv_heads + g) * (int64_t)d",
                                "((block * j->num_kv_heads + g) * b + p % b) * (int64_t)d")],
    # token order reversed inside a block
    "offset_reversed": [("(block * b + p % b)", "(block * b + (b - 1 - p % b))")],
    # wrong sign in the softmax exponent
    "softmax_sign": [("exp(scores[p] - m)", "exp(m - scores[p])")],
    # max not subtracted (overflows on large logits)
    "max_not_subtracted": [("exp(scores[p] - m)", "exp(scores[p])")],
    # output not normalised by the sum of weights
    "no_normalisation": [("o[i] /= l;", "o[i] /= 1.0;")],
    # values read from the K pool
    "v_from_k_pool": [("load_value(j->v_pool,", "load_value(j->k_pool,")],
    # bf16 widened with the wrong shift
    "bf16_widen": [("((uint32_t)half) << 16", "((uint32_t)half) << 15")],
    # KV write lands one slot late
    "write_offset": [("int64_t offset = slot % block_size;",
                      "int64_t offset = (slot + 1) % block_size;")],
    # copy-on-write copies one filled slot too few
    "cow_slot_short": [("int slots = ntok ? ntok[i] : block_size;",
                        "int slots = ntok ? ntok[i] - 1 : block_size;")],
    # copy-on-write copies the whole block, unfilled slots included
    "cow_whole_block": [("int slots = ntok ? ntok[i] : block_size;", "int slots = block_size;")],
    # copy direction reversed (the copy overwrites the shared block)
    "cow_reversed": [("memcpy((char*)k_pool + to * block_bytes, (const char*)k_pool + from * block_bytes, bytes);",
                      "memcpy((char*)k_pool + from * block_bytes, (const char*)k_pool + to * block_bytes, bytes);")],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    src = open(os.path.join(SRC_DIR, "oracle.c")).read()
    for old, new in MUTANTS[name]:
        assert old in src, (name, old)
        src = src.replace(old, new)
    d = tmp_path / name
    d.mkdir()
    shutil.copy(os.path.join(SRC_DIR, "oracle.h"), d / "oracle.h")
    (d / "oracle.c").write_text(src)
    so = oracle.build(str(d / "oracle.c"), str(d / "liboracle.so"), force=True)
    lib = oracle.load(so)
    caught = []
    for pin in P.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError) as e:  # a failing pin
            caught.append((pin.__name__, repr(e)[:80]))
            break
    assert caught, f"planted mistake {name} passed every pin"
