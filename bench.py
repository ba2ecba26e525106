"""Benchmark: paged-decode attention HBM GB/s and mixed-step tokens/s on GB300.

One step = one pass of the decode hot path over the decode batch of 64
sequences (32 query / 8 KV heads, head_dim 128, bf16, contexts uniform in
[512, 4096], tables from a shuffled pool of 20,000 blocks): the KV write of the
64 new tokens, then decode attention over the paged cache (block-table gather
fused). ``value`` is the step's algorithmic HBM bytes (every cached K/V byte
read once, q read, output written, new tokens read and written, tables read)
divided by the device time per step; inputs (613 MB of K/V) exceed the 129 MB
L2, so nothing is flushed between steps.

The mixed step (budget 2048: 128 decode tokens + 4 prefill chunks of
512/512/512/384 from 32,768-token prompts, 64/8 heads) is measured after the
timed region and reported under ``mixed_step`` in attention tokens/s.

``--impl reference`` times the fp64 CPU oracle on a bounded sample of the same
workload on the host cores. Under torchrun each rank runs its own replica
(weak scaling, no data-path collective); rank 0 prints the JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

MEASURED_PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

# The source pages' own figures: other hardware, whole-model serving, none a
# kernel number for this path; quoted beside the measurements as context only.
PAGES_CONTEXT = {
    "serving_tok_s_h100_sxm5_llama33_70b_fp8_128_concurrent": "2,200-2,400 (paged + continuous "
                                                             "+ chunked); ~1,800 without chunked "
                                                             "prefill",
    "decode_tok_s_h100_anchor_model_ctx4096": "~65 at batch 1, ~2,300 at 58 requests (a roofline "
                                              "bound, not measured)",
    "paged_attention_kernel_vs_fastertransformer": "20-26 % slower (hardware not stated)",
    "prefix_cache_ttft_1000_token_shared_prompt": "~50 ms -> ~5 ms (hardware not stated)",
}

# nominal GB300 figures, reported as a second column beside the measured peaks
SPEC_HBM_GBS = 7900.0        # HBM3e
SPEC_BF16_TFLOPS = 2250.0    # dense bf16 tensor

# DRAM bytes (read + write) of one pa_decode call (decode_kernel +
# decode_reduce_kernel) on the decode batch, from an ncu capture of
# `ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum`, valid for the
# kernel code whose sha256 prefix is given (see _src_sha); reported as null
# once the code changes.
NCU_DECODE_TRAFFIC = {"bytes": 643784960, "src_sha": "893b26b76f45472b"}


def _src_sha(path: str) -> str:
    """sha256 prefix of a source's code: lines stripped of // comments, blank
    lines dropped, so that editing prose does not mark counters stale."""
    lines = []
    with open(path) as f:
        for line in f:
            code = line.split("//", 1)[0].strip()
            if code:
                lines.append(code)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def peaks() -> dict:
    try:
        with open(MEASURED_PEAKS) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every ``interval_ms``."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 20):
        self.gpu = gpu_index
        self.interval_ms = interval_ms
        self.proc = None
        self.lines: list[str] = []
        self.skip = 0  # leading lines printed before the measured region
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def wait_first(self, limit_s: float = 3.0) -> "ClockSampler":
        """Block until nvidia-smi has printed its first sample (at most
        ``limit_s``), so that a short timed region is not spent while the
        sampler is still starting."""
        t0 = time.perf_counter()
        while self.proc is not None and not self.lines and time.perf_counter() - t0 < limit_s:
            time.sleep(0.005)
        return self

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines[self.skip:]:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "interval_ms": self.interval_ms}


def max_over_ranks(x: float, device=None) -> float:
    """Largest value of ``x`` over all ranks (``x`` itself without a process
    group). Used for the timed region: the job is as slow as its slowest rank."""
    import torch
    import torch.distributed as tdist
    if not (tdist.is_available() and tdist.is_initialized()) or tdist.get_world_size() == 1:
        return x
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def step_bytes(w) -> dict:
    """Algorithmic HBM bytes of one decode step (KV write + decode)."""
    elt = w.k_pool.element_size()
    tok = w.num_kv_heads * w.head_dim * elt
    kv_read = int(w.context_lens.to("cpu").long().sum()) * 2 * tok
    q_out = 2 * w.q.numel() * elt
    nblk = int(((w.context_lens.long() + 15) // 16).sum())
    tables = nblk * 4 + w.num_seqs * 4
    write = 2 * 2 * w.num_tokens * tok + w.num_tokens * 8 if w.slot_mapping is not None else 0
    decode = kv_read + q_out + tables
    return {"decode": decode, "write": write, "step": decode + write, "kv_read": kv_read}


def mixed_work(w) -> dict:
    """Algorithmic work of a mixed step: decode KV bytes, prefill causal FLOPs
    (QK^T and PV over the unmasked keys of every prefill row)."""
    cu = w.cu_q_lens.tolist()
    ctx = w.context_lens.tolist()
    elt = w.k_pool.element_size()
    tok = w.num_kv_heads * w.head_dim * elt
    dec_bytes, flops, pf_kv = 0, 0, 0
    for s in range(w.num_seqs):
        ql = cu[s + 1] - cu[s]
        if ql == 1:
            dec_bytes += ctx[s] * 2 * tok
        elif ql > 1:
            off = ctx[s] - ql
            keys = ql * off + ql * (ql + 1) // 2
            flops += 4 * w.num_q_heads * w.head_dim * keys
            pf_kv += ctx[s] * 2 * tok
    return {"decode_bytes": dec_bytes, "prefill_flops": flops, "prefill_kv_bytes": pf_kv}


# ------------------------------------------------------------------ GPU arm


def run_gpu(args, rank: int, world: int) -> dict | None:
    import torch
    import paged_kv_cache_176_gb300 as pa
    from paged_kv_cache_176_gb300 import workloads as W

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    pa.abi.load()
    w = W.decode_b64(seed=args.seed)
    nb = step_bytes(w)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        kp, vp = w.k_pool.to(dev), w.v_pool.to(dev)
        q, bt, cl = w.q.to(dev), w.block_tables.to(dev), w.context_lens.to(dev)
        kn, vn, sm = w.k_new.to(dev), w.v_new.to(dev), w.slot_mapping.to(dev)
        out = torch.empty_like(q)
        ws = torch.empty(pa.pa_decode_workspace_size(w.num_seqs, w.num_q_heads, w.head_dim,
                                                     w.max_blocks_per_seq),
                         dtype=torch.uint8, device=dev)
    torch.cuda.synchronize(dev)
    launches_per_step = 3  # KV write, decode, split-K merge

    def step():
        pa.pa_reshape_and_cache(kp, vp, kn, vn, sm, stream=stream)
        pa.pa_decode(out, q, kp, vp, bt, cl, w.scale, workspace=ws, stream=stream)

    # decode-call timing (dominant kernel pair), measured on its own stream
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    # events around every pa_decode call, in batches of 200 calls, until at
    # least 1 s of calls has run (whatever --steps is); clocks sampled meanwhile
    roof_clocks = ClockSampler(dev.index).start().wait_first()
    roof_clocks.skip = len(roof_clocks.lines)
    times, t_start = [], time.perf_counter()
    while time.perf_counter() - t_start < 1.0 or len(times) < 200:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(200)]
        for a, b in ev:
            pa.pa_reshape_and_cache(kp, vp, kn, vn, sm, stream=stream)
            a.record(stream)
            pa.pa_decode(out, q, kp, vp, bt, cl, w.scale, workspace=ws, stream=stream)
            b.record(stream)
        torch.cuda.synchronize(dev)
        times += [a.elapsed_time(b) for a, b in ev]
    roof_clk = roof_clocks.stop()
    decode_ms = statistics.median(times)
    gather = gather_ceiling(w, kp, vp, dev, stream)

    # timed region: exactly K steps
    dist = world > 1
    if dist:
        import torch.distributed as tdist
        tdist.barrier()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(dev.index).start().wait_first()
    clocks.skip = len(clocks.lines)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if not clk.get("samples"):
        # a timed region shorter than one sampling interval: report the
        # decode-call window's record (the same calls, >= 1 s, just before)
        clk = dict(roof_clk, source="decode-call window just before the timed region "
                   "(the timed region was shorter than one sampling interval)")
    ms = max_over_ranks(t0.elapsed_time(t1) / args.steps, dev)

    # end to end through the public API with host buffers: every step copies
    # its inputs (packed in one pinned buffer) to the device and reads its
    # output back. One stream moves step n+1's inputs and another step n-1's
    # output while the compute stream runs step n; device buffers are
    # double-buffered and events order their reuse.
    parts = [("q", w.q), ("k_new", w.k_new), ("v_new", w.v_new), ("slot", w.slot_mapping),
             ("bt", w.block_tables), ("cl", w.context_lens)]
    offs, o = {}, 0
    for name, t in parts:
        offs[name] = (o, t)
        o = (o + t.numel() * t.element_size() + 255) // 256 * 256
    in_bytes = o
    host_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    for name, t in parts:
        off, _ = offs[name]
        host_in[off:off + t.numel() * t.element_size()].copy_(
            t.contiguous().view(-1).view(torch.uint8))
    dev_in = [torch.empty(in_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]

    def view(buf, name):
        off, t = offs[name]
        n = t.numel() * t.element_size()
        return buf[off:off + n].view(t.dtype).view(t.shape)

    ins = [{name: view(b, name) for name, _ in parts} for b in dev_in]
    outs = [torch.empty_like(q) for _ in range(2)]
    host_out = [torch.empty(w.q.shape, dtype=w.q.dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for _, t in parts)
    d2h = host_out[0].numel() * host_out[0].element_size()
    e2e_steps = max(50, min(args.steps, 2000))
    copy_stream = torch.cuda.Stream(dev)   # host -> device
    read_stream = torch.cuda.Stream(dev)   # device -> host
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for e in ev_done + ev_out:
        e.record(stream)

    def e2e_step(i):
        k = i % 2
        d = ins[k]
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(ev_done[k])     # step i-2 no longer reads dev_in[k]
            dev_in[k].copy_(host_in, non_blocking=True)
            ev_in[k].record(copy_stream)
        stream.wait_event(ev_in[k])
        stream.wait_event(ev_out[k])               # step i-2's output has been read back
        pa.pa_reshape_and_cache(kp, vp, d["k_new"], d["v_new"], d["slot"], stream=stream)
        pa.pa_decode(outs[k], d["q"], kp, vp, d["bt"], d["cl"], w.scale, workspace=ws,
                     stream=stream)
        ev_done[k].record(stream)
        with torch.cuda.stream(read_stream):
            read_stream.wait_event(ev_done[k])
            host_out[k].copy_(outs[k], non_blocking=True)
            ev_out[k].record(read_stream)

    for i in range(5):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    wall0 = time.perf_counter()
    e0.record(copy_stream)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_stream(read_stream)
    stream.wait_stream(copy_stream)
    e1.record(stream)                              # after the last read-back
    torch.cuda.synchronize(dev)
    wall = (time.perf_counter() - wall0) / e2e_steps * 1e3

    # the same with every copy on the compute stream (no overlap), for reference
    def serial_step(i):
        k = i % 2
        d = ins[k]
        dev_in[k].copy_(host_in, non_blocking=True)
        pa.pa_reshape_and_cache(kp, vp, d["k_new"], d["v_new"], d["slot"], stream=stream)
        pa.pa_decode(outs[k], d["q"], kp, vp, d["bt"], d["cl"], w.scale, workspace=ws,
                     stream=stream)
        host_out[k].copy_(outs[k], non_blocking=True)

    with torch.cuda.stream(stream):
        for i in range(5):
            serial_step(i)
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for i in range(e2e_steps):
            serial_step(i)
        s1.record(stream)
        torch.cuda.synchronize(dev)
    serial_ms = max_over_ranks(s0.elapsed_time(s1) / e2e_steps, dev)
    e2e_ms = max_over_ranks(max(e0.elapsed_time(e1) / e2e_steps, wall), dev)

    # mixed step (secondary measurement)
    mixed = None
    if not args.skip_mixed:
        mixed = run_mixed(args, dev, stream)
    extra = None
    if not args.skip_extra:
        extra = run_extra(args, dev, stream)

    serving = prefix = None
    if not args.skip_serving:
        serving = run_serving(args, dev, stream)
        prefix = run_prefix_cache(args, dev, stream)

    pk = peaks()
    decode_gbs = nb["decode"] / (decode_ms * 1e-3) / 1e9
    src = os.path.join(ROOT, "paged_kv_cache_176_gb300", "csrc", "decode_impl.cuh")
    traffic = None
    if NCU_DECODE_TRAFFIC["bytes"] and NCU_DECODE_TRAFFIC["src_sha"] == _src_sha(src):
        traffic = NCU_DECODE_TRAFFIC["bytes"]
    value = world * nb["step"] / (ms * 1e-3) / 1e9
    res = {
        "metric": "paged-decode attention HBM GB/s (% of peak) and mixed-step tokens/s on 1 GB300",
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1), bf16-rounded; no dataset)",
        "config": {"workload": "decode_b64_bf16: 64 seqs, ctx U[512,4096], 32/8 heads, d 128, "
                               "block 16, pool 20000 shuffled blocks, + KV write of 64 tokens",
                   "kv_bytes_per_step": nb["kv_read"], "algorithmic_bytes_per_step": nb["step"],
                   "l2": "inputs 613 MB > 129 MB L2; no flush",
                   "parallelism": f"replicas x{world}"},
        "attention_tokens_per_s": round(world * w.num_seqs / (ms * 1e-3), 1),
        "kv_tokens_scanned_per_s": round(world * int(w.context_lens.sum()) / (ms * 1e-3), 1),
        "roofline": {"bound": "hbm", "kernel": "pa_decode (decode_kernel + decode_reduce_kernel)",
                     "achieved": round(decode_gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": round(decode_gbs / pk["hbm_gbs"], 4), "traffic": traffic,
                     "frac_of_spec": round(decode_gbs / SPEC_HBM_GBS, 4),
                     "spec_peak": SPEC_HBM_GBS,
                     "peak_source": pk["source"], "ms_per_launch": round(decode_ms, 5),
                     "launches_timed": len(times), "clocks": roof_clk,
                     "gather_ceiling": dict(gather, decode_frac_of_ceiling=round(
                         decode_gbs / gather["gbs"], 4)),
                     "algorithmic_bytes_per_launch": nb["decode"]},
        "e2e": {"value": round(world * nb["step"] / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 5),
                "copies": "every step copies its inputs (one packed pinned buffer) in and its "
                          "output out; step n+1's inputs and step n-1's output move on two copy "
                          "streams while step n computes (double-buffered device buffers)",
                "serial": {"value": round(world * nb["step"] / (serial_ms * 1e-3) / 1e9, 1),
                           "ms_per_step": round(serial_ms, 5),
                           "copies": "the same copies on the compute stream, no overlap"}},
        "gpu_launches": launches_per_step * args.steps,
        "pages_context": PAGES_CONTEXT,
        "clocks": clk,
        "build": build_record(),
    }
    if mixed is not None:
        res["mixed_step"] = mixed
    if extra is not None:
        res["other_decode_workloads"] = extra
    if serving is not None:
        res["serving_loop"] = serving
    if prefix is not None:
        res["prefix_cache"] = prefix
    return res


SHARED_PREFIX_WORKLOAD = ("shared_prefix_decode_bf16: 256 requests x 3 replies, 1000-token shared "
                          "prefix + 100 unique, replies U[22,356], 32/8 heads, d 128, + KV write of "
                          "768 tokens")


def run_extra(args, dev, stream) -> list:
    """The other decode workloads: wide-head GQA, and the shared-prefix
    batch through pa_decode and through pa_decode_cascade (one group over the
    62 prefix pages every sequence shares)."""
    from paged_kv_cache_176_gb300 import workloads as W
    out = [run_decode_workload("tiny_decode_f32: 4 seqs, ctx {17,40,64,100}, 8/2 heads, d 64 "
                               "(launch-bound)", W.tiny_decode_f32(seed=args.seed), dev, stream,
                               reps=200)]
    w = W.wide_gqa_decode(seed=args.seed)
    out.append(run_decode_workload("wide_gqa_decode_bf16: 58 seqs x 4096, 16/4 heads, d 256, "
                                   "pool 23305", w, dev, stream))
    w = W.shared_prefix_decode(seed=args.seed)
    out.append(run_decode_workload(SHARED_PREFIX_WORKLOAD, w, dev, stream))
    plen = w.info["shared_pages"] * 16
    out.append(run_decode_workload(SHARED_PREFIX_WORKLOAD + "; pa_decode_cascade, one group "
                                   f"sharing {plen} prefix tokens", w, dev, stream,
                                   groups=([0, w.num_seqs], [plen])))
    R, rep = w.info["num_requests"], w.info["replies"]
    prompt_full = (w.info["prompt_len"] // 16) * 16
    out.append(run_decode_workload(
        SHARED_PREFIX_WORKLOAD + f"; pa_decode_cascade_nested, one group sharing {plen} prefix "
        f"tokens and {R} sibling groups (a request's {rep} replies) sharing {prompt_full} prompt "
        "tokens", w, dev, stream, groups=([0, w.num_seqs], [plen]),
        siblings=([r * rep for r in range(R + 1)], [prompt_full] * R)))
    del w
    out.append(run_cow_step(args, dev, stream))
    return out


PREFIX_WORKLOAD = ("prefix_cache_stream_bf16: 512 requests = shared 1000-token system prompt + "
                   "100-token question, new tokens U[22,356]; budget 2048, chunk 512, <= 256 "
                   "running; 64/8 heads, d 128; vocab 8192")


def run_prefix_cache(args, dev, stream) -> dict:
    """The prefix-cache scenario of "Inference engine core techniques" 3.3:
    requests share a 1000-token system prompt and add a 100-token question.
    The same stream runs through the serving loop with the prefix cache off
    and on; reported per run: prefill tokens computed, prompt tokens served
    from the cache, wall time, query tokens/s, and the time to first token
    (from the stream's start, all requests queued at once)."""
    import torch
    from paged_kv_cache_176_gb300.serving import ServingLoop

    vocab = 8192
    g = np.random.default_rng(args.seed + 11)
    system = g.integers(0, vocab, size=1000).tolist()
    reqs = [(system + g.integers(0, vocab, size=100).tolist(), int(g.integers(22, 357)))
            for _ in range(512)]

    def make(cache):
        return ServingLoop(65536, 64, 8, 128, dtype=torch.bfloat16, token_budget=2048,
                           chunk_size=512, max_running=256, max_context=1100 + 356 + 16,
                           device=dev, seed=args.seed, stream=stream, vocab=vocab,
                           prefix_cache=cache)

    def run(cache, rq):
        loop = make(cache)
        for rid, (p, n) in enumerate(rq):
            loop.submit(rid, len(p), n, tokens=p)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        evs, toks = [], []
        t0 = time.perf_counter()
        while True:
            p = loop.step()
            if p is None:
                break
            ev = torch.cuda.Event(enable_timing=True)
            ev.record(stream)
            evs.append(ev)
            toks.append(p.num_tokens)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
        assert int(loop.status.item()) == 0
        st = loop.sched.stats()
        assert st["finished"] == len(rq)
        ttft = sorted(e0.elapsed_time(evs[k]) for k in loop.first_token_step.values())
        res = {"prefix_cache": cache, "steps": len(toks), "wall_s": round(wall, 4),
               "query_tokens_per_s": round(sum(toks) / wall, 1),
               "requests_per_s": round(len(rq) / wall, 1),
               "prefill_tokens": st["prefill_tokens"], "cached_prompt_tokens":
               loop.sched.cached_tokens, "decode_tokens": st["decode_tokens"],
               "ttft_ms_mean": round(sum(ttft) / len(ttft), 3),
               "ttft_ms_p50": round(ttft[len(ttft) // 2], 3)}
        del loop
        torch.cuda.empty_cache()
        return res

    run(True, reqs[:16])  # warm-up
    off, on = run(False, reqs), run(True, reqs)
    prompt = sum(len(p) for p, _ in reqs)
    return {"workload": PREFIX_WORKLOAD, "prompt_tokens": prompt, "cache_off": off, "cache_on": on,
            "prefill_saved_frac": round(1 - on["prefill_tokens"] / off["prefill_tokens"], 4),
            "wall_speedup": round(off["wall_s"] / on["wall_s"], 3)}


def run_cow_step(args, dev, stream, reps: int = 200) -> dict:
    """The copy-on-write step of the shared-prefix workload: each request's
    last prompt block (12 filled slots) is copied for two of its three
    replies (512 pairs) and the 768 new tokens are written. Fused
    (pa_reshape_and_cache_cow: one launch, filled slots only) against the
    separate pa_copy_blocks (whole blocks) + pa_reshape_and_cache."""
    import torch
    import paged_kv_cache_176_gb300 as pa
    from paged_kv_cache_176_gb300 import workloads as W
    from paged_kv_cache_176_gb300.serving import pa_copy_blocks, pa_reshape_and_cache_cow

    w = W.shared_prefix_decode(seed=args.seed)
    R, rep = w.info["num_requests"], w.info["replies"]
    prompt = 1100
    j, ntok = prompt // 16, prompt % 16
    bt = w.block_tables
    src = [int(bt[r * rep + rep - 1, j]) for r in range(R) for _ in range(rep - 1)]
    dst = [int(bt[r * rep + k, j]) for r in range(R) for k in range(rep - 1)]
    tok = 2 * w.num_kv_heads * w.head_dim * w.k_pool.element_size()
    fused_bytes = 2 * len(src) * ntok * tok + 2 * w.num_seqs * tok + 8 * w.num_seqs + 12 * len(src)
    with torch.cuda.stream(stream):
        kp, vp = w.k_pool.to(dev), w.v_pool.to(dev)
        kn, vn, sm = w.k_new.to(dev), w.v_new.to(dev), w.slot_mapping.to(dev)
        d_src = torch.tensor(src, dtype=torch.int32, device=dev)
        d_dst = torch.tensor(dst, dtype=torch.int32, device=dev)
        d_n = torch.full((len(src),), ntok, dtype=torch.int32, device=dev)

    def fused():
        pa_reshape_and_cache_cow(kp, vp, kn, vn, sm, d_src, d_dst, d_n, stream=stream)

    def separate():
        pa_copy_blocks(kp, vp, d_src, d_dst, stream=stream)
        pa.pa_reshape_and_cache(kp, vp, kn, vn, sm, stream=stream)

    def timed(fn):
        for _ in range(10):
            fn()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / reps * 1e3

    us_f, us_s = timed(fused), timed(separate)
    pk = peaks()
    gbs = fused_bytes / (us_f * 1e-6) / 1e9
    del kp, vp
    torch.cuda.empty_cache()
    return {"workload": f"shared-prefix copy-on-write step: {len(src)} pairs x {ntok} filled slots "
                        f"+ {w.num_seqs} new tokens, 8 KV heads, d 128, bf16",
            "fused_us": round(us_f, 2), "separate_us": round(us_s, 2),
            "fused_bytes": fused_bytes, "fused_gbs": round(gbs, 1),
            "fused_hbm_frac": round(gbs / pk["hbm_gbs"], 4), "launches_fused": 1,
            "launches_separate": 2}


def gather_ceiling(w, kp, vp, dev, stream, stages: int = 3, reps: int = 50) -> dict:
    """The decode batch's blocks streamed with the decode kernel's copies and
    stage ring and no compute (include/pa_probe.h): what HBM and the block
    gather allow on this pool, against which the decode kernel's own time
    shows how much is spent on the SMs."""
    import torch
    import paged_kv_cache_176_gb300 as pa

    ids = [int(w.block_tables[s, j]) for s in range(w.num_seqs)
           for j in range((int(w.context_lens[s]) + 15) // 16)]
    blocks = torch.tensor(ids, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(5):
        pa.abi.pa_gather_probe(kp, vp, blocks, stages=stages, d_status=st, stream=stream)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        pa.abi.pa_gather_probe(kp, vp, blocks, stages=stages, d_status=st, stream=stream)
    b.record(stream)
    torch.cuda.synchronize(dev)
    assert int(st.item()) == 0
    us = a.elapsed_time(b) / reps * 1e3
    nbytes = 2 * len(ids) * kp[0].numel() * kp.element_size()
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"us": round(us, 2), "bytes": nbytes, "gbs": round(gbs, 1),
            "frac_of_copy_peak": round(gbs / peaks()["hbm_gbs"], 4), "stages": stages}


def run_decode_workload(name: str, w, dev, stream, reps: int = 30, groups=None,
                        siblings=None) -> dict:
    """One decode step (KV write when the workload has one, then pa_decode, or
    pa_decode_cascade when ``groups`` = (cu_groups, prefix_lens) is given, or
    pa_decode_cascade_nested when ``siblings`` = (cu_siblings, sibling_lens)
    is given as well) on another workload, timed with CUDA events on its
    stream; GB/s over the logical K/V bytes (every sequence's context) and over
    the unique bytes (each physical block's filled slots counted once). A
    cascade also reports GB/s over the bytes it has to read: each group's
    prefix once, each sibling entry's shared tokens after that prefix once, and
    every sequence's tokens after what it shares."""
    import torch
    import paged_kv_cache_176_gb300 as pa

    tok = 2 * w.num_kv_heads * w.head_dim * w.k_pool.element_size()
    ctx = w.context_lens.tolist()
    bt = w.block_tables.tolist()
    filled = {}
    for s, c in enumerate(ctx):
        for j in range((c + 15) // 16):
            filled[bt[s][j]] = max(filled.get(bt[s][j], 0), min(16, c - 16 * j))
    logical = sum(ctx) * tok
    unique = sum(filled.values()) * tok
    cascade_bytes = None
    if groups is not None:
        cu, pl = groups
        skip = [0] * len(ctx)  # first-level prefix tokens of each sequence
        for g in range(len(pl)):
            for s in range(cu[g], cu[g + 1]):
                skip[s] = pl[g]
        own = [ctx[s] - skip[s] for s in range(len(ctx))]
        cascade_bytes = sum(pl) * tok
        if siblings is not None:
            # entries of 16 / G members on the tensor-core decode (8 KV heads, bf16)
            G = w.num_q_heads // w.num_kv_heads
            per = 16 // G if (w.num_kv_heads == 8 and w.k_pool.element_size() == 2
                              and w.head_dim <= 128) else 1
            scu, sl = siblings
            for j in range(len(sl)):
                for a in range(scu[j], scu[j + 1], per):
                    cascade_bytes += (sl[j] - skip[a]) * tok
                for s in range(scu[j], scu[j + 1]):
                    own[s] = ctx[s] - sl[j]
        cascade_bytes += sum(own) * tok
    with torch.cuda.stream(stream):
        d = {k: (None if getattr(w, k) is None else getattr(w, k).to(dev))
             for k in ("k_pool", "v_pool", "q", "context_lens", "block_tables", "k_new", "v_new",
                       "slot_mapping")}
        out = torch.empty_like(d["q"])
        if siblings is not None:
            nbytes = pa.pa_decode_cascade_nested_workspace_size(
                w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.max_blocks_per_seq)
        else:
            size = pa.pa_decode_cascade_workspace_size if groups else pa.pa_decode_workspace_size
            nbytes = size(w.num_seqs, w.num_q_heads, w.head_dim, w.max_blocks_per_seq)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        if groups is not None:
            d_cu = torch.tensor(groups[0], dtype=torch.int32, device=dev)
            d_pl = torch.tensor(groups[1], dtype=torch.int32, device=dev)
        if siblings is not None:
            d_scu = torch.tensor(siblings[0], dtype=torch.int32, device=dev)
            d_sl = torch.tensor(siblings[1], dtype=torch.int32, device=dev)

    def step():
        if d["slot_mapping"] is not None:
            pa.pa_reshape_and_cache(d["k_pool"], d["v_pool"], d["k_new"], d["v_new"],
                                    d["slot_mapping"], stream=stream)
        if groups is None:
            pa.pa_decode(out, d["q"], d["k_pool"], d["v_pool"], d["block_tables"],
                         d["context_lens"], w.scale, workspace=ws, stream=stream)
        elif siblings is None:
            pa.pa_decode_cascade(out, d["q"], d["k_pool"], d["v_pool"], d["block_tables"],
                                 d["context_lens"], d_cu, d_pl, w.scale, workspace=ws,
                                 stream=stream)
        else:
            pa.pa_decode_cascade_nested(out, d["q"], d["k_pool"], d["v_pool"],
                                        d["block_tables"], d["context_lens"], d_cu, d_pl, d_scu,
                                        d_sl, w.scale, workspace=ws, stream=stream)

    for _ in range(5):
        step()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b) / reps
    pk = peaks()
    res = {"workload": name, "ms_per_step": round(ms, 4),
           "logical_kv_gbs": round(logical / (ms * 1e-3) / 1e9, 1),
           "unique_kv_gbs": round(unique / (ms * 1e-3) / 1e9, 1),
           "unique_hbm_frac": round(unique / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
           "logical_kv_bytes": logical, "unique_kv_bytes": unique,
           "attention_tokens_per_s": round(w.num_seqs / (ms * 1e-3), 1)}
    if cascade_bytes is not None:
        gbs = cascade_bytes / (ms * 1e-3) / 1e9
        res.update(cascade_kv_bytes=cascade_bytes, cascade_kv_gbs=round(gbs, 1),
                   cascade_hbm_frac=round(gbs / pk["hbm_gbs"], 4))
    del d, out, ws
    torch.cuda.empty_cache()
    return res


def build_record() -> dict:
    """Whether the libpa.so this run loaded matches these sources and this
    machine (the build is redone on any other)."""
    from paged_kv_cache_176_gb300.build import build_record as rec
    return rec()


MIXED_WORKLOAD: list = []


def run_mixed(args, dev, stream) -> dict:
    import torch
    import paged_kv_cache_176_gb300 as pa
    from paged_kv_cache_176_gb300 import workloads as W

    w = W.mixed_step(seed=args.seed)
    MIXED_WORKLOAD[:] = [w]  # kept for the oracle sample after the GPU legs
    work = mixed_work(w)
    with torch.cuda.stream(stream):
        d = {k: getattr(w, k).to(dev) for k in ("k_pool", "v_pool", "q", "cu_q_lens",
                                               "context_lens", "block_tables", "k_new", "v_new",
                                               "slot_mapping")}
        out = torch.empty_like(d["q"])
        ws = torch.empty(pa.pa_mixed_workspace_size(w.num_seqs, w.num_tokens, w.num_q_heads,
                                                    w.head_dim, w.max_blocks_per_seq),
                         dtype=torch.uint8, device=dev)

    def step():
        pa.pa_mixed_step(out, d["q"], d["cu_q_lens"], d["context_lens"], d["block_tables"],
                         d["k_pool"], d["v_pool"], w.scale, w.token_budget, k_new=d["k_new"],
                         v_new=d["v_new"], slot_mapping=d["slot_mapping"], workspace=ws,
                         stream=stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    step()
    torch.cuda.synchronize(dev)
    one = time.perf_counter() - t0
    n = max(3, min(args.mixed_steps, int(10.0 / max(one, 1e-4))))
    def timed(fn, reps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / reps

    ms = timed(step, n)
    # the two slices on their own (each with its own KV write): sequences
    # 0 .. nd-1 are the decode rows, the rest the prefill chunks
    cu = w.cu_q_lens.tolist()
    nd = sum(1 for i in range(w.num_seqs) if cu[i + 1] - cu[i] == 1)
    S, T = w.num_seqs, w.num_tokens

    def sub(lo, hi):
        t0, t1 = cu[lo], cu[hi]
        cu_sub = (d["cu_q_lens"][lo:hi + 1] - t0).contiguous()

        def run():
            pa.pa_mixed_step(out[t0:t1], d["q"][t0:t1], cu_sub, d["context_lens"][lo:hi],
                             d["block_tables"][lo:hi], d["k_pool"], d["v_pool"], w.scale,
                             w.token_budget, k_new=d["k_new"][t0:t1], v_new=d["v_new"][t0:t1],
                             slot_mapping=d["slot_mapping"][t0:t1], workspace=ws, stream=stream)
        return run

    for f in (sub(0, nd), sub(nd, S)):
        for _ in range(3):
            f()
    ms_dec = timed(sub(0, nd), n)
    ms_pf = timed(sub(nd, S), n)
    pk = peaks()
    tflops = work["prefill_flops"] / (ms * 1e-3) / 1e12
    t_hbm = work["decode_bytes"] / (pk["hbm_gbs"] * 1e9) * 1e3
    t_tc = work["prefill_flops"] / (pk["bf16_tflops_sustained"] * 1e12) * 1e3
    pf_tflops = work["prefill_flops"] / (ms_pf * 1e-3) / 1e12
    return {
        "workload": "mixed_step_bf16: budget 2048 = 128 decode (ctx U[1024,8192]) + prefill "
                    "512/512/512/384 at 512-aligned offsets of 32768-token prompts; 64/8 heads, d 128",
        "steps": n,
        "ms_per_step": round(ms, 4),
        "tokens_per_s": round(w.num_tokens / (ms * 1e-3), 1),
        "prefill_tflops_step": round(tflops, 2),
        "tensor_frac_step": round(tflops / pk["bf16_tflops_sustained"], 4),
        "decode_gbs_step": round(work["decode_bytes"] / (ms * 1e-3) / 1e9, 1),
        "prefill_flops": work["prefill_flops"],
        "decode_bytes": work["decode_bytes"],
        "prefill_slice_ms": round(ms_pf, 4),
        "prefill_slice_tflops": round(pf_tflops, 2),
        "prefill_slice_tensor_frac": round(pf_tflops / pk["bf16_tflops_sustained"], 4),
        "prefill_slice_frac_of_spec": round(pf_tflops / SPEC_BF16_TFLOPS, 4),
        "decode_slice_ms": round(ms_dec, 4),
        "decode_slice_gbs": round(work["decode_bytes"] / (ms_dec * 1e-3) / 1e9, 1),
        "ideal_step_ms": round(max(t_hbm, t_tc), 4),
        "step_frac": round(max(t_hbm, t_tc) / ms, 4),
        "note": "ideal_step_ms = max(decode bytes / measured HBM peak, prefill FLOPs / measured "
                "sustained bf16 peak); slices timed alone, each with its own KV write",
    }


SERVING_WORKLOAD = ("serving_stream_bf16: 1024 requests, prompt U[512,4096], new tokens "
                    "U[22,356]; budget 2048, chunk 512, <= 256 running; 64/8 heads, d 128; "
                    "pool 65536 blocks")


def serving_requests(seed: int, n: int, prompt=(512, 4096), new=(22, 356)):
    g = np.random.default_rng(seed + 7)
    return [(int(g.integers(prompt[0], prompt[1] + 1)), int(g.integers(new[0], new[1] + 1)))
            for _ in range(n)]


def run_serving(args, dev, stream) -> dict:
    """Continuous batching through the native scheduler and pa_mixed_step:
    the whole loop (host planning, one pinned plan copy per step, CoW block
    copies, the fused KV write and the attention) from the first request to
    the last token. Throughput counts query tokens (prefill + decode)."""
    import torch
    from paged_kv_cache_176_gb300.serving import ServingLoop

    def make():
        return ServingLoop(65536, 64, 8, 128, dtype=torch.bfloat16, token_budget=2048,
                           chunk_size=512, max_running=256, max_context=4096 + 512, device=dev,
                           seed=args.seed, stream=stream, fresh_inputs=False)

    # warm-up stream, every step checked: packed tables and the paging bound
    loop = make()
    for rid, (pl, nn) in enumerate(serving_requests(args.seed + 1, 48)):
        loop.submit(rid, pl, nn)
    waste_max = 0
    while True:
        p = loop.step()
        if p is None:
            break
        S = p.num_seqs
        held = (p.tables >= 0).sum(axis=1)
        ctx = p.context_lens[:S].astype(np.int64)
        assert np.all(held == (ctx + 15) // 16)
        waste_max = max(waste_max, int((held * 16 - ctx).max()))
    torch.cuda.synchronize(dev)
    assert int(loop.status.item()) == 0 and loop.bm.num_free == 65536
    del loop

    reqs = serving_requests(args.seed, 1024)
    loop = make()
    for rid, (pl, nn) in enumerate(reqs):
        loop.submit(rid, pl, nn)
    torch.cuda.synchronize(dev)
    evs, toks, used = [], [], []
    e0 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    t0 = time.perf_counter()
    while True:
        p = loop.step()
        if p is None:
            break
        ev = torch.cuda.Event(enable_timing=True)
        ev.record(stream)
        evs.append(ev)
        toks.append(p.num_tokens)
        used.append(loop.bm.num_blocks - loop.bm.num_free)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t0
    assert int(loop.status.item()) == 0
    st = loop.sched.stats()
    assert st["finished"] == len(reqs)
    dev_s = e0.elapsed_time(evs[-1]) * 1e-3
    total = sum(toks)
    # steady state: from the first to the last step that filled the budget
    full = [i for i, t in enumerate(toks) if t == 2048]
    i0, i1 = full[0], full[-1]
    steady_s = evs[i0].elapsed_time(evs[i1]) * 1e-3 if i1 > i0 else float("nan")
    steady_tok = sum(toks[i0 + 1:i1 + 1])
    return {
        "workload": SERVING_WORKLOAD,
        "steps": len(toks),
        "wall_s": round(wall, 4),
        "tokens_per_s": round(total / wall, 1),
        "device_tokens_per_s": round(total / dev_s, 1),
        "steady_tokens_per_s": round(steady_tok / steady_s, 1),
        "steady_steps": i1 - i0,
        "prefill_tokens": st["prefill_tokens"],
        "decode_tokens": st["decode_tokens"],
        "decode_tokens_per_s": round(st["decode_tokens"] / wall, 1),
        "mean_tokens_per_step": round(total / len(toks), 1),
        "peak_blocks_in_use": max(used),
        "h2d_plan_bytes_per_step": round(loop.h2d_bytes / len(toks), 1),
        "max_waste_tokens_per_seq": waste_max,
    }


# ------------------------------------------------------------------ oracle arm


class OracleRunner:
    """The fp64 oracle, as it stands, on the decode workload: each call runs
    the KV write of the step's tokens and the attention of the next ``k``
    sequences (cycling through the batch) and returns the seconds taken and
    the algorithmic bytes covered, in the GPU arm's accounting."""

    def __init__(self, seed: int):
        import oracle
        from paged_kv_cache_176_gb300 import workloads as W
        self.oracle = oracle
        self.lib = oracle.load()
        self.w = W.decode_b64(seed=seed)
        self.kp, self.vp = self.w.k_pool.clone(), self.w.v_pool.clone()
        self.cores = os.cpu_count() or 1
        self.nb = step_bytes(self.w)
        self.tok_bytes = 2 * self.w.num_kv_heads * self.w.head_dim * self.w.k_pool.element_size()
        self.next = 0

    def run(self, k: int):
        import numpy as np
        w = self.w
        k = max(1, min(k, w.num_seqs))
        idx = [(self.next + i) % w.num_seqs for i in range(k)]
        self.next = (self.next + k) % w.num_seqs
        mask = np.zeros(w.num_seqs, dtype=np.uint8)
        mask[idx] = 1
        sm = w.slot_mapping.clone()
        sm[torch_tensor_bool(mask == 0)] = -1  # write only the sampled sequences' tokens
        t0 = time.perf_counter()
        self.oracle.reshape_and_cache(self.kp, self.vp, w.k_new, w.v_new, sm, lib=self.lib)
        self.oracle.paged_attention(w.q, self.kp, self.vp, w.cu_q_lens, w.context_lens,
                                    w.block_tables, w.scale, row_mask=mask,
                                    num_threads=self.cores, lib=self.lib)
        secs = time.perf_counter() - t0
        ctx = int(w.context_lens[idx].long().sum())
        frac = k / w.num_seqs
        nbytes = ctx * self.tok_bytes + frac * (self.nb["step"] - self.nb["kv_read"])
        return secs, nbytes, k


def torch_tensor_bool(a):
    import torch
    return torch.from_numpy(a.astype(bool))


def mixed_cpu_baseline(w, seed: int) -> dict:
    """The fp64 oracle, as it stands, on a bounded sample of the mixed step:
    every decode row and 8 seeded rows of each prefill chunk (all heads, the
    step's KV write included); its FLOP rate over those rows, counted as the
    GPU arm counts the prefill (4·d per unmasked query-key pair)."""
    import numpy as np
    import oracle
    cu = w.cu_q_lens.tolist()
    ctx = w.context_lens.tolist()
    rng = np.random.default_rng(seed + 11)
    mask = np.zeros(w.num_tokens, dtype=np.uint8)
    flops = 0
    for s in range(w.num_seqs):
        ql = cu[s + 1] - cu[s]
        rows = [cu[s]] if ql == 1 else sorted(rng.choice(np.arange(cu[s], cu[s + 1]), 8, replace=False))
        for r in rows:
            mask[r] = 1
            keys = ctx[s] - ql + (r - cu[s]) + 1
            flops += 4 * w.num_q_heads * w.head_dim * keys
    cores = os.cpu_count() or 1
    lib = oracle.load()
    t0 = time.perf_counter()
    oracle.workload_attention(w, row_mask=mask, num_threads=cores, lib=lib)
    secs = time.perf_counter() - t0
    return {"value": round(flops / secs / 1e9, 2), "unit": "GFLOP/s", "cores": cores,
            "kind": "oracle", "rows": int(mask.sum()), "flops": int(flops),
            "seconds": round(secs, 2),
            "sample": f"every decode row and 8 seeded rows of each prefill chunk "
                      f"({int(mask.sum())} of {w.num_tokens} query rows, all heads)"}


def cpu_baseline(seed: int, budget_s: float) -> dict:
    """Oracle throughput on whole passes over the decode batch, repeated until
    about ``budget_s`` seconds of CPU work."""
    r = OracleRunner(seed)
    secs = nbytes = 0.0
    passes = 0
    while secs < budget_s or passes == 0:
        s, b, _ = r.run(r.w.num_seqs)
        secs += s
        nbytes += b
        passes += 1
    return {"value": round(nbytes / secs / 1e9, 3), "unit": "GB/s", "cores": r.cores,
            "kind": "oracle",
            "sample": f"{passes} full pass(es) over the decode batch (KV write of 64 tokens + "
                      f"attention of 64 sequences, {r.nb['kv_read'] / 1e6:.0f} MB of K/V each), "
                      f"{secs:.1f} s of CPU time"}


def run_reference(args, rank: int, world: int) -> dict | None:
    """The oracle as the reference arm: each step a bounded sample of the
    decode workload, sized so the whole run stays within a few minutes."""
    if rank != 0:
        return None
    r = OracleRunner(args.seed)
    s1, _, _ = r.run(1)  # calibrate: seconds per sequence
    per_step = min(args.ref_budget_s, 150.0 / (args.steps + args.warmup))
    k = max(1, min(r.w.num_seqs, int(per_step / max(s1, 1e-6))))
    for _ in range(args.warmup):
        r.run(k)
    secs = nbytes = 0.0
    for _ in range(args.steps):
        s, b, _ = r.run(k)
        secs += s
        nbytes += b
    v = nbytes / secs / 1e9
    sample = (f"per step: KV write + attention of {k} of the {r.w.num_seqs} decode sequences "
              f"(cycling), fp64 on {r.cores} host threads")
    return {
        "impl": "reference",
        "metric": "paged-decode attention HBM GB/s (% of peak) and mixed-step tokens/s on 1 GB300",
        "value": round(v, 3), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1), bf16-rounded; no dataset)",
        "config": {"workload": "decode_b64_bf16: 64 seqs, ctx U[512,4096], 32/8 heads, d 128, "
                               "block 16, pool 20000 shuffled blocks, + KV write of 64 tokens",
                   "sample_seqs_per_step": k},
        "cpu_baseline": {"value": round(v, 3), "unit": "GB/s", "cores": r.cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(v, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--mixed-steps", type=int, default=200)
    ap.add_argument("--skip-mixed", action="store_true")
    ap.add_argument("--skip-extra", action="store_true",
                    help="skip the wide-head GQA and shared-prefix decode measurements")
    ap.add_argument("--only-mixed", action="store_true",
                    help="run only the mixed step (profiling); prints its measurement")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--skip-serving", action="store_true",
                    help="skip the continuous-batching serving-loop measurement")
    ap.add_argument("--only-serving", action="store_true",
                    help="run only the serving-loop measurement (1 GPU)")
    ap.add_argument("--only-extra", action="store_true",
                    help="run only the other decode workloads (1 GPU)")
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--ref-budget-s", type=float, default=8.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as tdist
        backend = "gloo" if args.impl == "reference" else "nccl"
        if args.impl != "reference":
            import torch
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        tdist.init_process_group(backend)
    if (args.only_mixed or args.only_serving or args.only_extra) and args.impl != "reference":
        import torch
        dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
        torch.cuda.set_device(dev)
        st = torch.cuda.Stream(dev)
        if args.only_serving:
            res = {"serving_loop": run_serving(args, dev, st),
                   "prefix_cache": run_prefix_cache(args, dev, st)}
        else:
            res = (run_mixed if args.only_mixed else run_extra)(args, dev, st)
    elif args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_gpu(args, rank, world)
        if res is not None and rank == 0 and not args.skip_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(args.seed, args.cpu_budget_s)
            if "mixed_step" in res and MIXED_WORKLOAD:
                res["mixed_step"]["cpu_baseline"] = mixed_cpu_baseline(MIXED_WORKLOAD[0], args.seed)
    if world > 1:
        import torch.distributed as tdist
        tdist.barrier()
        tdist.destroy_process_group()
    if rank == 0 and res is not None:
        print(json.dumps(res))


if __name__ == "__main__":
    main()
