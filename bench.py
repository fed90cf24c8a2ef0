#!/usr/bin/env python3
"""Benchmark: attention tokens/s of one continuous-batching step.

Workload (default ``mixed_2048``): the mixed chunked-prefill step -- 96 decode
requests (contexts U[256, 8192]), one prefill in flight on its second 1024-
token chunk (prompt 3000), new prompts U[64, 1024] filling a 2048-token
budget; 32 query / 8 KV heads, head_dim 128, bf16, 16-token blocks, a 65,536-
block pool with permuted physical blocks.  One step = cb_kv_append of the
step's new K/V + cb_paged_attention over the whole mixed batch.

JSON line keys (rank 0):
  value        tokens of the step / time of append+attention, inputs resident
               in HBM (KV read per step 1.7 GB >> 129 MB L2, so no flush).
  e2e          the same step through the public API with host buffers: C
               scheduler call, metadata + q/k/v host->device from pinned
               memory, append + attention, output device->host.
  roofline     the dominant kernel (split-KV decode): algorithmic bytes per
               launch / its CUDA-event duration, against measured HBM peak.
  prefill      the prefill-chunk kernel: algorithmic FLOPs / duration.
  cpu_baseline the CPU oracle on a bounded sample of the same step.

``--impl reference`` times the CPU oracle instead (bounded sample per step).
Multi-GPU: one process per GPU (torchrun), each an independent replica of
the workload (requests shard across GPUs with no exchange): weak scaling.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch of the
# decode kernel per workload, with the digest of the decode kernel's sources
# the capture was taken on (DECODE_SOURCES); the bench reports the figure
# only while the sources still have that digest, else null.
DECODE_SOURCES = ["decode_attention.cuh", "decode_launch.cuh", "decode_launch.h", "decode_bf16.cu",
                  "device_utils.cuh"]
DECODE_TRAFFIC = {
    # 1,716,311,808 B read + 7,330,304 B written (algorithmic 1,714,053,120 B)
    "mixed_2048": {"bytes": 1716311808 + 7330304, "sha16": "1cd717f935e971dd"},
    # 566,313,472 B read + 5,258,752 B written (algorithmic 564,916,224 B)
    "decode_64": {"bytes": 566313472 + 5258752, "sha16": "1cd717f935e971dd"},
}


def decode_sources_sha16():
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "paged_attention_continuous_gb300", "csrc")
    for name in DECODE_SOURCES:
        with open(os.path.join(d, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def decode_traffic(workload):
    """(bytes, digest) of the last capture for this workload if it was taken
    on the current decode sources, else (None, digest of the capture)."""
    rec = DECODE_TRAFFIC.get(workload)
    if rec is None:
        return None, None
    return (rec["bytes"] if rec["sha16"] == decode_sources_sha16() else None), rec["sha16"]


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------- work models
def decode_bytes(step, Hq, Hkv, D, elem, window=0):
    """Algorithmic bytes of the decode rows: each K and V row the query sees
    (all of them, or the last ``window``) read once per KV head, plus q read
    and out written."""
    nd = step["num_decodes"]
    seq = np.asarray(step["seq_lens"][:nd], dtype=np.int64)
    if window > 0:
        seq = np.minimum(seq, window)
    return int(seq.sum() * Hkv * D * 2 * elem + nd * Hq * D * 2 * elem)


def prefill_flops(step, Hq, D, window=0):
    """Algorithmic FLOPs of the prefill rows: 2*D for q.k and 2*D for p.v per
    unmasked (query, key) pair and query head (query position p sees p + 1
    keys, or min(p + 1, window))."""
    nd = step["num_decodes"]
    cu = np.asarray(step["cu_seqlens_q"], dtype=np.int64)
    seq = np.asarray(step["seq_lens"], dtype=np.int64)
    pairs = 0
    for r in range(nd, step["num_reqs"]):
        n = int(cu[r + 1] - cu[r])
        start = int(seq[r]) - n
        if window > 0:
            pairs += int(np.minimum(np.arange(start + 1, start + n + 1), window).sum())
        else:
            pairs += n * start + n * (n + 1) // 2
    return int(4 * D * Hq * pairs)


def append_bytes(step, Hkv, D, elem):
    return int(step["num_tokens"] * Hkv * D * 2 * elem * 2)


# ---------------------------------------------------------- the workload
def build_scenario(name, seed=0):
    return workloads.SCENARIOS[name](seed=seed)


def rank_scenario(name, rank):
    """Requests are independent, so ranks shard them with no exchange: each
    rank serves its own request set, drawn with seed = rank (weak scaling)."""
    return build_scenario(name, seed=rank)


def reduce_over_ranks(dist, value, op, device):
    """One float reduced over all ranks (timing MAX, token SUM)."""
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=op)
    return float(t.item())


def load_c_scheduler(cb, sc):
    s = cb.Scheduler(block_size=sc.block_size, num_blocks=sc.num_blocks,
                     max_batch_tokens=sc.max_batch_tokens,
                     max_requests_per_batch=sc.max_requests_per_batch,
                     max_blocks_per_seq=sc.max_blocks_per_seq,
                     max_prefill_chunk=sc.max_prefill_chunk, safety_margin=sc.safety_margin,
                     free_list=sc.free_list)
    for r in sc.running:
        s.add_running_request(r.req_id, r.prompt_len, r.output_len, r.num_cached)
    for w in sc.waiting:
        s.add_request(w.req_id, w.prompt_len, w.output_len)
    return s


def _sub_step(step, lo, hi):
    """Host metadata of rows [lo, hi) as a stand-alone step."""
    cu = np.asarray(step["cu_seqlens_q"])
    sub = dict(step)
    sub["num_reqs"] = hi - lo
    sub["cu_seqlens_q"] = (cu[lo:hi + 1] - cu[lo]).astype(np.int32)
    sub["seq_lens"] = np.asarray(step["seq_lens"])[lo:hi]
    sub["block_tables"] = np.asarray(step["block_tables"])[lo:hi]
    sub["slot_mapping"] = np.asarray(step["slot_mapping"])[cu[lo]:cu[hi]]
    sub["num_tokens"] = int(cu[hi] - cu[lo])
    sub["num_decodes"] = max(0, min(step["num_decodes"], hi) - lo)
    sub["max_q_len"] = int(np.diff(sub["cu_seqlens_q"]).max(initial=1))
    sub["max_seq_len"] = int(np.max(sub["seq_lens"], initial=1))
    return sub


def time_each(torch, fn, iters, stream):
    """Sum of per-launch device times: an event pair around every call, so
    host-side gaps between calls are not counted."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(iters)]
    torch.cuda.synchronize()
    for a, b in evs:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / 1e3


def time_median(torch, fn, iters, stream):
    """Median per-launch device time (an event pair around every call)."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(iters)]
    torch.cuda.synchronize()
    for a, b in evs:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return float(np.median([a.elapsed_time(b) for a, b in evs])) / 1e3


def time_loop(torch, fn, iters, stream):
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(iters):
        fn()
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / 1e3  # seconds


def attn_call(cb, torch, dev, sc, sub, q, out, kc, vc, ws):
    """A closure calling cb_paged_attention on a stand-alone step ``sub``
    whose query rows are ``q``; metadata is uploaded once, here."""
    if sub["num_reqs"] == 0:
        return None
    cu = torch.from_numpy(np.asarray(sub["cu_seqlens_q"], dtype=np.int32)).to(dev)
    sl = torch.from_numpy(np.asarray(sub["seq_lens"], dtype=np.int32)).to(dev)
    bt = torch.from_numpy(np.ascontiguousarray(sub["block_tables"], dtype=np.int32)).to(dev)

    def f():
        cb.paged_attention(q, kc, vc, cu, sl, bt, num_decodes=sub["num_decodes"],
                           max_q_len=sub["max_q_len"], max_seq_len=sub["max_seq_len"],
                           scale=sc.softmax_scale, workspace=ws, out=out)
    return f


def _runner_for(sc, dev, torch):
    from paged_attention_continuous_gb300.step import StepRunner
    runner = StepRunner(num_blocks=sc.num_blocks, num_q_heads=sc.num_q_heads,
                        num_kv_heads=sc.num_kv_heads, head_dim=sc.head_dim, dtype=sc.dtype,
                        max_reqs=sc.max_requests_per_batch, max_tokens=sc.max_batch_tokens,
                        max_blocks_per_seq=sc.max_blocks_per_seq, zero_cache=False)
    runner.k_cache[0].copy_(workloads.cache_fill(sc.num_blocks, sc.num_kv_heads, sc.block_size,
                                                 sc.head_dim, seed=1234, dtype=sc.dtype,
                                                 scale=sc.value_scale, device=dev))
    runner.v_cache[0].copy_(workloads.cache_fill(sc.num_blocks, sc.num_kv_heads, sc.block_size,
                                                 sc.head_dim, seed=1235, dtype=sc.dtype,
                                                 scale=sc.value_scale, device=dev))
    return runner


def _qkv(sc, T, dev, step=0):
    seeds = [workloads.step_seed(sc.seed, step, 0, w) for w in range(3)]
    mk = lambda n, s_: workloads.token_tensors(T, n, sc.head_dim, seed=s_, dtype=sc.dtype,
                                               scale=sc.value_scale, device=dev)
    return mk(sc.num_q_heads, seeds[0]), mk(sc.num_kv_heads, seeds[1]), mk(sc.num_kv_heads, seeds[2])


def measure_decode_only(cb, torch, dev, reps, hbm):
    """Decode-only step: 64 requests, contexts U[128, 4096], 32/8 heads,
    D = 128, 20,000-block pool.  Decode kernel GB/s vs HBM peak."""
    sc = workloads.decode_64()
    sched = load_c_scheduler(cb, sc)
    step = sched.schedule_step()
    runner = _runner_for(sc, dev, torch)
    T = step["num_tokens"]
    q, k, v = _qkv(sc, T, dev)
    out = torch.empty_like(q)
    ds = runner.upload(step)
    kc, vc = runner.k_cache[0], runner.v_cache[0]
    runner.run(ds, q, k, v, out=out)
    f = attn_call(cb, torch, dev, sc, step, q, out, kc, vc, runner.workspace)
    for _ in range(5):
        f()
    t = time_each(torch, f, reps, torch.cuda.current_stream()) / reps
    nbytes = decode_bytes(step, sc.num_q_heads, sc.num_kv_heads, sc.head_dim, 2)
    assert runner.workspace.read_errors() == 0
    gbs = nbytes / t / 1e9
    del runner
    torch.cuda.empty_cache()
    return {"workload": "decode_64 (64 decodes, ctx U[128,4096], 32Q/8KV, D=128)",
            "kernel": "decode_kernel", "achieved_gbs": round(gbs, 1), "peak_gbs": hbm,
            "frac": round(gbs / hbm, 4), "ms_per_launch": round(t * 1e3, 4),
            "algorithmic_bytes_per_launch": nbytes, "launches_timed": reps}


def measure_long_prompt(cb, torch, dev, reps, hbm, bf16, bf16s):
    """Long-prompt interleave: a 32,768-token prompt prefilled in 512-token
    chunks over 64 scheduler steps while 128 requests decode (64 Q / 8 KV
    heads, D = 128, budget 640).  Every step's append + attention is timed,
    and its prefill and decode launches separately (median of the reps of
    each step)."""
    sc = workloads.long_prompt_32k()
    sched = load_c_scheduler(cb, sc)
    runner = _runner_for(sc, dev, torch)
    kc, vc = runner.k_cache[0], runner.v_cache[0]
    ws = runner.workspace
    stream = torch.cuda.current_stream()
    q, k, v = _qkv(sc, sc.max_batch_tokens, dev)
    out = torch.empty_like(q)
    tot = {"tokens": 0, "t_step": 0.0, "t_pre": 0.0, "t_dec": 0.0, "flops": 0, "bytes": 0}
    per_step = []
    worst = None     # (step, TFLOP/s) of the slowest prefill chunk
    steps = 0
    while steps < 64:
        st = sched.schedule_step()
        if st["status"] != 0 or st["num_reqs"] == 0:
            break
        T, R, nd = st["num_tokens"], st["num_reqs"], st["num_decodes"]
        ds = runner.upload(st)
        qs, ks, vs, os_ = q[:T], k[:T], v[:T], out[:T]
        full = lambda: runner.run(ds, qs, ks, vs, out=os_)
        dsub, psub = _sub_step(st, 0, nd), _sub_step(st, nd, R)
        fd = attn_call(cb, torch, dev, sc, dsub, q[:nd], out[:nd], kc, vc, ws)
        fp = attn_call(cb, torch, dev, sc, psub, q[nd:T], out[nd:T], kc, vc, ws)
        full()
        if fd:
            fd()
        if fp:
            fp()
        t_step = time_median(torch, full, reps, stream)
        t_dec = time_median(torch, fd, reps, stream) if fd else 0.0
        t_pre = time_median(torch, fp, reps, stream) if fp else 0.0
        fl = prefill_flops(st, sc.num_q_heads, sc.head_dim)
        by = decode_bytes(st, sc.num_q_heads, sc.num_kv_heads, sc.head_dim, 2)
        tot["tokens"] += T; tot["t_step"] += t_step; tot["t_pre"] += t_pre
        tot["t_dec"] += t_dec; tot["flops"] += fl; tot["bytes"] += by
        if t_pre:
            tf = fl / t_pre / 1e12
            if worst is None or tf < worst[1]:
                worst = (steps, tf)
        if steps in (0, 16, 32, 48, 63):
            per_step.append({"step": steps, "chunk_start": int(st["seq_lens"][-1]) - int(
                np.diff(st["cu_seqlens_q"])[-1]), "prefill_tflops": round(fl / t_pre / 1e12, 1) if t_pre else 0,
                "decode_gbs": round(by / t_dec / 1e9, 1) if t_dec else 0,
                "ms_step": round(t_step * 1e3, 4)})
        sched.step_done()
        steps += 1
    assert ws.read_errors() == 0
    del runner
    torch.cuda.empty_cache()
    pt = tot["flops"] / tot["t_pre"] / 1e12 if tot["t_pre"] else 0.0
    dg = tot["bytes"] / tot["t_dec"] / 1e9 if tot["t_dec"] else 0.0
    return {"workload": "long_prompt_32k (32K prompt in 512-token chunks, 128 decodes, 64Q/8KV, D=128)",
            "steps": steps, "tokens_per_s": round(tot["tokens"] / tot["t_step"], 1),
            "ms_per_step": round(tot["t_step"] / max(steps, 1) * 1e3, 4),
            "prefill": {"kernel": "prefill_kernel (tcgen05)", "achieved_tflops": round(pt, 1),
                        "peak_tflops": bf16, "frac": round(pt / bf16, 4),
                        "frac_sustained": round(pt / bf16s, 4),
                        "algorithmic_flops": int(tot["flops"]),
                        "ms_total": round(tot["t_pre"] * 1e3, 3),
                        "slowest_chunk": {"step": worst[0], "tflops": round(worst[1], 1),
                                          "frac": round(worst[1] / bf16, 4)} if worst else None},
            "decode": {"kernel": "decode_kernel", "achieved_gbs": round(dg, 1), "peak_gbs": hbm,
                       "frac": round(dg / hbm, 4)},
            "sampled_steps": per_step, "reps_per_step": reps}


TRACE_DESC = "trace_2000 (2,000 requests, Poisson(20) arrivals, lognormal lengths, " \
             "4 layers x 65,536 blocks, 32Q/8KV, D=128, budget 8192 / 256 reqs)"


def scheduler_for(cb, sc):
    """The C scheduler configured from every option a workload sets."""
    return cb.Scheduler(block_size=sc.block_size, num_blocks=sc.num_blocks,
                        max_batch_tokens=sc.max_batch_tokens,
                        max_requests_per_batch=sc.max_requests_per_batch,
                        max_blocks_per_seq=sc.max_blocks_per_seq,
                        max_prefill_chunk=sc.max_prefill_chunk, safety_margin=sc.safety_margin,
                        free_list=sc.free_list, policy=sc.policy, offload=sc.offload,
                        swap_blocks=sc.swap_blocks, prefix_caching=sc.prefix_caching,
                        sliding_window=sc.sliding_window)


def measure_trace(cb, torch, dev, hbm, bf16, max_steps=20000, graphs=False, sc=None,
                  desc=TRACE_DESC):
    """A request trace run until every request has finished (by default the
    2,000-request trace: Poisson(20) arrivals per step, lognormal prompt /
    output lengths with medians 512 / 128, 4 layers each with its own
    65,536-block pool, budget 8,192 tokens and 256 requests per step).  Per
    step: the host scheduler call (timed on the host), the step's offload
    swaps and metadata upload (timed with CUDA events when the step has
    swaps), and per layer the step's fresh q/k/v (drawn per (step, layer),
    untimed) then append + attention (timed with CUDA events).  Reports
    whole-trace tokens/s, the additive roofline fraction (decode bytes / HBM
    peak + prefill FLOPs / tensor peak, over the measured kernel time) and
    the KV-block fragmentation (slots allocated but not yet holding a token,
    over all allocated slots, mean over steps).  With ``graphs`` every step
    (all layers) is one CUDA-graph replay of its padded bucket
    (GraphStepRunner); q/k/v are copied into its static buffers outside the
    timed replay."""
    from paged_attention_continuous_gb300.step import GraphStepRunner, StepRunner
    sc = workloads.trace_2000() if sc is None else sc
    s = scheduler_for(cb, sc)
    Runner = GraphStepRunner if graphs else StepRunner
    runner = Runner(num_blocks=sc.num_blocks, num_q_heads=sc.num_q_heads,
                    num_kv_heads=sc.num_kv_heads, head_dim=sc.head_dim, dtype=sc.dtype,
                    max_reqs=sc.max_requests_per_batch, max_tokens=sc.max_batch_tokens,
                    max_blocks_per_seq=sc.max_blocks_per_seq, num_layers=sc.num_layers,
                    device=dev, swap_blocks=sc.swap_blocks, sliding_window=sc.sliding_window)
    W = sc.sliding_window
    events = []
    swap_events = []
    swap_bytes = 0
    t_host = 0.0
    tokens = 0
    d_bytes = 0
    p_flops = 0
    frag = []
    finished = 0
    nxt = 0
    step = 0
    stalled_steps = 0
    while finished < len(sc.waiting) and step < max_steps:
        while nxt < len(sc.waiting) and sc.waiting[nxt].arrival_step <= step:
            w = sc.waiting[nxt]
            if w.tokens is not None:
                s.add_request(w.req_id, w.prompt_len, w.output_len, tokens=w.tokens)
            else:
                s.add_request(w.req_id, w.prompt_len, w.output_len)
            nxt += 1
        h0 = time.perf_counter()
        st = s.schedule_step()
        t_host += time.perf_counter() - h0
        has_swaps = len(st["swap_in"]) + len(st["swap_out"]) > 0
        if has_swaps:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
        if st["status"] != 0 or st["num_reqs"] == 0:
            swap_bytes += runner.apply_swaps(st)
            if has_swaps:
                e1.record()
                swap_events.append((e0, e1))
            if st["status"] == 0:
                s.step_done()
            stalled_steps += 1
            step += 1
            continue
        T = st["num_tokens"]
        if has_swaps:
            swap_bytes += (len(st["swap_in"]) + len(st["swap_out"])) * runner.swap.block_bytes * \
                2 * sc.num_layers
        if graphs:
            key, _ = runner.prepare(st)
        else:
            ds = runner.upload(st)
        if has_swaps:
            e1.record()
            swap_events.append((e0, e1))
        for layer in range(sc.num_layers):
            sd = [workloads.step_seed(sc.seed, step, layer, c) for c in range(3)]
            q = workloads.token_tensors(T, sc.num_q_heads, sc.head_dim, seed=sd[0], dtype=sc.dtype,
                                        scale=sc.value_scale, device=dev)
            k = workloads.token_tensors(T, sc.num_kv_heads, sc.head_dim, seed=sd[1], dtype=sc.dtype,
                                        scale=sc.value_scale, device=dev)
            v = workloads.token_tensors(T, sc.num_kv_heads, sc.head_dim, seed=sd[2], dtype=sc.dtype,
                                        scale=sc.value_scale, device=dev)
            if graphs:
                runner.q_buf[layer][:T].copy_(q)
                runner.k_buf[layer][:T].copy_(k)
                runner.v_buf[layer][:T].copy_(v)
                continue
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            runner.run(ds, q, k, v, layer=layer)
            e1.record()
            events.append((e0, e1))
        if graphs:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            runner.run(key)
            e1.record()
            events.append((e0, e1))
        h0 = time.perf_counter()
        finished += len(s.step_done())
        t_host += time.perf_counter() - h0
        tokens += T
        d_bytes += sc.num_layers * decode_bytes(st, sc.num_q_heads, sc.num_kv_heads, sc.head_dim, 2,
                                                W)
        p_flops += sc.num_layers * prefill_flops(st, sc.num_q_heads, sc.head_dim, W)
        sl = np.asarray(st["seq_lens"], dtype=np.int64)
        alloc = ((sl + sc.block_size - 1) // sc.block_size) * sc.block_size
        frag.append(float((alloc - sl).sum() / max(alloc.sum(), 1)))
        step += 1
    torch.cuda.synchronize()
    t_dev = sum(a.elapsed_time(b) for a, b in events) / 1e3
    t_swap = sum(a.elapsed_time(b) for a, b in swap_events) / 1e3
    assert runner.workspace.read_errors() == 0
    if runner.swap is not None:
        assert runner.swap.read_errors() == 0
    n_graphs = len(runner.graphs) if graphs else 0
    hits = s.prefix_stats()[0]
    del runner
    torch.cuda.empty_cache()
    t_roof = d_bytes / (hbm * 1e9) + p_flops / (bf16 * 1e12)
    extra = {}
    if sc.offload:
        # the swaps of this small trace are a few blocks per step: their
        # region time is launch latency; the bandwidth is measure_swap's
        extra["offload"] = {"swap_bytes": int(swap_bytes), "steps_with_swaps": len(swap_events),
                            "ms_swap_and_upload_regions": round(t_swap * 1e3, 3)}
    if sc.prefix_caching:
        extra["prefix_hit_tokens"] = int(hits)
        extra["prompt_tokens"] = int(sum(w.prompt_len for w in sc.waiting))
    if W:
        extra["sliding_window"] = W
    return {"graphs": n_graphs if graphs else None,
            "workload": desc, **extra,
            "steps": step, "steps_without_batch": stalled_steps, "finished": finished,
            "tokens": int(tokens),
            "tokens_per_s_device": round(tokens / t_dev, 1) if t_dev else 0.0,
            "tokens_per_s_with_host_scheduler": round(tokens / (t_dev + t_host), 1),
            "ms_device_total": round(t_dev * 1e3, 2), "ms_host_scheduler_total": round(t_host * 1e3, 2),
            "decode_bytes": int(d_bytes), "prefill_flops": int(p_flops),
            "roofline_frac_additive": round(t_roof / t_dev, 4) if t_dev else 0.0,
            "fragmentation_mean": round(float(np.mean(frag)) if frag else 0.0, 4),
            "timed": "per layer: cb_kv_append + cb_paged_attention (CUDA events); "
                     "scheduler calls on the host; q/k/v generation untimed"}


def measure_swap(cb, torch, dev, reps=5):
    """cb_kv_swap over the CPU-GPU link: 256 blocks of every layer's K and V
    of a 32-layer model (8 KV heads x 16 tokens x 128 dims bf16 = 32 KB per
    block and pool, 64 pools: 512 MiB per direction) moved from the device
    caches to the pinned swap pool and back, against one contiguous
    cudaMemcpyAsync of the same byte count (the copy engine) each way."""
    layers, nb, n = 32, 512, 256
    shape = (8, 16, 128)
    devp = [torch.empty((nb,) + shape, dtype=torch.bfloat16, device=dev) for _ in range(2 * layers)]
    hostp = [torch.empty((n,) + shape, dtype=torch.bfloat16, pin_memory=True)
             for _ in range(2 * layers)]
    blocks = torch.randperm(nb, device=dev)[:n].to(torch.int32)
    slots = torch.arange(n, dtype=torch.int32, device=dev)
    ew = torch.zeros(1, dtype=torch.int32, device=dev)
    nbytes = n * 2 * layers * devp[0][0].numel() * 2
    stream = torch.cuda.current_stream()
    out = lambda: cb.kv_swap(devp, hostp, blocks, slots, error_word=ew)
    back = lambda: cb.kv_swap(hostp, devp, slots, blocks, error_word=ew)
    hbuf = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    dbuf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d2h = lambda: hbuf.copy_(dbuf, non_blocking=True)
    h2d = lambda: dbuf.copy_(hbuf, non_blocking=True)
    res = {}
    for name, f in (("swap_out", out), ("swap_in", back), ("memcpy_d2h", d2h), ("memcpy_h2d", h2d)):
        f()
        f()
        # best of three rounds: a transfer over the CPU-GPU link can be
        # slowed by other traffic on the host
        t = min(time_each(torch, f, reps, stream) for _ in range(3)) / reps
        res[name + "_gbs"] = round(nbytes / t / 1e9, 1)
    torch.cuda.synchronize()
    assert int(ew.item()) == 0
    del devp, hostp, hbuf, dbuf
    torch.cuda.empty_cache()
    return {"kernel": "kv_swap_kernel", "bytes_per_direction": int(nbytes),
            "workload": "256 blocks x 64 pools (32 layers K and V, 32 KB blocks)", **res,
            "frac_of_memcpy_out": round(res["swap_out_gbs"] / res["memcpy_d2h_gbs"], 3),
            "frac_of_memcpy_in": round(res["swap_in_gbs"] / res["memcpy_h2d_gbs"], 3),
            "launches_timed": reps}


def measure_window_decode(cb, torch, dev, reps, hbm):
    """Decode on sliding-window layers: 256 requests with contexts
    U[2048, 32768] attending the last 4,096 tokens (32 Q / 8 KV heads,
    D = 128, bf16); block tables hold -1 before each window (recycled
    pages), so only window pages exist.  Decode kernel GB/s vs HBM peak."""
    rng = np.random.default_rng(7)
    R, W, Hq, Hkv, D = 256, 4096, 32, 8, 128
    L = rng.integers(2048, 32768, size=R, endpoint=True)
    first = np.maximum(L - W, 0) // 16
    pages = (L + 15) // 16
    nb = int((pages - first).sum())
    perm = rng.permutation(nb).astype(np.int32)
    Wmax = int(pages.max())
    bt = np.full((R, Wmax), -1, dtype=np.int32)
    o = 0
    for r in range(R):
        k = int(pages[r] - first[r])
        bt[r, first[r]:pages[r]] = perm[o:o + k]
        o += k
    kc = workloads.cache_fill(nb, Hkv, 16, D, seed=31, dtype="bf16", scale=0.5, device=dev)
    vc = workloads.cache_fill(nb, Hkv, 16, D, seed=32, dtype="bf16", scale=0.5, device=dev)
    q = workloads.token_tensors(R, Hq, D, seed=33, dtype="bf16", scale=0.5, device=dev)
    out = torch.empty_like(q)
    ws = cb.Workspace(R, Hq, Hkv, D, device=dev)
    cu = torch.arange(R + 1, dtype=torch.int32, device=dev)
    sl = torch.from_numpy(L.astype(np.int32)).to(dev)
    btd = torch.from_numpy(bt).to(dev)
    f = lambda: cb.paged_attention(q, kc, vc, cu, sl, btd, num_decodes=R, max_q_len=1,
                                   max_seq_len=int(L.max()), scale=1 / math.sqrt(D), workspace=ws,
                                   out=out, sliding_window=W)
    for _ in range(5):
        f()
    t = time_each(torch, f, reps, torch.cuda.current_stream()) / reps
    assert ws.read_errors() == 0
    nbytes = decode_bytes({"num_decodes": R, "seq_lens": L}, Hq, Hkv, D, 2, W)
    gbs = nbytes / t / 1e9
    del kc, vc, ws
    torch.cuda.empty_cache()
    return {"workload": "256 decodes, ctx U[2048,32768], window 4096, 32Q/8KV, D=128",
            "kernel": "decode_kernel (window)", "achieved_gbs": round(gbs, 1), "peak_gbs": hbm,
            "frac": round(gbs / hbm, 4), "ms_per_launch": round(t * 1e3, 4),
            "algorithmic_bytes_per_launch": int(nbytes), "launches_timed": reps}


def measure_prefix(cb, torch, dev, hbm, bf16):
    """The shared-system-prompt trace (48 requests over 4 system prompts of
    U[200, 1200] tokens plus U[16, 400]-token suffixes, 2 layers) with and
    without prefix caching: device time for the whole trace and the prompt
    tokens that were reused instead of recomputed."""
    import dataclasses
    sc = workloads.shared_prefix(0)
    desc = "shared_prefix (48 requests, 4 shared system prompts, 2 layers, 32Q/8KV)"
    on = measure_trace(cb, torch, dev, hbm, bf16, sc=sc, desc=desc)
    off = measure_trace(cb, torch, dev, hbm, bf16,
                        sc=dataclasses.replace(sc, prefix_caching=False), desc=desc)
    return {"workload": desc, "with_prefix_caching": on, "without": off,
            "device_time_ratio": round(off["ms_device_total"] / on["ms_device_total"], 3)
            if on["ms_device_total"] else None}


# ----------------------------------------------------------- CPU oracle
def oracle_sample(sc, step, pools_cpu, rows, prefill_token_cap=None):
    """Run the oracle on ``rows`` of ``step``: gather each row's cache blocks
    into its own float64 sub-pool, append the row's new K/V, attend (for a
    prefill row, optionally only its last ``prefill_token_cap`` queries).
    Returns (query tokens processed, seconds)."""
    from oracle import attention as oatt
    from oracle import paged_kv
    kp, vp, kn, vn, q = pools_cpu
    bs = sc.block_size
    cu = step["cu_seqlens_q"]
    t0 = time.perf_counter()
    ntok = 0
    for r in rows:
        a, b = int(cu[r]), int(cu[r + 1])
        L = int(step["seq_lens"][r])
        a2 = b - prefill_token_cap if (prefill_token_cap and b - a > prefill_token_cap) else a
        blocks = [int(x) for x in step["block_tables"][r] if x >= 0]
        sub_k = kp[blocks].astype(np.float64)
        sub_v = vp[blocks].astype(np.float64)
        table = np.arange(len(blocks))
        local = {blk: i for i, blk in enumerate(blocks)}
        slots = [local[int(s) // bs] * bs + int(s) % bs for s in step["slot_mapping"][a:b]]
        paged_kv.append(sub_k, sub_v, kn[a:b].astype(np.float64), vn[a:b].astype(np.float64),
                        np.asarray(slots), bs)
        K = oatt.gather_kv(sub_k, table, L, bs)
        V = oatt.gather_kv(sub_v, table, L, bs)
        oatt.attend_one_request(q[a2:b].astype(np.float64), K, V, L - (b - a2), sc.softmax_scale)
        ntok += b - a2
    return ntok, time.perf_counter() - t0


def choose_oracle_rows(step, budget_rows):
    nd = step["num_decodes"]
    R = step["num_reqs"]
    dec = list(np.linspace(0, nd - 1, num=min(nd, budget_rows), dtype=int)) if nd else []
    pre = list(range(nd, R))
    return sorted(set(int(x) for x in dec)), pre


def config_dict(sc, step, world):
    """The workload description both arms report (same keys and values)."""
    elem = 2 if sc.dtype == "bf16" else 4
    dbytes = decode_bytes(step, sc.num_q_heads, sc.num_kv_heads, sc.head_dim, elem)
    return {"workload": sc.name, "num_tokens": int(step["num_tokens"]),
            "num_reqs": int(step["num_reqs"]), "num_decodes": int(step["num_decodes"]),
            "q_heads": sc.num_q_heads, "kv_heads": sc.num_kv_heads,
            "head_dim": sc.head_dim, "block_size": sc.block_size,
            "num_blocks": sc.num_blocks, "max_batch_tokens": sc.max_batch_tokens,
            "l2": "inputs larger than L2 (decode KV %.2f GB per step), no flush" % (dbytes / 1e9),
            "parallelism": f"replicas x{world}"}


def measure_e2e(cb, torch, dev, sc, runner, rank, world, args):
    """The step end to end through the public C API with host buffers: one
    cb_executor_run_step per step -- the C scheduler call, pinned host ->
    device copies of the step's metadata and q/k/v, cb_kv_append +
    cb_paged_attention, and the device -> host copy of the output --
    double-buffered over copy-in / compute / copy-out streams.  The
    scheduler advances from the workload's first step.  The running
    requests are the workload's (long decodes and the in-flight prefill);
    its waiting prompts, and new prompts of the same length distribution
    (U[64, 1024] tokens) arriving so that four always wait, get 1-4 output
    tokens, so requests finish, the row cap never binds, and every step
    stays a budget-filled mix of about a hundred decodes and prefill chunks
    like the first.  Also reports the device-only rate of the same steps
    (the executor's CUDA events around each step's kernels)."""
    K = max(1, args.e2e_steps)
    rng = np.random.default_rng(4242 + rank)
    sched = cb.Scheduler(block_size=sc.block_size, num_blocks=sc.num_blocks,
                         max_batch_tokens=sc.max_batch_tokens,
                         max_requests_per_batch=sc.max_requests_per_batch,
                         max_blocks_per_seq=sc.max_blocks_per_seq,
                         max_prefill_chunk=sc.max_prefill_chunk, safety_margin=sc.safety_margin,
                         free_list=sc.free_list)
    for r in sc.running:
        sched.add_running_request(r.req_id, r.prompt_len, r.output_len, r.num_cached)
    for w in sc.waiting:
        sched.add_request(w.req_id, w.prompt_len, int(rng.integers(1, 5)))
    Tm = sc.max_batch_tokens
    ex = cb.Executor(runner.k_cache, runner.v_cache, num_q_heads=sc.num_q_heads,
                     max_reqs=sc.max_requests_per_batch, max_tokens=Tm,
                     max_blocks_per_seq=sc.max_blocks_per_seq, scale=sc.softmax_scale)
    mk = lambda h, seed: workloads.token_tensors(Tm, h, sc.head_dim, seed=seed, dtype=sc.dtype,
                                                  scale=sc.value_scale, device="cpu").pin_memory()
    hq, hk, hv = mk(sc.num_q_heads, 901), mk(sc.num_kv_heads, 902), mk(sc.num_kv_heads, 903)
    ho = torch.empty((Tm, sc.num_q_heads, sc.head_dim), dtype=hq.dtype, pin_memory=True)
    next_id = [10 ** 7]

    def top_up():
        waiting = sched.counts()[1]
        while waiting < 4:
            sched.add_request(next_id[0], int(rng.integers(64, 1025)), int(rng.integers(1, 5)))
            next_id[0] += 1
            waiting += 1

    for _ in range(3):
        top_up()
        ex.run_step(sched, hq, hk, hv, ho)
    ex.synchronize()
    ex.reset_stats()
    elem = hq.element_size()
    W = sc.max_blocks_per_seq
    h2d = d2h = 0
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(K):
        top_up()
        T, R = ex.run_step(sched, hq, hk, hv, ho)
        h2d += 4 * ((R + 1) + R + R * W + T) + T * (sc.num_q_heads + 2 * sc.num_kv_heads) * \
            sc.head_dim * elem
        d2h += T * sc.num_q_heads * sc.head_dim * elem
    ex.synchronize()
    t = time.perf_counter() - t0
    steps, toks, cms = ex.stats()
    assert ex.read_errors() == 0
    ex.close()
    tok_all, t_all, dev_s = float(toks), t, cms / 1e3
    if world > 1:
        dist = torch.distributed
        t_all = reduce_over_ranks(dist, t, dist.ReduceOp.MAX, dev)
        dev_s = reduce_over_ranks(dist, dev_s, dist.ReduceOp.MAX, dev)
        tok_all = reduce_over_ranks(dist, toks, dist.ReduceOp.SUM, dev)
    value = tok_all / t_all
    dev_value = tok_all / dev_s if dev_s else 0.0
    return {"value": round(value, 1), "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d / K), "d2h_bytes_per_step": int(d2h / K),
            "steps": int(steps), "tokens": int(toks),
            "device_value": round(dev_value, 1),
            "frac_of_device": round(value / dev_value, 4) if dev_value else None,
            "includes": "per step: cb_executor_run_step = cb_schedule_step + pinned H2D of the "
                        "step's metadata and q/k/v + cb_kv_append + cb_paged_attention + D2H of "
                        "the output + cb_step_done, double-buffered (copy-in / compute / "
                        "copy-out streams); the scheduler advances from the workload's first "
                        "step (prompts get 1-4 output tokens, arrivals keep four waiting, "
                        "steps stay budget-filled); timed from the first "
                        "call to the last output on the host; device_value = the same steps' "
                        "tokens / the sum of their kernel times (CUDA events)"}


# ----------------------------------------------------------------- main
def run_ours(args, rank, world):
    import torch
    import paged_attention_continuous_gb300 as cb
    from paged_attention_continuous_gb300.step import StepRunner

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    sc = rank_scenario(args.workload, rank)
    elem = 2 if sc.dtype == "bf16" else 4
    sched = load_c_scheduler(cb, sc)
    step = sched.schedule_step()
    assert step["status"] == 0
    T, R, nd = step["num_tokens"], step["num_reqs"], step["num_decodes"]
    # the kernel timings below use upload/run on the current stream; the
    # end-to-end loop runs the C step executor on the same caches afterwards
    runner = StepRunner(num_blocks=sc.num_blocks, num_q_heads=sc.num_q_heads,
                                 num_kv_heads=sc.num_kv_heads, head_dim=sc.head_dim,
                                 dtype=sc.dtype, max_reqs=sc.max_requests_per_batch,
                                 max_tokens=sc.max_batch_tokens,
                                 max_blocks_per_seq=sc.max_blocks_per_seq, zero_cache=False)
    # initial pool contents stand for K/V written by earlier steps
    runner.k_cache[0].copy_(workloads.cache_fill(sc.num_blocks, sc.num_kv_heads, sc.block_size,
                                                 sc.head_dim, seed=1234, dtype=sc.dtype,
                                                 scale=sc.value_scale, device=dev))
    runner.v_cache[0].copy_(workloads.cache_fill(sc.num_blocks, sc.num_kv_heads, sc.block_size,
                                                 sc.head_dim, seed=1235, dtype=sc.dtype,
                                                 scale=sc.value_scale, device=dev))
    seeds = [workloads.step_seed(sc.seed, 0, 0, w) for w in range(3)]
    q = workloads.token_tensors(T, sc.num_q_heads, sc.head_dim, seed=seeds[0], dtype=sc.dtype,
                                scale=sc.value_scale, device=dev)
    k = workloads.token_tensors(T, sc.num_kv_heads, sc.head_dim, seed=seeds[1], dtype=sc.dtype,
                                scale=sc.value_scale, device=dev)
    v = workloads.token_tensors(T, sc.num_kv_heads, sc.head_dim, seed=seeds[2], dtype=sc.dtype,
                                scale=sc.value_scale, device=dev)
    out = torch.empty_like(q)
    ds = runner.upload(step)
    stream = torch.cuda.current_stream()
    ws = runner.workspace
    kc, vc = runner.k_cache[0], runner.v_cache[0]

    def full_step():
        runner.run(ds, q, k, v, out=out)

    # decode-only and prefill-only views for per-kernel timing
    dstep = _sub_step(step, 0, nd)
    pstep = _sub_step(step, nd, R)

    def make_attn(sub, tok_lo):
        import torch as _t
        if sub["num_reqs"] == 0:
            return None
        cu = _t.from_numpy(np.asarray(sub["cu_seqlens_q"], dtype=np.int32)).to(dev)
        sl = _t.from_numpy(np.asarray(sub["seq_lens"], dtype=np.int32)).to(dev)
        bt = _t.from_numpy(np.ascontiguousarray(sub["block_tables"], dtype=np.int32)).to(dev)
        qs = q[tok_lo:tok_lo + sub["num_tokens"]]
        os_ = out[tok_lo:tok_lo + sub["num_tokens"]]

        def f():
            cb.paged_attention(qs, kc, vc, cu, sl, bt, num_decodes=sub["num_decodes"],
                               max_q_len=sub["max_q_len"], max_seq_len=sub["max_seq_len"],
                               scale=sc.softmax_scale, workspace=ws, out=os_)
        return f

    dec_fn = make_attn(dstep, 0)
    pre_fn = make_attn(pstep, nd)

    W, K = args.warmup, args.steps
    for _ in range(W):
        full_step()
        if dec_fn:
            dec_fn()
        if pre_fn:
            pre_fn()
    torch.cuda.synchronize()
    assert ws.read_errors() == 0

    if world > 1:
        torch.distributed.barrier()
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    t_step = time_loop(torch, full_step, K, stream)
    t_dec = time_each(torch, dec_fn, K, stream) if dec_fn else 0.0
    t_pre = time_each(torch, pre_fn, K, stream) if pre_fn else 0.0
    clk = clocks.stop()
    tokens_all = T
    if world > 1:
        dist = torch.distributed
        t_step = reduce_over_ranks(dist, t_step, dist.ReduceOp.MAX, dev)
        tokens_all = int(reduce_over_ranks(dist, T, dist.ReduceOp.SUM, dev))
        dist.barrier()
    assert ws.read_errors() == 0

    # ---- end to end through the public API: the C step executor
    e2e = measure_e2e(cb, torch, dev, sc, runner, rank, world, args)

    traffic, traffic_sha = decode_traffic(sc.name)
    pk, src = peaks()
    hbm = float(pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    bf16 = float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    bf16s = float(pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    dbytes = decode_bytes(step, sc.num_q_heads, sc.num_kv_heads, sc.head_dim, elem)
    pflops = prefill_flops(step, sc.num_q_heads, sc.head_dim)
    dec_s = t_dec / K if K else 0.0
    pre_s = t_pre / K if K else 0.0
    dec_gbs = dbytes / dec_s / 1e9 if dec_s else 0.0
    pre_tflops = pflops / pre_s / 1e12 if pre_s else 0.0
    step_s = t_step / K
    dec_launches = (nd + 1023) // 1024
    pre_launches = 1 if R > nd else 0
    launches = K * (1 + dec_launches + pre_launches) + K * dec_launches + K * pre_launches

    line = {
        "metric": "attention tokens/s per mixed step",
        "value": round(tokens_all / step_s, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(step_s * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": sc.dtype,
        "data": "synthetic (seeded N(0,1)*0.5 q/k/v, random-filled KV pool, permuted blocks)",
        "config": config_dict(sc, step, world),
        "e2e": e2e,
        "roofline": {"kernel": "decode_kernel (split-KV, bf16)", "bound": "hbm",
                     "achieved": round(dec_gbs, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(dec_gbs / hbm, 4), "peak_source": src,
                     "traffic": traffic, "traffic_capture_sha16": traffic_sha,
                     "kernel_sha16": decode_sources_sha16(),
                     "algorithmic_bytes_per_launch": dbytes,
                     "ms_per_launch": round(dec_s * 1e3, 4)},
        "prefill": {"kernel": "prefill rows", "bound": "tensor",
                    "achieved": round(pre_tflops, 2), "peak": bf16, "unit": "TFLOP/s",
                    "frac": round(pre_tflops / bf16, 4),
                    "frac_sustained": round(pre_tflops / bf16s, 4), "peak_source": src,
                    "algorithmic_flops_per_launch": pflops,
                    "ms_per_launch": round(pre_s * 1e3, 4)},
        "append": {"bytes_per_step": append_bytes(step, sc.num_kv_heads, sc.head_dim, elem)},
        "clocks": clk,
        "gpu_launches": int(launches),
    }
    if not args.no_extra and world == 1:
        line["decode_only"] = measure_decode_only(cb, torch, dev, max(K, 20), hbm)
        line["long_prompt"] = measure_long_prompt(cb, torch, dev, 5, hbm, bf16, bf16s)
        line["trace"] = measure_trace(cb, torch, dev, hbm, bf16)
        line["trace_graphs"] = measure_trace(cb, torch, dev, hbm, bf16, graphs=True)
        line["offload"] = {
            "swap": measure_swap(cb, torch, dev),
            "trace": measure_trace(cb, torch, dev, hbm, bf16, sc=workloads.offload_pressure(0),
                                   desc="offload_pressure (24 requests, 40-block pool, 8-block "
                                        "swap pool, 2 layers, 16Q/4KV)")}
        line["prefix_caching"] = measure_prefix(cb, torch, dev, hbm, bf16)
        line["sliding_window"] = {
            "decode": measure_window_decode(cb, torch, dev, max(K, 20), hbm),
            "trace": measure_trace(cb, torch, dev, hbm, bf16, sc=workloads.sliding_trace(0),
                                   desc="sliding_trace (32 requests, window 384, 512-block "
                                        "pool, 2 layers, 32Q/8KV)")}
    # compact copies of the fractions the targets are judged on
    fr = {"mixed_2048_decode_hbm": line["roofline"]["frac"],
          "mixed_2048_prefill_tensor": line["prefill"]["frac"]}
    if "decode_only" in line:
        fr["decode_64_hbm"] = line["decode_only"]["frac"]
        lp = line["long_prompt"]
        fr["long_prompt_decode_hbm"] = lp["decode"]["frac"]
        fr["long_prompt_prefill_tensor"] = lp["prefill"]["frac"]
        if lp["prefill"].get("slowest_chunk"):
            fr["long_prompt_slowest_chunk_tensor"] = lp["prefill"]["slowest_chunk"]["frac"]
        fr["window_decode_hbm"] = line["sliding_window"]["decode"]["frac"]
    fr["e2e_frac_of_device"] = line["e2e"].get("frac_of_device")
    items = list(line.items())
    k_at = [k for k, _ in items].index("prefill") + 1
    line = dict(items[:k_at] + [("fractions", fr)] + items[k_at:])
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(sc, step, runner, q, k, v, torch, dev,
                                            budget_s=args.cpu_seconds)
    return line


def _pristine_blocks(sc, blocks, dev, torch):
    kp = workloads.cache_fill(sc.num_blocks, sc.num_kv_heads, sc.block_size, sc.head_dim,
                              seed=1234, dtype=sc.dtype, scale=sc.value_scale, device=dev)
    vp = workloads.cache_fill(sc.num_blocks, sc.num_kv_heads, sc.block_size, sc.head_dim,
                              seed=1235, dtype=sc.dtype, scale=sc.value_scale, device=dev)
    sel = torch.tensor(blocks, dtype=torch.long, device=dev)
    k = kp.index_select(0, sel).float().cpu().numpy()
    v = vp.index_select(0, sel).float().cpu().numpy()
    del kp, vp
    return k, v


def oracle_setup(sc, step, rows, q, k, v, torch, dev):
    """The oracle's inputs for ``rows`` of ``step``: the pristine contents of
    the rows' cache blocks (a compact pool, tables remapped into it) and the
    step's q/k/v on the host."""
    blocks = sorted({int(b) for r in rows for b in step["block_tables"][r] if b >= 0})
    kpool, vpool = _pristine_blocks(sc, blocks, dev, torch)
    remap = {b: i for i, b in enumerate(blocks)}
    st = dict(step)
    bt = np.full_like(np.asarray(step["block_tables"]), -1)
    for r in rows:
        for c, b in enumerate(step["block_tables"][r]):
            if b >= 0:
                bt[r, c] = remap[int(b)]
    st["block_tables"] = bt
    st["slot_mapping"] = np.asarray([remap[int(s) // sc.block_size] * sc.block_size +
                                     int(s) % sc.block_size if (int(s) // sc.block_size) in remap
                                     else -1 for s in step["slot_mapping"]], dtype=np.int64)
    pools = (kpool, vpool, k.float().cpu().numpy(), v.float().cpu().numpy(), q.float().cpu().numpy())
    return st, pools


def cpu_threads():
    try:
        import threadpoolctl
        return max(p.get("num_threads", 1) for p in threadpoolctl.threadpool_info())
    except Exception:
        return os.cpu_count()


def cpu_baseline(sc, step, runner, q, k, v, torch, dev, budget_s=20.0, full=True):
    """The oracle, as it stands, timed on the host cores on the step's rows:
    all decode rows and all prefill rows, repeated until about ``budget_s``
    seconds have passed (``full``); or, when a whole pass would not fit the
    budget, a spread of decode rows plus each prefill row's last queries."""
    if full:
        dec_rows, pre_rows = list(range(step["num_decodes"])), list(range(step["num_decodes"],
                                                                          step["num_reqs"]))
    else:
        dec_rows, pre_rows = choose_oracle_rows(step, 16)
    rows = dec_rows + pre_rows
    st, pools = oracle_setup(sc, step, rows, q, k, v, torch, dev)
    if full:
        n_tot, t_tot, passes = 0, 0.0, 0
        while passes == 0 or t_tot < budget_s:
            n, t = oracle_sample(sc, st, pools, rows)
            n_tot += n; t_tot += t; passes += 1
        desc = (f"{sc.name} step 0: all {len(dec_rows)} decode rows and {len(pre_rows)} prefill rows "
                f"({n} query tokens) x {passes} passes, numpy float64")
    else:
        n, t = oracle_sample(sc, st, pools, dec_rows)
        cap = 64
        n2, t2 = oracle_sample(sc, st, pools, pre_rows, prefill_token_cap=cap)
        per_tok = t2 / max(n2, 1)
        room = max(budget_s - t, 0.05)
        cap = int(max(16, min(2048, room / max(per_tok, 1e-6) / max(len(pre_rows), 1))))
        n2, t2 = oracle_sample(sc, st, pools, pre_rows, prefill_token_cap=cap)
        n_tot, t_tot = n + n2, t + t2
        desc = (f"{sc.name} step 0: {len(dec_rows)} of {step['num_decodes']} decode rows "
                f"+ the last {cap} queries of each of {len(pre_rows)} prefill rows "
                f"({n_tot} query tokens), numpy float64")
    threads = cpu_threads()
    return {"value": round(n_tot / t_tot, 2), "unit": "tokens/s", "cores": int(threads),
            "host_cpus": os.cpu_count(), "kind": "oracle", "seconds": round(t_tot, 2),
            "sample": desc}


def run_reference(args, rank, world):
    """CPU oracle on the same workload, a bounded sample per step."""
    if rank != 0:
        return None
    import torch
    sc = build_scenario(args.workload)
    from oracle.scheduler import FifoScheduler
    o = FifoScheduler(block_size=sc.block_size, num_blocks=sc.num_blocks,
                      max_batch_tokens=sc.max_batch_tokens,
                      max_requests_per_batch=sc.max_requests_per_batch,
                      max_blocks_per_seq=sc.max_blocks_per_seq,
                      max_prefill_chunk=sc.max_prefill_chunk, safety_margin=sc.safety_margin,
                      free_list=sc.free_list)
    for r in sc.running:
        o.add_running_request(r.req_id, r.prompt_len, r.output_len, r.num_cached)
    for w in sc.waiting:
        o.add_request(w.req_id, w.prompt_len, w.output_len)
    step = o.schedule_step()
    step["max_q_len"] = int(np.diff(step["cu_seqlens_q"]).max())
    step["max_seq_len"] = int(step["seq_lens"].max())
    T = step["num_tokens"]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    seeds = [workloads.step_seed(sc.seed, 0, 0, w) for w in range(3)]
    q = workloads.token_tensors(T, sc.num_q_heads, sc.head_dim, seed=seeds[0], dtype=sc.dtype,
                                scale=sc.value_scale, device=dev)
    k = workloads.token_tensors(T, sc.num_kv_heads, sc.head_dim, seed=seeds[1], dtype=sc.dtype,
                                scale=sc.value_scale, device=dev)
    v = workloads.token_tensors(T, sc.num_kv_heads, sc.head_dim, seed=seeds[2], dtype=sc.dtype,
                                scale=sc.value_scale, device=dev)
    # The rows the cpu_baseline leg times (all of the step's).  A first,
    # untimed full pass sizes the per-step sample so that the K + W steps take
    # about --ref-seconds: the rows are dealt round-robin into n_parts groups
    # and step i runs group i mod n_parts.
    nd, R = step["num_decodes"], step["num_reqs"]
    rows = list(range(R))
    st, pools = oracle_setup(sc, step, rows, q, k, v, torch, dev)
    _, t_full = oracle_sample(sc, st, pools, rows)
    total = args.steps + args.warmup
    n_parts = max(1, min(R, int(np.ceil(t_full * total / max(args.ref_seconds, 1e-3)))))
    groups = [rows[i::n_parts] for i in range(n_parts)]
    tot_tok, tot_s = 0, 0.0
    for i in range(total):
        n, t = oracle_sample(sc, st, pools, groups[i % n_parts])
        if i >= args.warmup:
            tot_tok += n
            tot_s += t
    val = tot_tok / tot_s if tot_s else 0.0
    sample = (f"{sc.name} step 0: its {nd} decode and {R - nd} prefill rows dealt round-robin into "
              f"{n_parts} groups, one group per step (a full pass took {t_full:.2f} s), numpy float64")
    return {"impl": "reference", "metric": "attention tokens/s per mixed step",
            "value": round(val, 2), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(tot_s / max(args.steps, 1) * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "config": config_dict(sc, step, world),
            "cpu_baseline": {"kind": "oracle", "cores": int(cpu_threads()), "sample": sample,
                             "value": round(val, 2)},
            "e2e": {"value": round(val, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mixed_2048",
                    choices=["mixed_2048", "decode_64", "long_prompt_32k", "prefill_chunk_16k"])
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--ref-seconds", type=float, default=90.0,
                    help="reference arm: about this many seconds of oracle work in all")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the decode-only and long-prompt sub-measurements")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        # the CPU oracle: rank 0 alone runs it; other ranks exit without work
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    line = run_ours(args, rank, world)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
