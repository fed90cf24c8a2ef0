"""Drive a scheduler (the oracle or the C library) through a scenario and
collect every step's outputs as plain Python lists, so two schedulers can be
compared field by field."""
from __future__ import annotations

import numpy as np

FIELDS = ("status", "req_ids", "num_decodes", "cu_seqlens_q", "seq_lens",
          "block_tables", "slot_mapping", "stalled_ids", "stalled_demand", "swap_in", "swap_out")


def normalize(step: dict) -> dict:
    out = {}
    for k in FIELDS:
        v = step[k]
        if isinstance(v, np.ndarray):
            v = v.tolist()
        out[k] = v
    for k in ("swap_in", "swap_out"):
        out[k] = [list(map(int, p)) for p in out[k]]
    R = len(out["req_ids"])
    out["block_tables"] = [list(map(int, row)) for row in out["block_tables"]][:R]
    return out


def oracle_from_config(cfg: dict):
    from oracle.scheduler import FifoScheduler
    return FifoScheduler(block_size=cfg["block_size"], num_blocks=cfg["num_blocks"],
                         max_batch_tokens=cfg["max_batch_tokens"],
                         max_requests_per_batch=cfg["max_requests_per_batch"],
                         max_blocks_per_seq=cfg["max_blocks_per_seq"],
                         max_prefill_chunk=cfg["max_prefill_chunk"],
                         safety_margin=cfg["safety_margin"],
                         free_list=cfg.get("free_list"), policy=cfg.get("policy", 0),
                         max_prefill_reqs=cfg.get("max_prefill_reqs", 0),
                         long_prefill_tokens=cfg.get("long_prefill_tokens", 0),
                         max_long_prefills=cfg.get("max_long_prefills", 1),
                         offload=cfg.get("offload", False), swap_blocks=cfg.get("swap_blocks", 0),
                         prefix_caching=cfg.get("prefix_caching", False),
                         sliding_window=cfg.get("sliding_window", 0))


def run_trace(sched, requests, num_steps, arrivals=None):
    """requests: list of dicts {id, prompt_len, output_len[, arrival_step]}.
    Requests with arrival_step s are added before step s.  Returns a list of
    per-step dicts (normalize() fields plus 'finished')."""
    steps = []
    pending = sorted(requests, key=lambda r: r.get("arrival_step", 0))
    i = 0
    for s in range(num_steps):
        while i < len(pending) and pending[i].get("arrival_step", 0) <= s:
            r = pending[i]
            if r.get("tokens") is not None:
                sched.add_request(r["id"], r["prompt_len"], r["output_len"], tokens=r["tokens"])
            else:
                sched.add_request(r["id"], r["prompt_len"], r["output_len"])
            i += 1
        st = normalize(sched.schedule_step())
        if st["status"] == 0:
            st["finished"] = list(sched.step_done())
        else:
            st["finished"] = None
        steps.append(st)
    return steps


def scenario_to_config(sc) -> dict:
    return {"block_size": sc.block_size, "num_blocks": sc.num_blocks,
            "max_batch_tokens": sc.max_batch_tokens,
            "max_requests_per_batch": sc.max_requests_per_batch,
            "max_prefill_chunk": sc.max_prefill_chunk,
            "safety_margin": sc.safety_margin,
            "max_blocks_per_seq": sc.max_blocks_per_seq,
            "free_list": [int(x) for x in sc.free_list],
            "policy": sc.policy, "offload": sc.offload, "swap_blocks": sc.swap_blocks,
            "prefix_caching": sc.prefix_caching, "sliding_window": sc.sliding_window}


def c_from_config(cfg: dict):
    import paged_attention_continuous_gb300 as cb
    return cb.Scheduler(block_size=cfg["block_size"], num_blocks=cfg["num_blocks"],
                        max_batch_tokens=cfg["max_batch_tokens"],
                        max_requests_per_batch=cfg["max_requests_per_batch"],
                        max_blocks_per_seq=cfg["max_blocks_per_seq"],
                        max_prefill_chunk=cfg["max_prefill_chunk"],
                        safety_margin=cfg["safety_margin"], free_list=cfg.get("free_list"),
                        policy=cfg.get("policy", 0), max_prefill_reqs=cfg.get("max_prefill_reqs", 0),
                        long_prefill_tokens=cfg.get("long_prefill_tokens", 0),
                        max_long_prefills=cfg.get("max_long_prefills", 1),
                        offload=cfg.get("offload", False), swap_blocks=cfg.get("swap_blocks", 0),
                        prefix_caching=cfg.get("prefix_caching", False),
                        sliding_window=cfg.get("sliding_window", 0))


def load_scenario(sched, sc, up_to_step=None):
    """Load a workloads.Scenario: running requests first (in order), then the
    waiting requests whose arrival_step <= up_to_step (all if None)."""
    for r in sc.running:
        sched.add_running_request(r.req_id, r.prompt_len, r.output_len, r.num_cached)
    for w in sc.waiting:
        if up_to_step is None or w.arrival_step <= up_to_step:
            add_waiting(sched, w)


def add_waiting(sched, w):
    """Queue a workloads.WaitingRequest (with its token ids, if any)."""
    if w.tokens is not None:
        sched.add_request(w.req_id, w.prompt_len, w.output_len, tokens=w.tokens)
    else:
        sched.add_request(w.req_id, w.prompt_len, w.output_len)
