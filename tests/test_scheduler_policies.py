"""Scheduler policies beyond FIFO, on both the oracle and the C++ scheduler.

* PrefillFirst ("Continuous batching architecture", PrefillFirst): running
  prefills, then new prompts, then decodes with what is left of the budget;
  rows still emitted decodes first.
* A cap on prefill rows per step.
* The long-prefill cap (vLLM performance post, request-parallel prefill):
  at most ``max_long_prefills`` long prompts in their prefill phase at once;
  a long waiting prompt held by it is skipped, so shorter prompts behind it
  are not held up.

Pins: three traces derived by hand (tests/golden/scheduler_policy_traces.json);
invariants of each rule on random traces (oracle); the C++ scheduler equals
the oracle bit for bit on random traces under random policies and caps.
"""
import json
import os

import numpy as np
import pytest

from tests.sched_driver import oracle_from_config, run_trace
from tests.test_oracle_scheduler import _random_trace
from tests.test_scheduler_parity import c_from_config

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "scheduler_policy_traces.json")


def _traces():
    with open(GOLDEN) as f:
        return json.load(f)["traces"]


@pytest.mark.parametrize("impl", ["oracle", "c"])
@pytest.mark.parametrize("trace", _traces(), ids=lambda t: t["name"])
def test_hand_derived_policy_trace(trace, impl):
    make = oracle_from_config if impl == "oracle" else c_from_config
    s = make(trace["config"])
    got = run_trace(s, trace["requests"], len(trace["steps"]))
    for i, (g, e) in enumerate(zip(got, trace["steps"])):
        for k, v in e.items():
            assert g[k] == v, f"step {i}: {k} {g[k]} != {v}"
    free = list(s.free) if impl == "oracle" else s.free
    assert free == trace["final_free_list"]


def _policy_trace(seed):
    cfg, reqs = _random_trace(seed)
    rng = np.random.default_rng(1000 + seed)
    cfg["policy"] = int(rng.integers(0, 2))
    cfg["max_prefill_reqs"] = int(rng.choice([0, 0, 1, 2, 3]))
    cfg["long_prefill_tokens"] = int(rng.choice([0, 0, 5, 10, 20]))
    cfg["max_long_prefills"] = int(rng.choice([0, 1, 1, 2]))
    return cfg, reqs


@pytest.mark.parametrize("seed", range(40))
def test_policy_invariants_random_traces(seed):
    cfg, reqs = _policy_trace(seed)
    s = oracle_from_config(cfg)
    reqs = sorted(reqs, key=lambda r: r["arrival_step"])
    lt, mlp, mpr = cfg["long_prefill_tokens"], cfg["max_long_prefills"], cfg["max_prefill_reqs"]
    added = 0
    for step in range(80):
        while added < len(reqs) and reqs[added]["arrival_step"] <= step:
            r = reqs[added]
            s.add_request(r["id"], r["prompt_len"], r["output_len"])
            added += 1
        decoding_before = [r.req_id for r in s.running if r.state == "decoding"]
        prefilling_before = [r.req_id for r in s.running if r.state == "prefilling"]
        st = s.schedule_step()
        nd = st["num_decodes"]
        ids = [int(x) for x in st["req_ids"]]
        qlens = np.diff(st["cu_seqlens_q"])
        assert qlens.sum() <= cfg["max_batch_tokens"]
        assert len(ids) <= cfg["max_requests_per_batch"]
        assert (qlens[:nd] == 1).all()
        if mpr:
            assert len(ids) - nd <= mpr
        if lt:
            long_pref = [r for r in s.running if r.state == "prefilling" and r.prompt_len > lt]
            long_in_batch = [rid for rid in ids[nd:] if s.requests[rid].prompt_len > lt]
            # new long admissions only while the cap allowed them
            fresh_long = [rid for rid in long_in_batch if rid not in prefilling_before]
            already = len([rid for rid in prefilling_before if s.requests[rid].prompt_len > lt])
            assert already + len(fresh_long) <= max(mlp, already)
            del long_pref
        if cfg["policy"] == 1 and st["status"] == 0:
            # PrefillFirst: a decode is left out only if the prefills used the
            # budget or request cap or it stalled on blocks
            left = [rid for rid in decoding_before if rid not in ids[:nd]]
            if left:
                stalled = set(int(x) for x in st["stalled_ids"])
                assert (qlens.sum() == cfg["max_batch_tokens"] or
                        len(ids) == cfg["max_requests_per_batch"] or
                        all(rid in stalled for rid in left) or
                        any(rid in stalled for rid in decoding_before))
        if st["status"] == 0:
            s.step_done()
        # blocks are conserved
        held = sum(len(r.blocks) for r in s.running)
        assert held + len(s.free) == cfg["num_blocks"]


@pytest.mark.parametrize("seed", range(40))
def test_c_matches_oracle_policy_random_traces(seed):
    cfg, reqs = _policy_trace(seed)
    a = run_trace(oracle_from_config(cfg), reqs, 60)
    b = run_trace(c_from_config(cfg), reqs, 60)
    assert a == b
