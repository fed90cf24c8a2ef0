"""Offloading and soft reset ("Continuous batching architecture", Offloading,
Soft reset) on the oracle and the C++ scheduler.

Pins: two traces derived by hand (tests/golden/scheduler_offload_traces.json:
one with a 4-block swap pool, one without, both triggers, swap-ins oldest
first, a resumed request spared in its step); invariants on random
memory-pressure traces (blocks and swap slots conserved, the last active
request never taken, every request still finishes with its output count);
the C++ scheduler equals the oracle bit for bit on those traces.
"""
import json
import os

import numpy as np
import pytest

from tests.sched_driver import oracle_from_config, run_trace
from tests.test_scheduler_parity import c_from_config

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "scheduler_offload_traces.json")


def _traces():
    with open(GOLDEN) as f:
        return json.load(f)["traces"]


@pytest.mark.parametrize("impl", ["oracle", "c"])
@pytest.mark.parametrize("trace", _traces(), ids=lambda t: t["name"])
def test_hand_derived_offload_trace(trace, impl):
    make = oracle_from_config if impl == "oracle" else c_from_config
    s = make(trace["config"])
    got = run_trace(s, trace["requests"], len(trace["steps"]))
    for i, (g, e) in enumerate(zip(got, trace["steps"])):
        for k, v in e.items():
            assert g[k] == v, f"step {i}: {k} {g[k]} != {v}"
    free = list(s.free) if impl == "oracle" else s.free
    assert free == trace["final_free_list"]


def _pressure_trace(seed):
    rng = np.random.default_rng(seed)
    bs = int(rng.choice([2, 4]))
    nb = int(rng.integers(4, 24))
    cfg = dict(block_size=bs, num_blocks=nb, max_batch_tokens=int(rng.integers(4, 30)),
               max_requests_per_batch=int(rng.integers(2, 8)),
               max_prefill_chunk=int(rng.choice([0, 0, 4])),
               safety_margin=float(rng.choice([0.0, 0.0, 0.1])), max_blocks_per_seq=64,
               free_list=[int(x) for x in rng.permutation(nb)],
               policy=int(rng.integers(0, 2)), offload=True,
               swap_blocks=int(rng.choice([0, 2, 6, 20])))
    reqs = []
    for i in range(int(rng.integers(2, 10))):
        # together the requests outgrow the pool (stalls and offloads); each
        # one alone fits it, else it could never finish
        p = int(rng.integers(1, 3 * bs))
        o = int(rng.integers(1, 4 * bs))
        o = max(1, min(o, nb * bs - p + 1))
        reqs.append(dict(id=200 + i, prompt_len=p, output_len=o,
                         arrival_step=int(rng.integers(0, 4))))
    return cfg, reqs


@pytest.mark.parametrize("seed", range(60))
def test_offload_invariants_random_pressure(seed):
    cfg, reqs = _pressure_trace(seed)
    s = oracle_from_config(cfg)
    reqs = sorted(reqs, key=lambda r: r["arrival_step"])
    outputs = {r["id"]: r["output_len"] for r in reqs}
    produced = {r["id"]: 0 for r in reqs}
    finished = set()
    added = 0
    for step in range(400):
        while added < len(reqs) and reqs[added]["arrival_step"] <= step:
            r = reqs[added]
            s.add_request(r["id"], r["prompt_len"], r["output_len"])
            added += 1
        active_before = len(s.running)
        st = s.schedule_step()
        # the last active request is never taken off
        if active_before >= 1:
            assert len(s.running) >= 1
        if st["status"] == 0:
            ids = [int(x) for x in st["req_ids"]]
            nd = st["num_decodes"]
            qlens = np.diff(st["cu_seqlens_q"])
            completes = [i >= nd and s.requests[rid].num_cached + int(qlens[i]) ==
                         s.requests[rid].prompt_len for i, rid in enumerate(ids)]
            fin = s.step_done()
            # one output token per decode row and per prompt completed
            for i, rid in enumerate(ids):
                if i < nd or completes[i]:
                    produced[rid] += 1
            finished.update(fin)
        # conservation of blocks and swap slots
        held = sum(len(r.blocks) for r in s.running)
        assert held + len(s.free) == cfg["num_blocks"]
        in_swap = sum(len(r.swap_slots) for r in s.swapped)
        assert in_swap + len(s.swap_free) == cfg["swap_blocks"]
        if added == len(reqs) and not s.running and not s.waiting and not s.swapped:
            break
    # every request finished, having produced exactly its output count (a
    # soft reset re-produces nothing: its generated tokens became prompt)
    assert finished == set(outputs)
    assert produced == outputs


@pytest.mark.parametrize("seed", range(60))
def test_c_matches_oracle_random_pressure(seed):
    cfg, reqs = _pressure_trace(seed)
    a = run_trace(oracle_from_config(cfg), reqs, 200)
    b = run_trace(c_from_config(cfg), reqs, 200)
    assert a == b


@pytest.mark.parametrize("seed", range(4))
def test_offload_pressure_workload_swaps_and_resets(seed):
    """The GPU memory-pressure workload: every request finishes, blocks go
    through the swap pool and some requests are soft-reset; the C++
    scheduler agrees with the oracle on every step."""
    import workloads
    from tests.sched_driver import c_from_config, scenario_to_config
    sc = workloads.offload_pressure(seed)
    cfg = scenario_to_config(sc)
    reqs = [dict(id=w.req_id, prompt_len=w.prompt_len, output_len=w.output_len,
                 arrival_step=w.arrival_step) for w in sc.waiting]
    o = oracle_from_config(cfg)
    a = run_trace(o, reqs, 450)
    assert a == run_trace(c_from_config(cfg), reqs, 450)
    assert not o.running and not o.waiting and not o.swapped
    assert sum(len(s["swap_out"]) for s in a) > 100
    assert any(o.requests[r["id"]].prompt_len != r["prompt_len"] for r in reqs)
