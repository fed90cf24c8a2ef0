"""cb_schedule_step (C++) against the oracle scheduler: bit-exact batch
composition, block tables, slot mappings, stalled lists, finished lists and
free lists, step by step."""
import json
import os

import numpy as np
import pytest

import workloads
from tests.sched_driver import (c_from_config, load_scenario, normalize, oracle_from_config,
                                run_trace, scenario_to_config)
from tests.test_oracle_scheduler import _random_trace

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "scheduler_traces.json")


def _traces():
    with open(GOLDEN) as f:
        return json.load(f)["traces"]


@pytest.mark.parametrize("trace", _traces(), ids=lambda t: t["name"])
def test_c_matches_hand_derived_trace(trace):
    s = c_from_config(trace["config"])
    got = run_trace(s, trace["requests"], len(trace["steps"]))
    for i, (g, e) in enumerate(zip(got, trace["steps"])):
        for k, v in e.items():
            assert g[k] == v, f"step {i + 1} field {k}: {g[k]} != {v}"
    assert s.free == trace["final_free_list"]


@pytest.mark.parametrize("seed", range(60))
def test_c_matches_oracle_random_traces(seed):
    cfg, reqs = _random_trace(seed)
    a = run_trace(oracle_from_config(cfg), reqs, 60)
    c = c_from_config(cfg)
    b = run_trace(c, reqs, 60)
    assert a == b


def _compare_scenario(sc, steps, arrivals=False):
    cfg = scenario_to_config(sc)
    o = oracle_from_config(cfg)
    c = c_from_config(cfg)
    load_scenario(o, sc, up_to_step=0 if arrivals else None)
    load_scenario(c, sc, up_to_step=0 if arrivals else None)
    waiting = sorted(sc.waiting, key=lambda w: w.arrival_step)
    nxt = sum(1 for w in waiting if w.arrival_step <= 0) if arrivals else len(waiting)
    n = 0
    for step in range(steps):
        if arrivals:
            while nxt < len(waiting) and waiting[nxt].arrival_step <= step:
                w = waiting[nxt]
                o.add_request(w.req_id, w.prompt_len, w.output_len)
                c.add_request(w.req_id, w.prompt_len, w.output_len)
                nxt += 1
        so, sc_ = o.schedule_step(), c.schedule_step()
        assert normalize(so) == normalize(sc_), f"step {step}"
        if so["status"] != 0:
            break
        assert o.step_done() == c.step_done()
        assert list(o.free) == c.free
        n += 1
        if not o.running and not o.waiting and nxt >= len(waiting):
            break
    return n


def test_mixed_2048_first_steps():
    sc = workloads.mixed_2048()
    _compare_scenario(sc, 6)
    # the batch composition the workload is built for
    o = oracle_from_config(scenario_to_config(sc))
    load_scenario(o, sc)
    st = o.schedule_step()
    q = np.diff(st["cu_seqlens_q"])
    assert st["num_decodes"] == 96 and q[96] == 1024 and q.sum() == 2048
    assert st["num_reqs"] > 98


def test_long_prompt_interleave_64_steps():
    sc = workloads.long_prompt_32k()
    n = _compare_scenario(sc, 64)
    assert n == 64
    o = oracle_from_config(scenario_to_config(sc))
    load_scenario(o, sc)
    for _ in range(64):
        st = o.schedule_step()
        q = np.diff(st["cu_seqlens_q"])
        assert st["num_decodes"] == 128 and q[-1] == 512
        o.step_done()


def test_decode_64_step():
    sc = workloads.decode_64()
    _compare_scenario(sc, 3)


def test_trace_2000_prefix():
    sc = workloads.trace_2000()
    n = _compare_scenario(sc, 250, arrivals=True)
    assert n > 100
