"""Pins for the oracle scheduler: hand-derived traces and invariants."""
import json
import math
import os

import numpy as np
import pytest

from oracle.scheduler import FifoScheduler, DECODING, PREFILLING
from tests.sched_driver import oracle_from_config, run_trace

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "scheduler_traces.json")


def _traces():
    with open(GOLDEN) as f:
        return json.load(f)["traces"]


@pytest.mark.parametrize("trace", _traces(), ids=lambda t: t["name"])
def test_hand_derived_trace(trace):
    sched = oracle_from_config(trace["config"])
    got = run_trace(sched, trace["requests"], len(trace["steps"]))
    for i, (g, e) in enumerate(zip(got, trace["steps"])):
        for k, v in e.items():
            assert g[k] == v, f"step {i + 1} field {k}: {g[k]} != {v}"
    assert list(sched.free) == trace["final_free_list"]


def test_worked_example_chunks():
    """1000-token prompt under a 256-token budget -> 256/256/256/232."""
    with open(os.path.join(os.path.dirname(__file__), "golden",
                           "chunked_prefill_worked_example.json")) as f:
        g = json.load(f)
    s = FifoScheduler(block_size=16, num_blocks=64, max_batch_tokens=g["chunk"],
                      max_requests_per_batch=4, max_blocks_per_seq=64,
                      safety_margin=0.0)
    s.add_request(0, g["prompt_len"], 1)
    chunks = []
    while True:
        st = s.schedule_step()
        if st["num_reqs"] == 0:
            break
        chunks.append(int(st["cu_seqlens_q"][1]))
        s.step_done()
    assert chunks == g["chunks"]


def test_margin_rounding_matches_float32():
    s = FifoScheduler(block_size=16, num_blocks=65536, max_batch_tokens=8,
                      max_requests_per_batch=4, max_blocks_per_seq=8,
                      safety_margin=0.15)
    assert s.reserved_blocks == math.ceil(float(np.float32(0.15)) * 65536) == 9831


def _random_trace(seed):
    rng = np.random.default_rng(seed)
    bs = int(rng.choice([2, 4, 16]))
    nb = int(rng.integers(4, 60))
    cfg = dict(block_size=bs, num_blocks=nb,
               max_batch_tokens=int(rng.integers(1, 40)),
               max_requests_per_batch=int(rng.integers(1, 6)),
               max_prefill_chunk=int(rng.choice([0, 0, 3, 8])),
               safety_margin=float(rng.choice([0.0, 0.1, 0.15, 0.3])),
               max_blocks_per_seq=64,
               free_list=[int(x) for x in rng.permutation(nb)])
    reqs = []
    for i in range(int(rng.integers(1, 12))):
        reqs.append(dict(id=100 + i, prompt_len=int(rng.integers(1, 30)),
                         output_len=int(rng.integers(1, 8)),
                         arrival_step=int(rng.integers(0, 6))))
    return cfg, reqs


@pytest.mark.parametrize("seed", range(60))
def test_invariants_random_traces(seed):
    cfg, reqs = _random_trace(seed)
    s = oracle_from_config(cfg)
    bs, nb = cfg["block_size"], cfg["num_blocks"]
    reqs = sorted(reqs, key=lambda r: r["arrival_step"])
    added = 0
    for step in range(80):
        while added < len(reqs) and reqs[added]["arrival_step"] <= step:
            r = reqs[added]
            s.add_request(r["id"], r["prompt_len"], r["output_len"])
            added += 1
        before = {r.req_id: (r.state, r.num_cached) for r in s.running}
        waiting_before = [r.req_id for r in s.waiting]
        st = s.schedule_step()
        R = st["num_reqs"]
        qlens = np.diff(st["cu_seqlens_q"])
        # token budget and request cap
        assert qlens.sum() <= cfg["max_batch_tokens"]
        assert R <= cfg["max_requests_per_batch"]
        assert (qlens >= 1).all()
        nd = st["num_decodes"]
        ids = list(st["req_ids"])
        # decodes first (one token each), then prefills
        for i, rid in enumerate(ids):
            if i < nd:
                assert before[rid][0] == DECODING and qlens[i] == 1
            else:
                assert rid not in before or before[rid][0] == PREFILLING
        # new admissions are a prefix of the waiting queue, in arrival order
        new = [rid for rid in ids if rid not in before]
        assert new == waiting_before[:len(new)]
        # block tables cover exactly the scheduled tokens; slots follow them
        for i, rid in enumerate(ids):
            L = st["seq_lens"][i]
            row = st["block_tables"][i]
            nblk = int((row >= 0).sum())
            assert nblk == -(-L // bs)
            start = L - qlens[i]
            for j, t in enumerate(range(st["cu_seqlens_q"][i], st["cu_seqlens_q"][i + 1])):
                pos = start + j
                assert st["slot_mapping"][t] == row[pos // bs] * bs + pos % bs
            if rid in before:
                assert start == before[rid][1]
        # stalled requests are active and were not scheduled
        for rid in st["stalled_ids"]:
            assert rid in before and rid not in ids
        if st["status"] == 0:
            s.step_done()
        # conservation: free + allocated == pool, no duplicates
        alloc = [b for r in s.running for b in r.blocks]
        assert len(s.free) + len(alloc) == nb
        assert len(set(list(s.free) + alloc)) == nb
        if added == len(reqs) and not s.running and not s.waiting:
            break
    # a request that can never fit may stay waiting; everything else drains
    if not s.waiting:
        assert len(s.free) == nb


def test_add_running_request_states():
    s = FifoScheduler(block_size=16, num_blocks=100, max_batch_tokens=64,
                      max_requests_per_batch=8, max_blocks_per_seq=20,
                      safety_margin=0.0, free_list=list(range(100)))
    s.add_running_request(1, prompt_len=40, output_len=10, num_cached=45)
    s.add_running_request(2, prompt_len=100, output_len=10, num_cached=33)
    assert s.requests[1].state == DECODING and s.requests[1].num_generated == 6
    assert s.requests[1].blocks == [0, 1, 2]
    assert s.requests[2].state == PREFILLING and s.requests[2].blocks == [3, 4, 5]
    st = s.schedule_step()
    assert list(st["req_ids"]) == [1, 2] and st["num_decodes"] == 1
    assert list(st["seq_lens"]) == [46, 96]
    assert st["slot_mapping"][0] == 2 * 16 + 13
    with pytest.raises(ValueError):
        s.add_running_request(3, prompt_len=10, output_len=2, num_cached=11)
