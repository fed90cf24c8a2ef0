"""Prefix caching and eviction ("Continuous batching architecture", Prefix
caching, Eviction) on the oracle and the C++ scheduler.

Pins:
* a hand-derived trace (tests/golden/scheduler_prefix_traces.json): reuse
  of a leading run of blocks, the one-token cap for a prompt that is a whole
  number of blocks, reference counts, freed keyed blocks kept and matched
  again, the newest initialized block demoted when the free queue is empty,
  and no match past a dropped key;
* a content model on random traces with shared prompt prefixes (with and
  without offloading): every slot records which token's K/V was last
  written to it (and swaps move those records), and every row of every step
  must see, at each of its positions, its own token -- the property prefix
  sharing exists to keep.  Reference counts, pool conservation and key
  consistency are checked every step;
* with no token ids, prefix caching changes nothing;
* the C++ scheduler equals the oracle bit for bit.
"""
import json
import os

import numpy as np
import pytest

from tests.sched_driver import c_from_config, oracle_from_config, run_trace
from tests.test_oracle_scheduler import _random_trace

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "scheduler_prefix_traces.json")


def _traces():
    with open(GOLDEN) as f:
        return json.load(f)["traces"]


@pytest.mark.parametrize("impl", ["oracle", "c"])
@pytest.mark.parametrize("trace", _traces(), ids=lambda t: t["name"])
def test_hand_derived_prefix_trace(trace, impl):
    make = oracle_from_config if impl == "oracle" else c_from_config
    s = make(trace["config"])
    got = run_trace(s, trace["requests"], len(trace["steps"]))
    for i, (g, e) in enumerate(zip(got, trace["steps"])):
        for k, v in e.items():
            assert g[k] == v, f"step {i}: {k} {g[k]} != {v}"
    if impl == "oracle":
        assert s.free_list() == trace["final_free_list"]
        assert s.prefix_hit_tokens == trace["prefix_hit_tokens"]
    else:
        assert s.free == trace["final_free_list"]
        assert s.prefix_stats()[0] == trace["prefix_hit_tokens"]


def _prefix_trace(seed, offload=None):
    rng = np.random.default_rng(seed)
    bs = int(rng.choice([2, 4]))
    nb = int(rng.integers(8, 40))
    if offload is None:
        offload = bool(rng.integers(0, 2))
    cfg = dict(block_size=bs, num_blocks=nb, max_batch_tokens=int(rng.integers(4, 40)),
               max_requests_per_batch=int(rng.integers(2, 8)),
               max_prefill_chunk=int(rng.choice([0, 0, 3, 8])),
               safety_margin=float(rng.choice([0.0, 0.0, 0.1])), max_blocks_per_seq=64,
               free_list=[int(x) for x in rng.permutation(nb)], policy=int(rng.integers(0, 2)),
               prefix_caching=True, offload=offload,
               swap_blocks=int(rng.choice([0, 4, 12])) if offload else 0)
    # a few shared "system prompts" over a tiny vocabulary, so that equal
    # leading blocks, partial matches and diverging suffixes all occur
    systems = [rng.integers(0, 3, size=int(rng.integers(1, 5 * bs))) for _ in range(3)]
    reqs = []
    for i in range(int(rng.integers(3, 14))):
        sysp = systems[int(rng.integers(0, 3))]
        toks = np.concatenate([sysp, rng.integers(0, 3, size=int(rng.integers(0, 3 * bs)))])
        p = len(toks)
        o = int(rng.integers(1, 4 * bs))
        o = max(1, min(o, nb * bs - p + 1))
        kind = rng.integers(0, 6)
        known = None if kind == 0 else (toks[:int(rng.integers(0, p + 1))] if kind == 1 else toks)
        reqs.append(dict(id=300 + i, prompt_len=p, output_len=o,
                         arrival_step=int(rng.integers(0, 6)),
                         tokens=None if known is None else [int(t) for t in known]))
    return cfg, reqs


def _check_pool(s, num_blocks):
    in_use = {}
    for r in s.running:
        for b in r.blocks:
            in_use[b] = in_use.get(b, 0) + 1
    assert in_use == s.refs
    free, init = list(s.free), list(s.free_init)
    assert len(set(free)) == len(free) and len(set(init)) == len(init)
    assert not (set(free) & set(init)) and not (set(free + init) & set(in_use))
    assert len(in_use) + len(free) + len(init) == num_blocks
    # keys and keyed blocks are one to one; initialized blocks are keyed,
    # free-queue blocks are not
    assert {b: k for k, b in s.cache_index.items()} == s.block_key
    assert set(init) <= set(s.block_key) and not (set(free) & set(s.block_key))


def _run_content_model(cfg, reqs, steps=300):
    s = oracle_from_config(cfg)
    bs = cfg["block_size"]
    known = {r["id"]: (r["tokens"] or []) for r in reqs}
    expect = lambda rid, p: known[rid][p] if p < len(known[rid]) else ("own", rid, p)
    content = {}                        # cache slot -> what was written there
    swap = {}                           # swap slot -> list of bs records
    pending = sorted(reqs, key=lambda r: r["arrival_step"])
    nxt = 0
    for step in range(steps):
        while nxt < len(pending) and pending[nxt]["arrival_step"] <= step:
            r = pending[nxt]
            s.add_request(r["id"], r["prompt_len"], r["output_len"], tokens=r["tokens"])
            nxt += 1
        st = s.schedule_step()
        for slot, blk in st["swap_in"]:
            for j, rec in enumerate(swap.pop(int(slot))):
                content[int(blk) * bs + j] = rec
        for blk, slot in st["swap_out"]:
            swap[int(slot)] = [content.get(int(blk) * bs + j) for j in range(bs)]
        if st["status"] == 0:
            cu = st["cu_seqlens_q"]
            for i, rid in enumerate(st["req_ids"]):
                rid = int(rid)
                L = int(st["seq_lens"][i])
                n = int(cu[i + 1] - cu[i])
                table = st["block_tables"][i]
                for t, p in zip(range(cu[i], cu[i + 1]), range(L - n, L)):
                    assert st["slot_mapping"][t] == table[p // bs] * bs + p % bs
                    content[int(st["slot_mapping"][t])] = expect(rid, p)
            # every row sees its own tokens at every position it attends
            for i, rid in enumerate(st["req_ids"]):
                rid = int(rid)
                table = st["block_tables"][i]
                for p in range(int(st["seq_lens"][i])):
                    got = content.get(int(table[p // bs]) * bs + p % bs)
                    assert got == expect(rid, p), (step, rid, p, got)
            s.step_done()
        _check_pool(s, cfg["num_blocks"])
        # a keyed block holds the last block of its key
        for key, b in s.cache_index.items():
            for j in range(bs):
                assert content.get(b * bs + j) == key[len(key) - bs + j]
        if nxt == len(pending) and not s.running and not s.waiting and not s.swapped:
            break
    return s


@pytest.mark.parametrize("seed", range(80))
def test_prefix_content_model_random_traces(seed):
    cfg, reqs = _prefix_trace(seed)
    _run_content_model(cfg, reqs)


def test_prefix_hits_occur_on_random_traces():
    hits = 0
    for seed in range(20):
        cfg, reqs = _prefix_trace(seed)
        hits += _run_content_model(cfg, reqs).prefix_hit_tokens
    assert hits > 50


@pytest.mark.parametrize("seed", range(20))
def test_prefix_caching_without_tokens_changes_nothing(seed):
    cfg, reqs = _random_trace(seed)
    a = run_trace(oracle_from_config(cfg), reqs, 60)
    b = run_trace(oracle_from_config(dict(cfg, prefix_caching=True)), reqs, 60)
    assert a == b


@pytest.mark.parametrize("seed", range(60))
def test_c_matches_oracle_prefix_random_traces(seed):
    cfg, reqs = _prefix_trace(seed)
    o, c = oracle_from_config(cfg), c_from_config(cfg)
    assert run_trace(o, reqs, 200) == run_trace(c, reqs, 200)
    assert c.free == o.free_list()
    assert c.prefix_stats()[0] == o.prefix_hit_tokens
