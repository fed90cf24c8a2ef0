"""Sliding-window layers ("Continuous batching architecture", Memory
management: sliding layers keep a fixed window of recent tokens by recycling
a small set of pages) on the oracle and the C++ scheduler, and sliding-window
attention end to end through the oracle's paging.

Pins:
* a hand-derived trace (tests/golden/scheduler_window_traces.json): pages
  freed once wholly before every future query's window, entries -1, the
  freed pages reused;
* a content model on random traces (with and without offloading): every
  row reads its own K/V at every position of its window, the pages it
  still holds are bounded by the window, and blocks are conserved;
* prompts run through the oracle scheduler with a window, the paged append
  and the windowed paged attention equal an explicit loop over each
  query's window on the dense tensors (chunk sizes and block order do not
  matter);
* windowed attention of one query equals torch's scaled_dot_product_attention
  over that window's keys, a window of 1 returns the query's own V, a window
  at least the sequence length equals full attention, and an off-by-one
  window is caught;
* the C++ scheduler equals the oracle bit for bit.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import paged_kv
from oracle.scheduler import FifoScheduler
from tests.sched_driver import c_from_config, oracle_from_config, run_trace

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "scheduler_window_traces.json")


def _traces():
    with open(GOLDEN) as f:
        return json.load(f)["traces"]


@pytest.mark.parametrize("impl", ["oracle", "c"])
@pytest.mark.parametrize("trace", _traces(), ids=lambda t: t["name"])
def test_hand_derived_window_trace(trace, impl):
    make = oracle_from_config if impl == "oracle" else c_from_config
    s = make(trace["config"])
    got = run_trace(s, trace["requests"], len(trace["steps"]))
    for i, (g, e) in enumerate(zip(got, trace["steps"])):
        for k, v in e.items():
            assert g[k] == v, f"step {i}: {k} {g[k]} != {v}"
    free = s.free_list() if impl == "oracle" else s.free
    assert free == trace["final_free_list"]


def test_window_refuses_prefix_caching():
    with pytest.raises(ValueError):
        FifoScheduler(block_size=4, num_blocks=8, max_batch_tokens=8, max_requests_per_batch=2,
                      max_blocks_per_seq=4, prefix_caching=True, sliding_window=8)
    import paged_attention_continuous_gb300 as cb
    with pytest.raises(cb.CBError):
        cb.Scheduler(block_size=4, num_blocks=8, max_batch_tokens=8, max_requests_per_batch=2,
                     max_blocks_per_seq=4, prefix_caching=True, sliding_window=8)


def _window_trace(seed, offload=None):
    rng = np.random.default_rng(seed)
    bs = int(rng.choice([2, 4]))
    nb = int(rng.integers(6, 30))
    if offload is None:
        offload = bool(rng.integers(0, 2))
    W = int(rng.choice([1, 2, 3, 5, 8, 13]))
    cfg = dict(block_size=bs, num_blocks=nb, max_batch_tokens=int(rng.integers(3, 30)),
               max_requests_per_batch=int(rng.integers(2, 8)),
               max_prefill_chunk=int(rng.choice([0, 0, 3, 8])),
               safety_margin=float(rng.choice([0.0, 0.0, 0.1])), max_blocks_per_seq=64,
               free_list=[int(x) for x in rng.permutation(nb)], policy=int(rng.integers(0, 2)),
               offload=offload, swap_blocks=int(rng.choice([0, 4, 12])) if offload else 0,
               sliding_window=W)
    reqs = []
    for i in range(int(rng.integers(2, 10))):
        p = int(rng.integers(1, 5 * bs))
        # long outputs: the window keeps them within the pool
        o = int(rng.integers(1, 12 * bs))
        reqs.append(dict(id=500 + i, prompt_len=p, output_len=o,
                         arrival_step=int(rng.integers(0, 5))))
    return cfg, reqs


def _run_window_model(cfg, reqs, steps=400):
    s = oracle_from_config(cfg)
    bs, W = cfg["block_size"], cfg["sliding_window"]
    content, swap = {}, {}
    pending = sorted(reqs, key=lambda r: r["arrival_step"])
    nxt, ran = 0, 0
    for step in range(steps):
        while nxt < len(pending) and pending[nxt]["arrival_step"] <= step:
            r = pending[nxt]
            s.add_request(r["id"], r["prompt_len"], r["output_len"])
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
                L, n = int(st["seq_lens"][i]), int(cu[i + 1] - cu[i])
                for t, p in zip(range(cu[i], cu[i + 1]), range(L - n, L)):
                    content[int(st["slot_mapping"][t])] = (int(rid), p)
            for i, rid in enumerate(st["req_ids"]):
                L, n = int(st["seq_lens"][i]), int(cu[i + 1] - cu[i])
                table = st["block_tables"][i]
                lo = max(0, L - n - W + 1)
                for p in range(lo, L):
                    b = int(table[p // bs])
                    assert b >= 0, (step, int(rid), p)
                    assert content.get(b * bs + p % bs) == (int(rid), p), (step, int(rid), p)
                # nothing before the window is still held
                assert all(int(b) < 0 for b in table[:lo // bs])
            s.step_done()
            ran += 1
        # conservation and the window's bound on pages held
        held = [b for r in s.running for b in r.blocks if b >= 0]
        assert len(held) == len(set(held)) and not (set(held) & set(s.free))
        assert len(held) + len(s.free) == cfg["num_blocks"]
        for r in s.running:
            live = sum(1 for b in r.blocks if b >= 0)
            assert live <= -(-(W - 1) // bs) + 1 + -(-cfg["max_batch_tokens"] // bs) + 1
        if nxt == len(pending) and not s.running and not s.waiting and not s.swapped:
            break
    return s, ran


@pytest.mark.parametrize("seed", range(80))
def test_window_content_model_random_traces(seed):
    cfg, reqs = _window_trace(seed)
    _run_window_model(cfg, reqs)


@pytest.mark.parametrize("seed", range(60))
def test_c_matches_oracle_window_random_traces(seed):
    cfg, reqs = _window_trace(seed)
    o, c = oracle_from_config(cfg), c_from_config(cfg)
    assert run_trace(o, reqs, 250) == run_trace(c, reqs, 250)
    assert c.free == o.free_list()


# --------------------------------------------------------------- attention
def _window_loop(q, k, v, W, scale):
    """Explicit loops: query i of a prompt attends keys max(0, i-W+1)..i."""
    L, Hq, D = q.shape
    Hkv = k.shape[1]
    out = np.zeros_like(q)
    for i in range(L):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            js = range(max(0, i - W + 1), i + 1)
            sc = [scale * float(np.dot(q[i, h], k[j, g])) for j in js]
            m = max(sc)
            w = [math.exp(x - m) for x in sc]
            z = sum(w)
            out[i, h] = sum(wj * v[j, g] for wj, j in zip(w, js)) / z
    return out


@pytest.mark.parametrize("case", [
    dict(lens=[30, 9, 17], W=5, chunk=7, bs=4, Hq=2, Hkv=1, D=4),
    dict(lens=[40], W=16, chunk=16, bs=16, Hq=4, Hkv=2, D=3),
    dict(lens=[23, 23], W=1, chunk=5, bs=4, Hq=2, Hkv=2, D=5),
    dict(lens=[12, 33], W=40, chunk=9, bs=4, Hq=3, Hkv=1, D=4),
])
def test_windowed_prompts_through_paging_match_loops(case):
    rng = np.random.default_rng(case["W"] * 31 + len(case["lens"]))
    Hq, Hkv, D, bs, W = case["Hq"], case["Hkv"], case["D"], case["bs"], case["W"]
    qs = [rng.standard_normal((L, Hq, D)) for L in case["lens"]]
    ks = [rng.standard_normal((L, Hkv, D)) for L in case["lens"]]
    vs = [rng.standard_normal((L, Hkv, D)) for L in case["lens"]]
    nb = sum(-(-L // bs) for L in case["lens"]) + 2
    s = FifoScheduler(block_size=bs, num_blocks=nb, max_batch_tokens=case["chunk"],
                      max_requests_per_batch=4, max_blocks_per_seq=-(-max(case["lens"]) // bs),
                      safety_margin=0.0, free_list=rng.permutation(nb).tolist(),
                      sliding_window=W)
    for i, L in enumerate(case["lens"]):
        s.add_request(i, L, 1)
    kc = np.full((nb, Hkv, bs, D), np.nan)      # never-written slots would poison the result
    vc = np.full_like(kc, np.nan)
    outs = [np.zeros_like(q) for q in qs]
    scale = 1.0 / math.sqrt(D)
    dropped = 0
    while True:
        st = s.schedule_step()
        if st["num_reqs"] == 0:
            break
        T = st["num_tokens"]
        qb, kb, vb = np.zeros((T, Hq, D)), np.zeros((T, Hkv, D)), np.zeros((T, Hkv, D))
        for i, rid in enumerate(st["req_ids"]):
            t0, t1 = st["cu_seqlens_q"][i], st["cu_seqlens_q"][i + 1]
            p1 = st["seq_lens"][i]; p0 = p1 - (t1 - t0)
            qb[t0:t1], kb[t0:t1], vb[t0:t1] = qs[rid][p0:p1], ks[rid][p0:p1], vs[rid][p0:p1]
        dropped += int((st["block_tables"][:, 0] < 0).sum())
        paged_kv.append(kc, vc, kb, vb, st["slot_mapping"], bs)
        o = oatt.paged_attention(qb, kc, vc, st["cu_seqlens_q"], st["seq_lens"],
                                 st["block_tables"], bs, scale, window=W)
        for i, rid in enumerate(st["req_ids"]):
            t0, t1 = st["cu_seqlens_q"][i], st["cu_seqlens_q"][i + 1]
            p1 = st["seq_lens"][i]; p0 = p1 - (t1 - t0)
            outs[rid][p0:p1] = o[t0:t1]
        s.step_done()
    for q, k, v, o in zip(qs, ks, vs, outs):
        assert np.max(np.abs(_window_loop(q, k, v, W, scale) - o)) < 1e-12
    if W < max(case["lens"]) - case["chunk"] - bs:
        assert dropped > 0                       # pages really were recycled


def test_window_matches_torch_sdpa_over_the_window():
    rng = np.random.default_rng(21)
    L, Hq, Hkv, D, W = 50, 4, 2, 16, 13
    q = rng.standard_normal((1, Hq, D))
    k = rng.standard_normal((L, Hkv, D))
    v = rng.standard_normal((L, Hkv, D))
    got = oatt.attend_one_request(q, k, v, L - 1, 0.2, window=W)
    kw = torch.from_numpy(np.repeat(k[L - W:], Hq // Hkv, axis=1)).permute(1, 0, 2)
    vw = torch.from_numpy(np.repeat(v[L - W:], Hq // Hkv, axis=1)).permute(1, 0, 2)
    qt = torch.from_numpy(q).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kw, vw, scale=0.2)
    assert np.max(np.abs(ref.permute(1, 0, 2).numpy() - got)) < 1e-12


def test_window_special_cases_and_a_slip():
    rng = np.random.default_rng(22)
    L, Hq, Hkv, D = 30, 4, 2, 8
    q = rng.standard_normal((L, Hq, D)); k = rng.standard_normal((L, Hkv, D))
    v = rng.standard_normal((L, Hkv, D))
    one = oatt.attend_one_request(q, k, v, 0, 0.3, window=1)
    for i in range(L):
        for h in range(Hq):
            assert np.array_equal(one[i, h], v[i, h // 2])
    full = oatt.attend_one_request(q, k, v, 0, 0.3)
    assert np.array_equal(oatt.attend_one_request(q, k, v, 0, 0.3, window=L), full)
    good = _window_loop(q, k, v, 7, 0.3)
    assert np.max(np.abs(oatt.attend_one_request(q, k, v, 0, 0.3, window=7) - good)) < 1e-12
    assert np.max(np.abs(oatt.attend_one_request(q, k, v, 0, 0.3, window=8) - good)) > 1e-3
    assert np.max(np.abs(oatt.attend_one_request(q, k, v, 0, 0.3, window=6) - good)) > 1e-3
