"""Offloading on the GPU ("Continuous batching architecture", Offloading):
cb_kv_swap moves whole blocks between the device caches and a pinned host
swap pool, and a serving trace under memory pressure -- requests swapped
out, soft-reset and resumed -- still matches the oracle step by step.

Bars: swapped bytes bit-exact (a block copy); attention outputs within the
bf16 bound of the other parity tests; the graph runner bit-identical to the
eager runner with swaps queued ahead of each replay.
"""
import numpy as np
import pytest
import torch

import workloads
from tests.gpu_harness import ParityRun, tolerance_ok

pytestmark = pytest.mark.gpu


def _cb():
    import paged_attention_continuous_gb300 as cb
    return cb


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_kv_swap_round_trip_bit_exact(dtype):
    cb = _cb()
    nb, ns, L, Hkv, bs, D = 64, 24, 3, 4, 16, 128
    dev = [workloads.cache_fill(nb, Hkv, bs, D, seed=10 + i, dtype=dtype, device="cuda")
           for i in range(2 * L)]
    orig = [t.clone() for t in dev]
    host = [torch.zeros((ns, Hkv, bs, D), dtype=dev[0].dtype, pin_memory=True) for _ in dev]
    rng = np.random.default_rng(5)
    blocks = rng.choice(nb, size=17, replace=False).astype(np.int32)
    slots = rng.choice(ns, size=17, replace=False).astype(np.int32)
    b_d = torch.from_numpy(blocks).cuda()
    s_d = torch.from_numpy(slots).cuda()
    # device -> pinned host
    cb.kv_swap(dev, host, b_d, s_d)
    torch.cuda.synchronize()
    for d, h in zip(dev, host):
        assert torch.equal(h[torch.from_numpy(slots).long()], d.cpu()[torch.from_numpy(blocks).long()])
    untouched = np.setdiff1d(np.arange(ns), slots)
    for h in host:
        assert not h[torch.from_numpy(untouched).long()].any()
    # pinned host -> other device blocks
    dest = rng.choice(np.setdiff1d(np.arange(nb), blocks), size=17, replace=False).astype(np.int32)
    for t in dev:
        t[torch.from_numpy(dest).long().cuda()] = 0
    cb.kv_swap(host, dev, s_d, torch.from_numpy(dest).cuda())
    torch.cuda.synchronize()
    for d, o in zip(dev, orig):
        assert torch.equal(d[torch.from_numpy(dest).long().cuda()],
                           o[torch.from_numpy(blocks).long().cuda()])
        keep = torch.from_numpy(np.setdiff1d(np.arange(nb), dest)).long().cuda()
        assert torch.equal(d[keep], o[keep])
    # device -> device (the same call moves blocks within GPU memory)
    other = [torch.zeros_like(t) for t in dev]
    cb.kv_swap(dev, other, b_d, b_d)
    torch.cuda.synchronize()
    for d, o in zip(dev, other):
        assert torch.equal(o[b_d.long()], d[b_d.long()])


def test_kv_swap_out_of_range_pair_flagged_and_skipped():
    cb = _cb()
    nb, ns = 8, 4
    dev = [workloads.cache_fill(nb, 2, 16, 64, seed=3, dtype="bf16", device="cuda")]
    host = [torch.zeros((ns, 2, 16, 64), dtype=torch.bfloat16, pin_memory=True)]
    ew = torch.zeros(1, dtype=torch.int32, device="cuda")
    src = torch.tensor([1, 2, 3], dtype=torch.int32, device="cuda")
    dst = torch.tensor([0, ns, 2], dtype=torch.int32, device="cuda")  # ns is out of range
    cb.kv_swap(dev, host, src, dst, error_word=ew)
    torch.cuda.synchronize()
    assert int(ew.item()) & cb.DEVERR_BLOCK_RANGE
    d = dev[0].cpu()
    assert torch.equal(host[0][0], d[1]) and torch.equal(host[0][2], d[3])
    assert not host[0][1].any() and not host[0][3].any()


def test_kv_swap_refuses_pageable_host_memory():
    cb = _cb()
    dev = [torch.zeros((4, 2, 16, 64), dtype=torch.bfloat16, device="cuda")]
    pageable = [torch.zeros((4, 2, 16, 64), dtype=torch.bfloat16)]
    ids = torch.tensor([0], dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        cb.kv_swap(dev, pageable, ids, ids)      # caught by the binding
    import ctypes
    P = ctypes.c_void_p * 1
    a = cb.cb_swap_args(1, ids.data_ptr(), ids.data_ptr(), 1,
                        ctypes.cast(P(dev[0].data_ptr()), ctypes.POINTER(ctypes.c_void_p)),
                        ctypes.cast(P(pageable[0].data_ptr()), ctypes.POINTER(ctypes.c_void_p)),
                        4, 4, 2 * 16 * 64 * 2, None)
    assert cb.library().cb_kv_swap(ctypes.byref(a), None) == cb.CB_ERR_INVALID_ARG
    torch.cuda.synchronize()


@pytest.mark.parametrize("seed", [0, 3])
def test_offload_pressure_trace_matches_oracle(seed):
    """The whole memory-pressure trace: every step on both sides, until all
    requests finished; swaps and soft resets both occur."""
    sc = workloads.offload_pressure(seed)
    run = ParityRun(sc, arrivals=True)
    steps = 0
    for _ in range(600):
        st, g, r, toks = run.step()
        if st == 0:
            for layer in range(sc.num_layers):
                ok, err, excess = tolerance_ok(g[layer], r[layer], "bf16")
                assert ok, f"step {run.step_idx - 1} layer {layer}: max err {err:.3e}"
        steps += 1
        if (run.next_arrival == len(sc.waiting) and not run.o.running and not run.o.waiting
                and not run.o.swapped):
            break
    assert not run.o.running and not run.o.waiting and not run.o.swapped
    assert run.swap_pairs > 100
    resets = sum(1 for w in sc.waiting if run.o.requests[w.req_id].prompt_len != w.prompt_len)
    assert resets > 0
    assert steps > 200


def test_offload_pressure_graph_matches_eager():
    import paged_attention_continuous_gb300 as cb
    from paged_attention_continuous_gb300.step import GraphStepRunner, StepRunner
    from tests.sched_driver import c_from_config, scenario_to_config
    sc = workloads.offload_pressure(1)
    s = c_from_config(scenario_to_config(sc))
    kw = dict(num_blocks=sc.num_blocks, num_q_heads=sc.num_q_heads, num_kv_heads=sc.num_kv_heads,
              head_dim=sc.head_dim, dtype=sc.dtype, max_reqs=sc.max_requests_per_batch,
              max_tokens=sc.max_batch_tokens, max_blocks_per_seq=sc.max_blocks_per_seq,
              num_layers=sc.num_layers, device="cuda", swap_blocks=sc.swap_blocks)
    eager, graph = StepRunner(**kw), GraphStepRunner(**kw)
    nxt, ran, swaps = 0, 0, 0
    for step in range(200):
        while nxt < len(sc.waiting) and sc.waiting[nxt].arrival_step <= step:
            w = sc.waiting[nxt]
            s.add_request(w.req_id, w.prompt_len, w.output_len)
            nxt += 1
        st = s.schedule_step()
        swaps += len(st["swap_in"]) + len(st["swap_out"])
        if st["status"] != 0 or st["num_reqs"] == 0:
            eager.apply_swaps(st)
            graph.apply_swaps(st)
            if st["status"] == 0:
                s.step_done()
            continue
        T = st["num_tokens"]
        ds = eager.upload(st)
        key, _ = graph.prepare(st)
        outs = []
        for layer in range(sc.num_layers):
            sd = [workloads.step_seed(sc.seed, step, layer, c) for c in range(3)]
            q = workloads.token_tensors(T, sc.num_q_heads, sc.head_dim, seed=sd[0], device="cuda")
            k = workloads.token_tensors(T, sc.num_kv_heads, sc.head_dim, seed=sd[1], device="cuda")
            v = workloads.token_tensors(T, sc.num_kv_heads, sc.head_dim, seed=sd[2], device="cuda")
            outs.append(eager.run(ds, q, k, v, layer=layer))
            graph.q_buf[layer][:T].copy_(q)
            graph.k_buf[layer][:T].copy_(k)
            graph.v_buf[layer][:T].copy_(v)
        graph.run(key)
        for layer in range(sc.num_layers):
            assert torch.equal(graph.out_buf[layer][:T], outs[layer]), f"step {step} layer {layer}"
        s.step_done()
        ran += 1
    torch.cuda.synchronize()
    for layer in range(sc.num_layers):
        assert torch.equal(graph.k_cache[layer], eager.k_cache[layer])
        assert torch.equal(graph.swap.v[layer], eager.swap.v[layer])
    assert eager.swap.read_errors() == 0 and graph.swap.read_errors() == 0
    assert eager.workspace.read_errors() == 0 and graph.workspace.read_errors() == 0
    assert swaps > 50 and ran > 150
