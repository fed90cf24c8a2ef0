"""CUDA-graph step replay (GraphStepRunner) against the eager StepRunner.

Both run the same scheduler steps of the request trace (per-step Poisson
arrivals, 4 layers) on the same q/k/v.  The graph runner pads every step to
a power-of-two bucket (padding rows with query length 0 and seq_len 0,
padding tokens with slot -1) and replays one captured graph per bucket; the
kernels compute every real row exactly as in the eager call, so the outputs
must be bit-identical.  The eager path is itself checked against the oracle
in the parity tests.
"""
import numpy as np
import pytest
import torch

import workloads
from paged_attention_continuous_gb300.step import bucket

pytestmark = pytest.mark.gpu


def test_bucket():
    assert [bucket(n) for n in (0, 1, 2, 3, 5, 64, 65)] == [0, 1, 2, 4, 8, 64, 128]
    assert bucket(3, 16) == 16


def test_graph_replay_matches_eager_over_trace_steps():
    import paged_attention_continuous_gb300 as cb
    from paged_attention_continuous_gb300.step import GraphStepRunner, StepRunner
    sc = workloads.trace_2000(num_blocks=16384)
    s = cb.Scheduler(block_size=sc.block_size, num_blocks=sc.num_blocks,
                     max_batch_tokens=sc.max_batch_tokens,
                     max_requests_per_batch=sc.max_requests_per_batch,
                     max_blocks_per_seq=sc.max_blocks_per_seq,
                     max_prefill_chunk=sc.max_prefill_chunk, safety_margin=sc.safety_margin,
                     free_list=sc.free_list)
    kw = dict(num_blocks=sc.num_blocks, num_q_heads=sc.num_q_heads, num_kv_heads=sc.num_kv_heads,
              head_dim=sc.head_dim, dtype=sc.dtype, max_reqs=sc.max_requests_per_batch,
              max_tokens=sc.max_batch_tokens, max_blocks_per_seq=sc.max_blocks_per_seq,
              num_layers=sc.num_layers, device="cuda")
    eager, graph = StepRunner(**kw), GraphStepRunner(**kw)
    nxt, ran = 0, 0
    for step in range(40):
        while nxt < len(sc.waiting) and sc.waiting[nxt].arrival_step <= step:
            w = sc.waiting[nxt]
            s.add_request(w.req_id, w.prompt_len, w.output_len)
            nxt += 1
        st = s.schedule_step()
        if st["status"] != 0 or st["num_reqs"] == 0:
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
            assert torch.equal(graph.k_cache[layer], eager.k_cache[layer])
        s.step_done()
        ran += 1
    assert eager.workspace.read_errors() == 0
    assert graph.workspace.read_errors() == 0
    assert ran > 30
    assert len(graph.graphs) < ran  # buckets are reused


def test_graph_replay_matches_eager_sliding_window():
    """The sliding-window trace (recycled pages, -1 entries in the tables):
    graph replay of padded buckets equals the eager runner bit for bit."""
    from paged_attention_continuous_gb300.step import GraphStepRunner, StepRunner
    from tests.sched_driver import c_from_config, scenario_to_config
    sc = workloads.sliding_trace(1)
    s = c_from_config(scenario_to_config(sc))
    kw = dict(num_blocks=sc.num_blocks, num_q_heads=sc.num_q_heads, num_kv_heads=sc.num_kv_heads,
              head_dim=sc.head_dim, dtype=sc.dtype, max_reqs=sc.max_requests_per_batch,
              max_tokens=sc.max_batch_tokens, max_blocks_per_seq=sc.max_blocks_per_seq,
              num_layers=sc.num_layers, device="cuda", sliding_window=sc.sliding_window)
    eager, graph = StepRunner(**kw), GraphStepRunner(**kw)
    nxt, ran, dropped = 0, 0, 0
    for step in range(120):
        while nxt < len(sc.waiting) and sc.waiting[nxt].arrival_step <= step:
            w = sc.waiting[nxt]
            s.add_request(w.req_id, w.prompt_len, w.output_len)
            nxt += 1
        st = s.schedule_step()
        if st["status"] != 0 or st["num_reqs"] == 0:
            if st["status"] == 0:
                s.step_done()
            continue
        dropped += int((st["block_tables"][:, 0] < 0).sum())
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
    assert eager.workspace.read_errors() == 0 and graph.workspace.read_errors() == 0
    assert ran > 100 and dropped > 100
