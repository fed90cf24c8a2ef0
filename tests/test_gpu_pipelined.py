"""Async double-buffered batching ("Continuous batching architecture",
Async batching) on the GPU: PipelinedStepRunner overlaps each step's input
copies and the previous step's output copy with compute, on separate
streams.  Over the memory-pressure trace (2 layers, swaps and soft resets)
its outputs, read back from pinned host memory, must be bit-identical to
the eager StepRunner's, and the caches and swap pools must end equal.
"""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


def test_pipelined_runner_matches_eager_over_pressure_trace():
    from paged_attention_continuous_gb300.step import PipelinedStepRunner, StepRunner
    from tests.sched_driver import c_from_config, scenario_to_config
    sc = workloads.offload_pressure(2)
    kw = dict(num_blocks=sc.num_blocks, num_q_heads=sc.num_q_heads, num_kv_heads=sc.num_kv_heads,
              head_dim=sc.head_dim, dtype=sc.dtype, max_reqs=sc.max_requests_per_batch,
              max_tokens=sc.max_batch_tokens, max_blocks_per_seq=sc.max_blocks_per_seq,
              num_layers=sc.num_layers, device="cuda", swap_blocks=sc.swap_blocks)
    eager, pipe = StepRunner(**kw), PipelinedStepRunner(**kw)
    sa = c_from_config(scenario_to_config(sc))
    sb = c_from_config(scenario_to_config(sc))
    keep, pending = [], []
    nxt, ran, swaps = 0, 0, 0
    for step in range(250):
        while nxt < len(sc.waiting) and sc.waiting[nxt].arrival_step <= step:
            w = sc.waiting[nxt]
            sa.add_request(w.req_id, w.prompt_len, w.output_len)
            sb.add_request(w.req_id, w.prompt_len, w.output_len)
            nxt += 1
        st, st2 = sa.schedule_step(), sb.schedule_step()
        swaps += len(st["swap_in"]) + len(st["swap_out"])
        if st["status"] != 0 or st["num_reqs"] == 0:
            eager.apply_swaps(st)
            with torch.cuda.stream(pipe.compute_stream):
                pipe.apply_swaps(st2)
            for s_, x in ((sa, st), (sb, st2)):
                if x["status"] == 0:
                    s_.step_done()
            continue
        T = st["num_tokens"]
        ds = eager.upload(st)
        hq, hk, hv, hout, ref = [], [], [], [], []
        for layer in range(sc.num_layers):
            sd = [workloads.step_seed(sc.seed, step, layer, c) for c in range(3)]
            q = workloads.token_tensors(T, sc.num_q_heads, sc.head_dim, seed=sd[0], device="cuda")
            k = workloads.token_tensors(T, sc.num_kv_heads, sc.head_dim, seed=sd[1], device="cuda")
            v = workloads.token_tensors(T, sc.num_kv_heads, sc.head_dim, seed=sd[2], device="cuda")
            ref.append(eager.run(ds, q, k, v, layer=layer).cpu())
            hq.append(q.cpu().pin_memory())
            hk.append(k.cpu().pin_memory())
            hv.append(v.cpu().pin_memory())
            hout.append(torch.empty(T, sc.num_q_heads, sc.head_dim, dtype=q.dtype,
                                    pin_memory=True))
        ev = pipe.submit(st2, hq, hk, hv, hout)
        keep.append((hq, hk, hv))
        pending.append((ev, hout, ref, step))
        sa.step_done()
        sb.step_done()
        ran += 1
    pipe.synchronize()
    torch.cuda.synchronize()
    for ev, hout, ref, step in pending:
        assert ev.query()
        for layer in range(sc.num_layers):
            assert torch.equal(hout[layer], ref[layer]), f"step {step} layer {layer}"
    for layer in range(sc.num_layers):
        assert torch.equal(pipe.k_cache[layer], eager.k_cache[layer])
        assert torch.equal(pipe.v_cache[layer], eager.v_cache[layer])
        assert torch.equal(pipe.swap.k[layer], eager.swap.k[layer])
    assert eager.workspace.read_errors() == 0 and pipe.workspace.read_errors() == 0
    assert ran > 150 and swaps > 50
