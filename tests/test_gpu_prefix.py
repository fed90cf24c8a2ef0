"""Prefix caching on the GPU ("Continuous batching architecture", Prefix
caching, Eviction): requests that reuse another request's prompt blocks
start their prefill at the end of the reused run and attend blocks they
never wrote; the whole trace matches the oracle step by step (its sub-pool
shares blocks by physical id exactly as the block tables do).

Bars: bf16 outputs within the bound of the other parity tests; scheduler
metadata bit-exact (checked by the harness every step).
"""
import dataclasses

import pytest

import workloads
from tests.gpu_harness import ParityRun, tolerance_ok

pytestmark = pytest.mark.gpu


def _run_all(sc, max_steps=1000):
    run = ParityRun(sc, arrivals=True)
    ran = 0
    for _ in range(max_steps):
        st, g, r, toks = run.step()
        if st == 0:
            for layer in range(sc.num_layers):
                ok, err, _ = tolerance_ok(g[layer], r[layer], "bf16")
                assert ok, f"step {run.step_idx - 1} layer {layer}: max err {err:.3e}"
            ran += 1
        if (run.next_arrival == len(sc.waiting) and not run.o.running and not run.o.waiting
                and not run.o.swapped):
            break
    assert not run.o.running and not run.o.waiting and not run.o.swapped
    return run, ran


def test_shared_prefix_trace_matches_oracle():
    """48 requests over 4 shared system prompts: about two thirds of the
    prompt tokens are reused rather than recomputed."""
    sc = workloads.shared_prefix(0)
    run, ran = _run_all(sc)
    total = sum(w.prompt_len for w in sc.waiting)
    assert run.o.prefix_hit_tokens > total // 2
    assert run.c.prefix_stats()[0] == run.o.prefix_hit_tokens
    assert ran > 50


def test_shared_prefix_under_memory_pressure_matches_oracle():
    """The same kind of trace on a 400-block pool with offloading: keyed
    blocks are demoted and reused, shared blocks are swapped out with their
    requests, and reset requests match their old prefix again."""
    sc = dataclasses.replace(workloads.shared_prefix(1, num_blocks=400), offload=True,
                             swap_blocks=64)
    run, ran = _run_all(sc)
    assert run.swap_pairs > 100
    assert run.o.prefix_hit_tokens > 10000
    assert ran > 100
