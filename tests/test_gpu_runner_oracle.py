"""The CUDA-graph, pipelined and native-executor step paths against the
oracle, directly.

"Continuous batching architecture" (CUDA graphs; Async batching): the graph
runner pads each step to a power-of-two bucket and replays a captured graph
(padding rows of query length 0 and seq_len 0, padding tokens of slot -1,
which the eager path never sends); the pipelined runner and the C step
executor (cb_executor_submit, and cb_executor_run_step, which also
schedules and commits each step itself) take their inputs and return their
output in pinned host memory, copied on their own streams.  Each is run step
by step next to the oracle (its own scheduler, append and attention) on the
same seeded inputs, and compared element by element at the bf16 bound:
|gpu - oracle| <= 2e-2 + 1e-2 |oracle|.
"""
import pytest

import workloads
from tests.gpu_harness import ParityRun, tolerance_ok
from tests.test_gpu_parity import _mixed_small

pytestmark = pytest.mark.gpu

RUNNERS = ["graph", "pipelined", "native", "native_run"]
SWAP_RUNNERS = ["graph", "pipelined"]   # the executor owns no swap pool


def _check_all(run, g, r, what):
    for layer in range(len(g)):
        ok, err, excess = tolerance_ok(g[layer], r[layer], run.dtype)
        assert ok, f"{run.kind} {what} layer {layer}: max err {err:.3e}, excess {excess:.3e}"


@pytest.mark.parametrize("runner", RUNNERS)
def test_runner_mixed_steps_match_oracle(runner):
    """Decodes, an in-flight prefill and new prompts, five steps."""
    sc = _mixed_small("bf16", 32, 8, 128)
    run = ParityRun(sc, runner=runner)
    for step in range(5):
        st, g, r, _ = run.step()
        assert st == 0
        _check_all(run, g, r, f"mixed step {step}")


@pytest.mark.parametrize("runner", RUNNERS)
def test_runner_trace_steps_match_oracle(runner):
    """The request trace's first 12 steps (per-step arrivals, 4 layers with
    their own pools); the oracle follows four requests, and the buckets of
    the graph runner carry padding rows next to them."""
    sc = workloads.trace_2000(num_blocks=16384)
    run = ParityRun(sc, sample=[1, 5, 25, 39], arrivals=True, runner=runner)
    seen = 0
    for step in range(12):
        st, g, r, toks = run.step()
        assert st == 0
        if len(toks):
            _check_all(run, g, r, f"trace step {step}")
        seen += len(toks)
    assert seen > 0


@pytest.mark.parametrize("runner", SWAP_RUNNERS)
def test_runner_offload_trace_matches_oracle(runner):
    """The whole memory-pressure trace (swaps and soft resets) until every
    request has finished."""
    sc = workloads.offload_pressure(1)
    run = ParityRun(sc, arrivals=True, runner=runner)
    steps = 0
    for _ in range(600):
        st, g, r, toks = run.step()
        if st == 0:
            _check_all(run, g, r, f"step {run.step_idx - 1}")
        steps += 1
        if (run.next_arrival == len(sc.waiting) and not run.o.running and not run.o.waiting
                and not run.o.swapped):
            break
    assert not run.o.running and not run.o.waiting and not run.o.swapped
    assert run.swap_pairs > 100 and steps > 200


@pytest.mark.parametrize("runner", RUNNERS)
def test_runner_sliding_trace_matches_oracle(runner):
    """Sliding-window layers with recycled pages (-1 table entries), the
    first 120 steps of the trace."""
    sc = workloads.sliding_trace(1)
    run = ParityRun(sc, arrivals=True, runner=runner)
    ran = 0
    for _ in range(120):
        st, g, r, toks = run.step()
        if st == 0:
            _check_all(run, g, r, f"step {run.step_idx - 1}")
            ran += 1
    assert ran > 100
