"""Sliding-window layers on the GPU ("Continuous batching architecture",
Memory management: sliding layers keep a fixed window of recent tokens by
recycling pages): the decode, tensor-core prefill and CUDA-core kernels with
a window against the oracle, with the pages before each window recycled by
the scheduler (their table entries -1 from the second step on).

Bars: bf16 |gpu - oracle| <= 2e-2 + 1e-2 |oracle|; fp32 max-abs <= 1e-4;
scheduler metadata bit-exact and no device error bits (checked by the
harness every step).
"""
import dataclasses

import pytest

import workloads
from tests.gpu_harness import ParityRun, tolerance_ok
from tests.test_gpu_parity import EDGE_CTX, _decode_scenario, _mixed_small

pytestmark = pytest.mark.gpu


def _check(g, r, dtype, what):
    ok, err, excess = tolerance_ok(g, r, dtype)
    assert ok, f"{what}: max err {err:.3e}, worst excess over bound {excess:.3e}"


@pytest.mark.parametrize("W", [1, 16, 17, 100, 5000])
@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f32", 64), ("bf16", 64)])
@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (16, 2), (8, 8)])
def test_decode_window_edges(W, dtype, D, Hq, Hkv):
    sc = dataclasses.replace(_decode_scenario(EDGE_CTX, Hq, Hkv, D, dtype), sliding_window=W)
    run = ParityRun(sc)
    for step in range(3):
        st, g, r, _ = run.step()
        assert st == 0
        _check(g[0], r[0], dtype, f"decode window {W} step {step}")
    if W < 1000:
        assert (run.last["block_tables"][:, 0] < 0).any()   # pages were recycled


@pytest.mark.parametrize("W", [1, 64, 127, 128, 129, 300])
@pytest.mark.parametrize("dtype,Hq,Hkv,D", [("bf16", 32, 8, 128), ("bf16", 16, 16, 128),
                                           ("bf16", 64, 4, 128), ("bf16", 16, 8, 128),
                                           ("f32", 8, 2, 64)])
def test_mixed_steps_window(W, dtype, Hq, Hkv, D):
    """Decodes plus prefill chunks of up to 128 tokens at offsets up to ~600
    (the tensor-core kernel for bf16 / D = 128 at GQA 4, 1, 16 and 2; the
    CUDA-core kernel for fp32): windows shorter than, equal to and longer
    than a 128-key tile."""
    sc = dataclasses.replace(_mixed_small(dtype, Hq, Hkv, D), sliding_window=W)
    run = ParityRun(sc)
    for step in range(5):
        st, g, r, _ = run.step()
        assert st == 0
        _check(g[0], r[0], dtype, f"mixed window {W} step {step}")


def test_sliding_trace_matches_oracle():
    """A trace whose pool only fits because out-of-window pages are
    recycled: every step on both layers until all requests finish."""
    sc = workloads.sliding_trace(0)
    run = ParityRun(sc, arrivals=True)
    ran, dropped = 0, 0
    for _ in range(1000):
        st, g, r, toks = run.step()
        if st == 0:
            for layer in range(sc.num_layers):
                _check(g[layer], r[layer], "bf16", f"step {run.step_idx - 1} layer {layer}")
            dropped += int((run.last["block_tables"][:, 0] < 0).sum())
            ran += 1
        if run.next_arrival == len(sc.waiting) and not run.o.running and not run.o.waiting:
            break
    assert not run.o.running and not run.o.waiting
    assert ran > 200 and dropped > 1000
