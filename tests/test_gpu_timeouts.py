"""Bounded device waits that run out, without a GPU fault.

Every wait in the attention kernels (a page or tile copy landing, a tensor-
core result, a turn of the other softmax warpgroup) is bounded: when one
runs out the kernel records CB_DEVERR_TIMEOUT, drains what it started and
returns, and the workspace stays ready for the next call.  The test hook
cb_debug_inject_wait_timeout shortens the bound to a few milliseconds and
withholds the copies of one decode work item, or of one K tile of the
prefill kernel's first CTA, so that the wait on them runs out; nothing
faults and nothing hangs.  After each such call the hook is cleared and the
same step runs again on the same workspace: it must report no error and
match the oracle.
"""
import pytest

import workloads
from tests.gpu_harness import ParityRun, tolerance_ok
from tests.sched_driver import c_from_config, load_scenario, scenario_to_config
from tests.test_gpu_parity import _decode_scenario, _mixed_small

pytestmark = pytest.mark.gpu

LIMIT_NS = 5_000_000  # 5 ms


def _cb():
    import paged_attention_continuous_gb300 as cb
    return cb


def _faulty_then_correct(sc, decode_item=-1, prefill_tile=-1):
    cb = _cb()
    run = ParityRun(sc)
    # the step the parity run will schedule first, from a scheduler of its own
    side = c_from_config(scenario_to_config(sc))
    load_scenario(side, sc)
    st = side.schedule_step()
    T = st["num_tokens"]
    seeds = [workloads.step_seed(sc.seed, 0, 0, w) for w in range(3)]
    q = workloads.token_tensors(T, sc.num_q_heads, sc.head_dim, seed=seeds[0], dtype=sc.dtype,
                                scale=sc.value_scale, device="cuda")
    k = workloads.token_tensors(T, sc.num_kv_heads, sc.head_dim, seed=seeds[1], dtype=sc.dtype,
                                scale=sc.value_scale, device="cuda")
    v = workloads.token_tensors(T, sc.num_kv_heads, sc.head_dim, seed=seeds[2], dtype=sc.dtype,
                                scale=sc.value_scale, device="cuda")
    ds = run.runner.upload(st)
    try:
        cb.inject_wait_timeout(LIMIT_NS, decode_item, prefill_tile)
        # the append writes the same K/V the real step writes again below
        run.runner.run(ds, q, k, v)
    finally:
        cb.inject_wait_timeout(0, -1, -1)
    bits = run.runner.workspace.read_errors()
    assert bits & cb.DEVERR_TIMEOUT, f"error bits {bits:#x}"
    # the same step on the same workspace, hook cleared: no error, oracle parity
    status, g, r, toks = run.step()
    assert status == 0 and len(toks) == T
    ok, err, excess = tolerance_ok(g[0], r[0], sc.dtype)
    assert ok, f"after the timeout: max err {err:.3e}, excess {excess:.3e}"


@pytest.mark.parametrize("item", [0, 57])
def test_decode_wait_runs_out_then_workspace_is_clean(item):
    """Long rows cut into many splits: the warp holding the withheld item
    gives up on it, still counts every split it was dealt (so each row's
    split counter returns to zero), and the next call is exact."""
    ctx = [3000, 5000, 2000, 7000, 4100, 900, 6000, 2500, 33, 8000, 1200, 3500]
    sc = _decode_scenario(ctx, 32, 8, 128, "bf16")
    _faulty_then_correct(sc, decode_item=item)


def test_prefill_wait_runs_out_then_next_call_is_correct():
    """The first CTA of the tensor-core prefill kernel never gets its first
    K tile: its MMA issuer, softmax warpgroups and producers give up within
    the bound and the CTA returns; the next call is exact."""
    sc = _mixed_small("bf16", 32, 8, 128)
    _faulty_then_correct(sc, prefill_tile=0)
