"""Multi-process host logic of the benchmark's N>1 path, on CPU with gloo.

With several GPUs each process serves its own request set (requests are
independent, so they shard with no data-path exchange) and the only
collectives are the timing ones: the step time is the MAX over ranks and the
token count the SUM.  Two gloo ranks check that

* each rank's workload comes from its own seed and differs from the other's;
* on every rank the C scheduler's first batches match the oracle scheduler's
  bit for bit (each rank is a complete, independent replica);
* the reductions bench.py applies give max(time) and sum(tokens).
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, workload, steps, q):
    try:
        sys.path.insert(0, ROOT)
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        dist.init_process_group("gloo", rank=rank, world_size=world)
        import bench
        import paged_attention_continuous_gb300 as cb
        from tests.sched_driver import load_scenario, normalize, oracle_from_config, \
            scenario_to_config

        sc = bench.rank_scenario(workload, rank)
        c = bench.load_c_scheduler(cb, sc)
        o = oracle_from_config(scenario_to_config(sc))
        load_scenario(o, sc)
        tokens = []
        for i in range(steps):
            a, b = normalize(c.schedule_step()), normalize(o.schedule_step())
            assert a == b, f"rank {rank} step {i}"
            if a["status"] != 0:
                break
            tokens.append(int(a["cu_seqlens_q"][-1]))
            assert list(c.step_done()) == list(o.step_done())
        assert c.free == list(o.free)
        t = 1.0 + rank  # a stand-in per-rank step time
        t_max = bench.reduce_over_ranks(dist, t, dist.ReduceOp.MAX, "cpu")
        n_sum = bench.reduce_over_ranks(dist, tokens[0], dist.ReduceOp.SUM, "cpu")
        fp = [int(x) for x in sc.free_list[:8]] + [r.req_id for r in sc.running[:4]] + \
            [int(r.num_cached) for r in sc.running[:4]]
        q.put((rank, tokens, t_max, n_sum, fp))
        dist.barrier()
        dist.destroy_process_group()
    except BaseException as e:  # report, never hang the parent
        q.put((rank, "error", repr(e)))
        raise


@pytest.mark.parametrize("workload,steps", [("mixed_2048", 3), ("decode_64", 3)])
def test_two_gloo_ranks_are_independent_replicas(workload, steps):
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, workload, steps, q))
             for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    try:
        for _ in range(world):
            item = q.get(timeout=240)
            assert item[1] != "error", item
            res[item[0]] = item
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    (_, tok0, tmax0, nsum0, fp0), (_, tok1, tmax1, nsum1, fp1) = res[0], res[1]
    assert fp0 != fp1, "ranks must draw different request sets"
    assert tmax0 == tmax1 == 2.0
    assert nsum0 == nsum1 == tok0[0] + tok1[0]
    assert len(tok0) == len(tok1) == steps
