"""Host-side pieces of the step runners, on the CPU.

StepRunner._pack lays a step's metadata out as one int32 run (cu_seqlens_q,
seq_lens, block_tables, slot_mapping) for a single pinned copy; every
runner's device views are slices of it at the returned offsets.  bucket()
gives the padding intervals of the graph runner.
"""
import numpy as np
import pytest

from paged_attention_continuous_gb300.step import StepRunner, bucket


def _host_runner(max_reqs, max_tokens, W):
    # the packing needs no device state: build the object without __init__
    r = object.__new__(StepRunner)
    r.max_reqs, r.max_tokens, r.W = max_reqs, max_tokens, W
    return r


def _step():
    return {"num_reqs": 3, "num_decodes": 2, "num_tokens": 6,
            "cu_seqlens_q": np.array([0, 1, 2, 6], dtype=np.int32),
            "seq_lens": np.array([17, 5, 40], dtype=np.int32),
            "block_tables": np.array([[7, 8, -1], [9, -1, -1], [1, 2, 3]], dtype=np.int32),
            "slot_mapping": np.array([128, 148, 36, 37, 38, 39], dtype=np.int32)}


def test_pack_layout():
    r = _host_runner(4, 8, 3)
    st = _step()
    h = np.full(64, -7, dtype=np.int32)
    n, (o1, o2, o3) = r._pack(st, h)
    assert (o1, o2, o3, n) == (4, 7, 16, 22)
    assert list(h[:o1]) == [0, 1, 2, 6]
    assert list(h[o1:o2]) == [17, 5, 40]
    assert list(h[o2:o3]) == [7, 8, -1, 9, -1, -1, 1, 2, 3]
    assert list(h[o3:n]) == [128, 148, 36, 37, 38, 39]
    assert h[n] == -7                       # nothing written past the run


def test_pack_refuses_oversized_or_misshapen_steps():
    st = _step()
    with pytest.raises(ValueError):
        _host_runner(2, 8, 3)._pack(st, np.zeros(64, np.int32))     # 3 rows > 2
    with pytest.raises(ValueError):
        _host_runner(4, 5, 3)._pack(st, np.zeros(64, np.int32))     # 6 tokens > 5
    with pytest.raises(ValueError):
        _host_runner(4, 8, 4)._pack(st, np.zeros(64, np.int32))     # table width 3 != 4


def test_empty_step_packs_to_one_word():
    r = _host_runner(4, 8, 3)
    st = {"num_reqs": 0, "num_decodes": 0, "num_tokens": 0,
          "cu_seqlens_q": np.zeros(1, np.int32), "seq_lens": np.zeros(0, np.int32),
          "block_tables": np.zeros((0, 3), np.int32), "slot_mapping": np.zeros(0, np.int32)}
    n, _ = r._pack(st, np.zeros(8, np.int32))
    assert n == 1


def test_bucket_intervals():
    assert [bucket(n) for n in (0, 1, 2, 3, 5, 64, 65, 1000)] == [0, 1, 2, 4, 8, 64, 128, 1024]
    assert [bucket(n, 16) for n in (0, 1, 16, 17)] == [0, 16, 16, 32]


class _Ev:
    def record(self, *a):
        pass

    def synchronize(self):
        pass


class _Cuda:
    Event = _Ev


class _TorchStub:
    cuda = _Cuda


def test_graph_runner_pads_to_buckets():
    """3 decodes and 3 prefill rows (chunks 2, 3, 1): buckets (16 tokens,
    4 decode rows, 4 prefill rows, chunk 4); rows are real decodes, one
    decode padding row, real prefills, one prefill padding row; padding rows
    have no queries, seq_len 0 and -1 tables; padding tokens slot -1."""
    import torch
    from paged_attention_continuous_gb300.step import GraphStepRunner
    g = object.__new__(GraphStepRunner)
    g.torch = _TorchStub
    g.swap = None
    g.W, g.T_cap, g.R_cap = 3, 64, 16
    cap = 1024
    g._host = [torch.zeros(cap, dtype=torch.int32) for _ in range(2)]
    g._copied = [None, None]
    g._turn = 0
    g._dev = torch.zeros(cap, dtype=torch.int32)
    st = {"num_reqs": 6, "num_decodes": 3, "num_tokens": 9,
          "cu_seqlens_q": np.array([0, 1, 2, 3, 5, 8, 9], dtype=np.int32),
          "seq_lens": np.array([10, 20, 30, 2, 40, 7], dtype=np.int32),
          "block_tables": np.array([[1, -1, -1], [2, 3, -1], [4, 5, 6], [7, -1, -1],
                                    [8, 9, 10], [11, -1, -1]], dtype=np.int32),
          "slot_mapping": np.arange(100, 109, dtype=np.int32)}
    key, T = g.prepare(st)
    assert key == (16, 4, 4, 4) and T == 9
    d = g._dev.numpy()
    Rb, W = 8, 3
    cu = d[0:Rb + 1]
    sl = d[Rb + 1:2 * Rb + 1]
    bt = d[2 * Rb + 1:2 * Rb + 1 + Rb * W].reshape(Rb, W)
    sm = d[2 * Rb + 1 + Rb * W:2 * Rb + 1 + Rb * W + 16]
    assert list(cu) == [0, 1, 2, 3, 3, 5, 8, 9, 9]
    assert list(sl) == [10, 20, 30, 0, 2, 40, 7, 0]
    assert bt[3].tolist() == [-1, -1, -1] and bt[7].tolist() == [-1, -1, -1]
    assert bt[1].tolist() == [2, 3, -1] and bt[5].tolist() == [8, 9, 10]
    assert list(sm[:9]) == list(range(100, 109)) and (sm[9:] == -1).all()


def test_swap_pool_orders_swap_ins_before_swap_outs(monkeypatch):
    """SwapPool.apply queues every swap-in (slot -> block) before any
    swap-out (block -> slot), each over every layer's K and V, chunked to
    at most 128 pools per call; the ids it passes are the step's pairs."""
    import torch
    import paged_attention_continuous_gb300.step as step_mod
    calls = []

    def fake_kv_swap(src, dst, src_ids, dst_ids, error_word=None):
        calls.append((list(src), list(dst), src_ids.tolist(), dst_ids.tolist()))

    monkeypatch.setattr(step_mod, "kv_swap", fake_kv_swap)
    p = object.__new__(step_mod.SwapPool)
    p.torch = _TorchStub
    layers = 70                                    # 140 pools: two calls per direction
    cache = [("cache", i) for i in range(2 * layers)]
    pool = [("pool", i) for i in range(2 * layers)]
    p._cache, p._pool = cache, pool
    p.swap_blocks = 8
    p.block_bytes = 4096
    p._host = [torch.zeros(32, dtype=torch.int32) for _ in range(2)]
    p._copied = [None, None]
    p._turn = 0
    p._dev = torch.zeros(32, dtype=torch.int32)
    p.error_word = None
    step = {"swap_in": np.array([[3, 10], [5, 11]], dtype=np.int32),      # (slot, block)
            "swap_out": np.array([[20, 3], [21, 6], [22, 7]], dtype=np.int32)}  # (block, slot)
    moved = p.apply(step)
    assert moved == 5 * 2 * layers * 4096
    assert [len(c[0]) for c in calls] == [128, 12, 128, 12]
    for c in calls[:2]:                            # swap-ins: pool -> cache
        assert c[0][0][0] == "pool" and c[1][0][0] == "cache"
        assert c[2] == [3, 5] and c[3] == [10, 11]
    for c in calls[2:]:                            # swap-outs: cache -> pool
        assert c[0][0][0] == "cache" and c[1][0][0] == "pool"
        assert c[2] == [20, 21, 22] and c[3] == [3, 6, 7]
    assert calls[0][0][0] == ("pool", 0) and calls[1][0][0] == ("pool", 128)
    calls.clear()
    assert p.apply({"swap_in": np.zeros((0, 2)), "swap_out": np.zeros((0, 2))}) == 0
    assert not calls


def test_pipelined_runner_dependencies(monkeypatch):
    """PipelinedStepRunner.submit, with recording stand-ins for streams and
    events: step n uses buffer set n % 2; its copy-in waits for the compute
    of step n-2 (same set), its compute waits for its own copy-in and for
    the copy-out of step n-2 (the set's output buffer), and its copy-out
    waits for its compute."""
    import contextlib
    import torch
    from paged_attention_continuous_gb300.step import PipelinedStepRunner
    log = []

    class Ev:
        n = 0

        def __init__(self):
            Ev.n += 1
            self.id = Ev.n
            self.tag = None

        def record(self, stream=None):
            self.tag = (stream.name, len(log))
            log.append(("record", stream.name, self.id))

        def synchronize(self):
            pass

    class Stream:
        def __init__(self, name):
            self.name = name

        def wait_event(self, ev):
            log.append(("wait", self.name, ev.id))

    current = {"s": None}

    @contextlib.contextmanager
    def stream_ctx(s):
        prev, current["s"] = current["s"], s
        yield
        current["s"] = prev

    class Cuda:
        Event = Ev
        stream = staticmethod(stream_ctx)

    class TorchStub:
        cuda = Cuda

    r = object.__new__(PipelinedStepRunner)
    r.torch = TorchStub
    r.swap = None
    r.max_reqs, r.max_tokens, r.W = 4, 8, 3
    r.k_cache = [None]
    L = 1
    mk = lambda: [torch.zeros(8, 2, 4) for _ in range(L)]
    r._sets = [dict(q=mk(), k=mk(), v=mk(), out=mk(), meta=torch.zeros(64, dtype=torch.int32),
                    stage=torch.zeros(64, dtype=torch.int32)) for _ in range(2)]
    r.in_stream, r.compute_stream, r.out_stream = Stream("in"), Stream("compute"), Stream("out")
    r._copied_in, r._computed, r._copied_out = [None, None], [None, None], [None, None]
    r._slot = 0
    runs = []
    r.run = lambda ds, q, k, v, layer=0, out=None: runs.append(current["s"].name)
    step = _step()
    events = []
    for n in range(4):
        before = len(log)
        ev = r.submit(step, torch.zeros(6, 2, 4), torch.zeros(6, 2, 4), torch.zeros(6, 2, 4),
                      torch.zeros(6, 2, 4))
        events.append([e for e in log[before:]])
    assert runs == ["compute"] * 4
    # event ids per step: copy_in, computed, copied_out are created in order
    ids = []
    for n, evs in enumerate(events):
        rec = [e for e in evs if e[0] == "record"]
        assert [e[1] for e in rec] == ["in", "compute", "out"]
        ids.append({"in": rec[0][2], "comp": rec[1][2], "out": rec[2][2]})
    for n, evs in enumerate(events):
        waits = [(e[1], e[2]) for e in evs if e[0] == "wait"]
        want = []
        if n >= 2:
            want.append(("in", ids[n - 2]["comp"]))
        want.append(("compute", ids[n]["in"]))
        if n >= 2:
            want.append(("compute", ids[n - 2]["out"]))
        want.append(("out", ids[n]["comp"]))
        assert waits == want, (n, waits, want)
