"""Fault injection on the scheduler: blocks held away from the pool.

hold_blocks(n) takes blocks exactly as allocation would; release_blocks
returns them to the free queue's tail in the given order.  Pins: a case
derived by hand (a prompt that cannot be admitted while blocks are held,
admitted after a partial release, with the released order visible in its
block table); on random traces with offloading, prefix caching or sliding
windows and random holds and releases, the C++ scheduler equals the oracle
bit for bit, blocks are conserved (in use + free + held = pool), and once
everything is released every request still finishes.
"""
import numpy as np
import pytest

from tests.sched_driver import c_from_config, normalize, oracle_from_config
from tests.test_scheduler_offload import _pressure_trace
from tests.test_scheduler_prefix import _prefix_trace
from tests.test_scheduler_window import _window_trace

CFG = dict(block_size=4, num_blocks=6, max_batch_tokens=16, max_requests_per_batch=4,
           max_prefill_chunk=0, safety_margin=0.0, max_blocks_per_seq=8, free_list=None)


@pytest.mark.parametrize("impl", ["oracle", "c"])
def test_hand_derived_hold_and_release(impl):
    s = (oracle_from_config if impl == "oracle" else c_from_config)(CFG)
    # holding 3 of 6 blocks takes the free queue's head: 0, 1, 2
    assert list(s.hold_blocks(3)) == [0, 1, 2]
    s.add_request(1, 14, 1)
    st = s.schedule_step()
    # a 14-token prompt needs 4 blocks, only 3 are free: nothing fits
    assert st["status"] == 2 and st["num_reqs"] == 0
    # released in the order 1, 0: free queue 3, 4, 5, 1, 0
    s.release_blocks([1, 0])
    st = s.schedule_step()
    assert st["status"] == 0
    assert list(st["block_tables"][0][:4]) == [3, 4, 5, 1]
    assert list(st["slot_mapping"]) == [12, 13, 14, 15, 16, 17, 18, 19, 20, 21, 22, 23, 4, 5]
    assert s.step_done() == [1]
    # block 2 is still held: releasing it twice, or an unheld block, fails
    with pytest.raises(Exception):
        s.release_blocks([2, 2])
    with pytest.raises(Exception):
        s.release_blocks([3])
    s.release_blocks([2])


def _free(s, impl):
    return s.free_list() if impl == "oracle" else s.free


def _drive(s, impl, cfg, reqs, steps, seed):
    """Run a trace with random holds and releases; returns per-step records."""
    rng = np.random.default_rng(seed)
    pending = sorted(reqs, key=lambda r: r["arrival_step"])
    held, out, nxt = [], [], 0
    for step in range(steps):
        while nxt < len(pending) and pending[nxt]["arrival_step"] <= step:
            r = pending[nxt]
            if r.get("tokens") is not None:
                s.add_request(r["id"], r["prompt_len"], r["output_len"], tokens=r["tokens"])
            else:
                s.add_request(r["id"], r["prompt_len"], r["output_len"])
            nxt += 1
        ev = None
        if step < steps // 2:
            u = rng.random()
            if u < 0.15:
                got = [int(b) for b in s.hold_blocks(int(rng.integers(1, 6)))]
                held.extend(got)
                ev = ("hold", got)
            elif u < 0.3 and held:
                k = int(rng.integers(1, len(held) + 1))
                rel = [held[i] for i in rng.permutation(len(held))[:k]]
                s.release_blocks(rel)
                held = [b for b in held if b not in rel]
                ev = ("release", rel)
        elif held:
            s.release_blocks(held)
            ev = ("release", list(held))
            held = []
        st = normalize(s.schedule_step())
        st["event"] = ev
        st["finished"] = list(s.step_done()) if st["status"] == 0 else None
        st["free"] = list(_free(s, impl))
        if impl == "oracle":
            in_use = {b for r in s.running for b in r.blocks if b >= 0}
            assert len(in_use) + len(st["free"]) + len(s.held) == cfg["num_blocks"]
            assert not (in_use & set(s.held)) and not (set(st["free"]) & set(s.held))
        out.append(st)
    return out


def _traces():
    for seed in range(15):
        yield "pressure", _pressure_trace(seed)
        yield "prefix", _prefix_trace(seed, offload=True)
        yield "window", _window_trace(seed, offload=bool(seed % 2))


@pytest.mark.parametrize("case", list(range(45)))
def test_c_matches_oracle_with_holds(case):
    kind, (cfg, reqs) = list(_traces())[case]
    a = _drive(oracle_from_config(cfg), "oracle", cfg, reqs, 240, case)
    b = _drive(c_from_config(cfg), "c", cfg, reqs, 240, case)
    assert a == b


@pytest.mark.parametrize("seed", range(20))
def test_holds_conserve_blocks_and_requests_finish(seed):
    cfg, reqs = _pressure_trace(seed)
    s = oracle_from_config(cfg)
    _drive(s, "oracle", cfg, reqs, 400, seed)          # conservation checked every step
    assert not s.held
    # everything released by the second half: the trace drains
    assert not s.running and not s.waiting and not s.swapped
