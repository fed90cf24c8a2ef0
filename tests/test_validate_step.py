"""cb_validate_step: host validation of a step's metadata.

Every step the scheduler emits passes (FIFO, offloading, prefix caching,
sliding windows, graph padding); each kind of corruption fails with a
message that names the row or token and the broken rule.
"""
import numpy as np
import pytest

import workloads
from tests.sched_driver import add_waiting, c_from_config, scenario_to_config


def _cb():
    import paged_attention_continuous_gb300 as cb
    return cb


def _run_and_validate(sc, steps, window=0):
    cb = _cb()
    s = c_from_config(scenario_to_config(sc))
    for r in sc.running:
        s.add_running_request(r.req_id, r.prompt_len, r.output_len, r.num_cached)
    nxt, checked = 0, 0
    for step in range(steps):
        while nxt < len(sc.waiting) and sc.waiting[nxt].arrival_step <= step:
            add_waiting(s, sc.waiting[nxt])
            nxt += 1
        st = s.schedule_step()
        if st["status"] != 0:
            continue
        cb.validate_step(st, num_blocks=sc.num_blocks, block_size=sc.block_size,
                         sliding_window=window)
        checked += 1
        s.step_done()
    return checked


@pytest.mark.parametrize("name", ["offload_pressure", "shared_prefix", "sliding_trace",
                                  "mixed_2048"])
def test_scheduler_steps_validate(name):
    sc = workloads.SCENARIOS[name]()
    assert _run_and_validate(sc, 60, window=sc.sliding_window) > 0


def _good_step():
    # two decodes, one prefill chunk of 5 at offset 11, block size 4, 6 blocks wide
    return {"num_reqs": 3, "num_decodes": 2, "num_tokens": 7,
            "cu_seqlens_q": np.array([0, 1, 2, 7], dtype=np.int32),
            "seq_lens": np.array([9, 4, 16], dtype=np.int32),
            "block_tables": np.array([[3, 4, 5, -1, -1, -1],
                                      [6, -1, -1, -1, -1, -1],
                                      [0, 1, 2, 7, -1, -1]], dtype=np.int32),
            "slot_mapping": np.array([20, 7, 10, 11, 28, 29, 30], dtype=np.int32)}


def test_good_step_passes():
    _cb().validate_step(_good_step(), num_blocks=8, block_size=4)


def _bad(mutate, match, **kw):
    cb = _cb()
    st = _good_step()
    mutate(st)
    with pytest.raises(cb.CBError) as e:
        cb.validate_step(st, num_blocks=kw.get("num_blocks", 8), block_size=4,
                         sliding_window=kw.get("window", 0))
    assert e.value.status == cb.CB_ERR_INVALID_ARG
    assert match in str(e.value), str(e.value)


def test_corruptions_are_named():
    def dec(st): st["cu_seqlens_q"][3] = 1                      # 2 -> 1 decreases
    _bad(dec, "row 2: cu_seqlens_q decreases")
    def two(st): st["cu_seqlens_q"][1] = 2                      # decode row 0 gets 2 tokens
    _bad(two, "decode row 0 has 2 query tokens")
    def short(st): st["seq_lens"][2] = 3                        # seq_len < q_len
    _bad(short, "row 2: seq_len 3 < query length 5")
    def empty(st):
        st["cu_seqlens_q"][:] = [0, 1, 2, 2]
        st["num_tokens"] = 2
    _bad(empty, "row 2: no queries but seq_len 16")
    def long_(st): st["seq_lens"][2] = 25                       # 7 blocks > 6
    _bad(long_, "needs 7 blocks > 6")
    def hole(st): st["block_tables"][0, 1] = -1
    _bad(hole, "row 0: block_tables[1] = -1")
    def far(st): st["block_tables"][2, 3] = 8
    _bad(far, "row 2: block_tables[3] = 8 outside [0, 8)")
    def slot(st): st["slot_mapping"][4] = 32
    _bad(slot, "slot_mapping[4] = 32")
    def past(st): st["num_tokens"] = 6
    _bad(past, "row 2: queries end at 7 > num_tokens 6")


def test_window_allows_recycled_pages_before_it():
    cb = _cb()
    st = _good_step()
    st["block_tables"][2, 0] = -1          # page 0 (keys 0-3) of the chunk row
    st["block_tables"][0, 0] = -1          # page 0 of decode row 0 (keys 0-3)
    # window 5: the chunk's first query (position 11) reads keys 7..11,
    # decode row 0 (position 8) reads keys 4..8: page 0 is never read
    cb.validate_step(st, num_blocks=8, block_size=4, sliding_window=5)
    with pytest.raises(cb.CBError):
        cb.validate_step(st, num_blocks=8, block_size=4, sliding_window=0)
    with pytest.raises(cb.CBError):
        cb.validate_step(st, num_blocks=8, block_size=4, sliding_window=9)


def test_graph_padding_rows_pass():
    cb = _cb()
    st = _good_step()
    st["num_reqs"] = 4
    st["cu_seqlens_q"] = np.array([0, 1, 2, 7, 7], dtype=np.int32)
    st["seq_lens"] = np.array([9, 4, 16, 0], dtype=np.int32)
    st["block_tables"] = np.vstack([st["block_tables"], np.full((1, 6), -1, dtype=np.int32)])
    st["num_tokens"] = 8
    st["slot_mapping"] = np.append(st["slot_mapping"], np.int32(-1))
    cb.validate_step(st, num_blocks=8, block_size=4)
