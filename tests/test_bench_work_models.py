"""The benchmark's algorithmic work counts, against brute-force counts.

Every roofline fraction bench.py reports divides one of these counts by a
measured time, so they are checked on small steps by enumerating what the
attention definition touches: for decode rows, every K and V row the query
sees (all of them, or the last ``window``) once per KV head plus q and out;
for prefill rows, 4 * D FLOP per query head and per (query, visible key)
pair, with a key visible when it is at or before the query's absolute
position and, with a window, inside it.
"""
import numpy as np
import pytest

import bench


def _step(rows, num_decodes):
    """rows: list of (q_len, seq_len); decode rows first."""
    cu = np.concatenate([[0], np.cumsum([q for q, _ in rows])]).astype(np.int32)
    return {"num_reqs": len(rows), "num_decodes": num_decodes,
            "cu_seqlens_q": cu, "seq_lens": np.asarray([L for _, L in rows], dtype=np.int32),
            "num_tokens": int(cu[-1])}


def _brute_pairs(q_len, L, window):
    n = 0
    for i in range(q_len):
        p = L - q_len + i
        for j in range(L):
            if j <= p and (window == 0 or j > p - window):
                n += 1
    return n


@pytest.mark.parametrize("window", [0, 1, 5, 16, 100])
def test_prefill_flops_match_enumeration(window):
    rng = np.random.default_rng(window + 3)
    rows = [(1, int(rng.integers(1, 50))) for _ in range(3)]           # decodes
    for _ in range(4):
        q = int(rng.integers(1, 40))
        rows.append((q, q + int(rng.integers(0, 60))))
    st = _step(rows, 3)
    Hq, D = 6, 8
    want = sum(4 * D * Hq * _brute_pairs(q, L, window) for q, L in rows[3:])
    assert bench.prefill_flops(st, Hq, D, window) == want


@pytest.mark.parametrize("window", [0, 1, 7, 64])
def test_decode_bytes_match_enumeration(window):
    rng = np.random.default_rng(window + 11)
    rows = [(1, int(rng.integers(1, 200))) for _ in range(9)] + [(17, 40)]
    st = _step(rows, 9)
    Hq, Hkv, D, elem = 8, 2, 16, 2
    keys = sum(_brute_pairs(1, L, window) for _, L in rows[:9])     # keys each decode query sees
    want = keys * Hkv * D * 2 * elem + 9 * Hq * D * 2 * elem
    assert bench.decode_bytes(st, Hq, Hkv, D, elem, window) == want


def test_sub_step_slices_rows_and_tokens():
    st = _step([(1, 10), (1, 20), (5, 30), (3, 3)], 2)
    st["block_tables"] = np.arange(16, dtype=np.int32).reshape(4, 4)
    st["slot_mapping"] = np.arange(st["num_tokens"], dtype=np.int32)
    sub = bench._sub_step(st, 2, 4)
    assert sub["num_reqs"] == 2 and sub["num_decodes"] == 0 and sub["num_tokens"] == 8
    assert list(sub["cu_seqlens_q"]) == [0, 5, 8]
    assert list(sub["seq_lens"]) == [30, 3]
    assert list(sub["slot_mapping"]) == list(range(2, 10))
    assert sub["max_q_len"] == 5 and sub["max_seq_len"] == 30
    dec = bench._sub_step(st, 0, 2)
    assert dec["num_decodes"] == 2 and dec["num_tokens"] == 2


def test_reference_arm_sizes_its_sample_to_the_budget(monkeypatch):
    """The reference arm deals the step's rows round-robin into groups so
    that K + W steps take about --ref-seconds of oracle time, runs group
    i mod n in step i, and reports the timed steps' query tokens over their
    oracle seconds, under the same config object as the GPU arm."""
    import types
    calls = []

    def fake_setup(sc, step, rows, q, k, v, torch, dev):
        return step, None

    def fake_sample(sc, st, pools, rows, prefill_token_cap=None):
        calls.append(list(rows))
        return len(rows), 0.01 * len(rows)   # 10 ms of oracle time per row

    monkeypatch.setattr(bench, "oracle_setup", fake_setup)
    monkeypatch.setattr(bench, "oracle_sample", fake_sample)
    args = types.SimpleNamespace(workload="mixed_2048", steps=20, warmup=3, ref_seconds=2.0)
    line = bench.run_reference(args, 0, 1)
    R = line["config"]["num_reqs"]
    full = calls[0]
    assert full == list(range(R))                      # the sizing pass: every row
    n_parts = int(np.ceil(0.01 * R * 23 / 2.0))
    groups = calls[1:]
    assert len(groups) == 23
    assert groups[0] == list(range(0, R, n_parts))
    assert sorted(r for g in groups[:n_parts] for r in g) == list(range(R))
    timed = groups[3:]
    assert line["value"] == pytest.approx(sum(len(g) for g in timed) /
                                          sum(0.01 * len(g) for g in timed), rel=1e-6)
    assert bench.run_reference(args, 1, 2) is None     # other ranks do no work
