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
