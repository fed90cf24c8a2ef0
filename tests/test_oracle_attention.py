"""Pins for the oracle attention and paged append.

Each test checks the oracle against something other than itself: the
worked example of the Chunked Prefill page, torch's dense
scaled_dot_product_attention (a library routine for the one-request special
case), explicit loops on tiny inputs, and invariants that hold exactly.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import workloads
from oracle import attention as oatt
from oracle import paged_kv
from oracle.scheduler import FifoScheduler

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _run_prompts_through_paging(prompts_q, prompts_k, prompts_v, *, chunk,
                                num_blocks, free_list, block_size=16,
                                max_reqs=8, scale=None):
    """Prefill each prompt (lists of [L, H, D] float64 arrays) through the
    oracle scheduler + paged append + paged attention.  Returns per-prompt
    outputs [L, Hq, D] assembled from all steps, and the chunk sizes seen."""
    Hq, D = prompts_q[0].shape[1:]
    Hkv = prompts_k[0].shape[1]
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    max_len = max(q.shape[0] for q in prompts_q)
    s = FifoScheduler(block_size=block_size, num_blocks=num_blocks,
                      max_batch_tokens=chunk, max_requests_per_batch=max_reqs,
                      max_blocks_per_seq=-(-max_len // block_size),
                      safety_margin=0.0, free_list=free_list)
    for i, q in enumerate(prompts_q):
        s.add_request(i, q.shape[0], 1)
    kc = np.zeros((num_blocks, Hkv, block_size, D))
    vc = np.zeros_like(kc)
    outs = [np.zeros_like(q) for q in prompts_q]
    chunks = []
    while True:
        st = s.schedule_step()
        if st["num_reqs"] == 0:
            break
        T = st["num_tokens"]
        qb = np.zeros((T, Hq, D)); kb = np.zeros((T, Hkv, D)); vb = np.zeros((T, Hkv, D))
        for i, rid in enumerate(st["req_ids"]):
            t0, t1 = st["cu_seqlens_q"][i], st["cu_seqlens_q"][i + 1]
            p1 = st["seq_lens"][i]; p0 = p1 - (t1 - t0)
            qb[t0:t1] = prompts_q[rid][p0:p1]
            kb[t0:t1] = prompts_k[rid][p0:p1]
            vb[t0:t1] = prompts_v[rid][p0:p1]
            chunks.append((int(rid), int(t1 - t0)))
        paged_kv.append(kc, vc, kb, vb, st["slot_mapping"], block_size)
        o = oatt.paged_attention(qb, kc, vc, st["cu_seqlens_q"], st["seq_lens"],
                                 st["block_tables"], block_size, scale)
        for i, rid in enumerate(st["req_ids"]):
            t0, t1 = st["cu_seqlens_q"][i], st["cu_seqlens_q"][i + 1]
            p1 = st["seq_lens"][i]; p0 = p1 - (t1 - t0)
            outs[rid][p0:p1] = o[t0:t1]
        s.step_done()
    return outs, chunks


def test_worked_example_chunked_equals_one_shot():
    with open(os.path.join(GOLDEN, "chunked_prefill_worked_example.json")) as f:
        g = json.load(f)
    q, k, v = workloads.worked_example_qkv()            # [1, 8, 1000, 64]
    # [L, H, D] float64 views of the float32 draw
    qn = q[0].permute(1, 0, 2).double().numpy()
    kn = k[0].permute(1, 0, 2).double().numpy()
    vn = v[0].permute(1, 0, 2).double().numpy()
    sc = workloads.chunked_prefill_1000()
    outs, chunks = _run_prompts_through_paging([qn], [kn], [vn], chunk=g["chunk"],
                                               num_blocks=sc.num_blocks,
                                               free_list=sc.free_list)
    assert [c for _, c in chunks] == g["chunks"]
    chunked = outs[0]
    one_shot = oatt.dense_causal_attention(qn, kn, vn, 1.0 / math.sqrt(g["head_dim"]))
    # the page's own check
    assert np.allclose(one_shot, chunked, atol=g["atol"], rtol=0)
    # the definition reached exactly up to rounding order
    assert np.max(np.abs(one_shot - chunked)) < 1e-12
    # library routine, special case of one request: torch SDPA in float64
    ref = torch.nn.functional.scaled_dot_product_attention(
        q.double(), k.double(), v.double(), is_causal=True)[0].permute(1, 0, 2).numpy()
    assert np.max(np.abs(ref - one_shot)) < 1e-12
    # the page's float32 one-shot vs chunked pass agrees with the oracle to
    # float32 accuracy
    ref32 = torch.nn.functional.scaled_dot_product_attention(
        q, k, v, is_causal=True)[0].permute(1, 0, 2).double().numpy()
    assert np.max(np.abs(ref32 - chunked)) < 1e-5


@pytest.mark.parametrize("Hq,Hkv,L,D", [(4, 4, 37, 16), (8, 2, 50, 32), (6, 3, 19, 8), (4, 1, 64, 16)])
def test_dense_matches_torch_sdpa_gqa(Hq, Hkv, L, D):
    rng = np.random.default_rng(Hq * 100 + L)
    q = rng.standard_normal((L, Hq, D)); k = rng.standard_normal((L, Hkv, D))
    v = rng.standard_normal((L, Hkv, D))
    scale = 1.0 / math.sqrt(D)
    got = oatt.dense_causal_attention(q, k, v, scale)
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]
    tk = torch.from_numpy(k).permute(1, 0, 2)[None]
    tv = torch.from_numpy(v).permute(1, 0, 2)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, is_causal=True, enable_gqa=True)[0].permute(1, 0, 2).numpy()
    assert np.max(np.abs(ref - got)) < 1e-12


def _brute_force(q_tok, k_tok, v_tok, scale):
    """Explicit loops: q_tok [L, Hq, D], k_tok/v_tok [L, Hkv, D] of ONE
    request in token order (no paging); query i attends keys 0..i."""
    L, Hq, D = q_tok.shape
    Hkv = k_tok.shape[1]
    out = np.zeros((L, Hq, D))
    for i in range(L):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            scores = []
            for j in range(i + 1):
                dot = 0.0
                for d in range(D):
                    dot += q_tok[i, h, d] * k_tok[j, g, d]
                scores.append(scale * dot)
            m = max(scores)
            w = [math.exp(s - m) for s in scores]
            z = sum(w)
            for d in range(D):
                out[i, h, d] = sum(w[j] * v_tok[j, g, d] for j in range(i + 1)) / z
    return out


@pytest.mark.parametrize("case", [
    dict(lens=[1, 17, 3], Hq=2, Hkv=1, D=4, chunk=8, bs=4),
    dict(lens=[40, 5], Hq=4, Hkv=2, D=3, chunk=16, bs=16),
    dict(lens=[16, 15, 33], Hq=1, Hkv=1, D=5, chunk=7, bs=4),
])
def test_brute_force_tiny(case):
    rng = np.random.default_rng(len(case["lens"]) * 7 + case["D"])
    qs = [rng.standard_normal((L, case["Hq"], case["D"])) for L in case["lens"]]
    ks = [rng.standard_normal((L, case["Hkv"], case["D"])) for L in case["lens"]]
    vs = [rng.standard_normal((L, case["Hkv"], case["D"])) for L in case["lens"]]
    nb = sum(-(-L // case["bs"]) for L in case["lens"]) + 3
    free = rng.permutation(nb).tolist()
    outs, _ = _run_prompts_through_paging(qs, ks, vs, chunk=case["chunk"], num_blocks=nb,
                                          free_list=free, block_size=case["bs"])
    scale = 1.0 / math.sqrt(case["D"])
    for q, k, v, o in zip(qs, ks, vs, outs):
        assert np.max(np.abs(_brute_force(q, k, v, scale) - o)) < 1e-12


def _three_prompts(seed=3, D=16, Hq=4, Hkv=2):
    rng = np.random.default_rng(seed)
    lens = [70, 33, 129]
    qs = [rng.standard_normal((L, Hq, D)) for L in lens]
    ks = [rng.standard_normal((L, Hkv, D)) for L in lens]
    vs = [rng.standard_normal((L, Hkv, D)) for L in lens]
    return qs, ks, vs


def test_paging_is_invisible_permuted_blocks():
    qs, ks, vs = _three_prompts()
    a, _ = _run_prompts_through_paging(qs, ks, vs, chunk=64, num_blocks=40,
                                       free_list=list(range(40)))
    b, _ = _run_prompts_through_paging(qs, ks, vs, chunk=64, num_blocks=40,
                                       free_list=np.random.default_rng(9).permutation(40).tolist())
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_chunk_size_invariance():
    qs, ks, vs = _three_prompts()
    ref = [oatt.dense_causal_attention(q, k, v, 0.25) for q, k, v in zip(qs, ks, vs)]
    for chunk in (1, 7, 16, 256):
        got, _ = _run_prompts_through_paging(qs, ks, vs, chunk=chunk, num_blocks=40,
                                             free_list=list(range(40)))
        for r, g in zip(ref, got):
            assert np.max(np.abs(r - g)) < 1e-12


def test_seq_len_one_returns_v0():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 4, 8)); k = rng.standard_normal((1, 2, 8))
    v = rng.standard_normal((1, 2, 8))
    o = oatt.dense_causal_attention(q, k, v, 0.3)
    for h in range(4):
        assert np.array_equal(o[0, h], v[0, h // 2])


def test_identical_keys_give_running_mean_of_v():
    rng = np.random.default_rng(6)
    L = 25
    q = rng.standard_normal((L, 2, 8))
    k = np.repeat(rng.standard_normal((1, 1, 8)), L, axis=0)
    v = rng.standard_normal((L, 1, 8))
    o = oatt.dense_causal_attention(q, k, v, 0.5)
    for i in range(L):
        assert np.allclose(o[i, 0], v[:i + 1, 0].mean(axis=0), atol=1e-14, rtol=0)


def test_append_brute_force_slot_walk():
    rng = np.random.default_rng(8)
    nb, Hkv, bs, D, T = 6, 2, 4, 3, 9
    kc = np.zeros((nb, Hkv, bs, D)); vc = np.zeros_like(kc)
    kn = rng.standard_normal((T, Hkv, D)); vn = rng.standard_normal((T, Hkv, D))
    slots = np.array([5, 0, -1, 23, 12, 13, -1, 7, 1], dtype=np.int32)
    paged_kv.append(kc, vc, kn, vn, slots, bs)
    flat_k = kc.transpose(0, 2, 1, 3).reshape(nb * bs, Hkv, D)
    flat_v = vc.transpose(0, 2, 1, 3).reshape(nb * bs, Hkv, D)
    written = set()
    for t, s in enumerate(slots):
        if s >= 0:
            assert np.array_equal(flat_k[s], kn[t]) and np.array_equal(flat_v[s], vn[t])
            written.add(int(s))
    for s in range(nb * bs):
        if s not in written:
            assert not flat_k[s].any() and not flat_v[s].any()


def test_mistakes_are_caught():
    """A plausible slip anywhere in the attention definition (scale, causal
    offset, GQA mapping) changes the result beyond the pins' tolerance."""
    rng = np.random.default_rng(11)
    L, Hq, Hkv, D = 21, 4, 2, 8
    q = rng.standard_normal((L, Hq, D)); k = rng.standard_normal((L, Hkv, D))
    v = rng.standard_normal((L, Hkv, D))
    good = _brute_force(q, k, v, 1 / math.sqrt(D))
    assert np.max(np.abs(oatt.dense_causal_attention(q, k, v, 1 / math.sqrt(D)) - good)) < 1e-12
    assert np.max(np.abs(oatt.attend_one_request(q, k, v, 1, 1 / math.sqrt(D)) - good)) > 1e-3
    assert np.max(np.abs(oatt.dense_causal_attention(q, k, v, 1 / D) - good)) > 1e-3
    k_swapped = k[:, ::-1, :]
    assert np.max(np.abs(oatt.dense_causal_attention(q, k_swapped, v[:, ::-1, :], 1 / math.sqrt(D)) - good)) > 1e-3
