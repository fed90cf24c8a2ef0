"""Oracle attention (TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__``).

What is computed (*Chunked Prefill*, Ultralytics glossary, section "How
chunked prefill works", and its PyTorch example): every chunk attends, under a
causal mask over ABSOLUTE positions, to the cached keys/values of all earlier
chunks plus its own; so query i of a chunk that starts at position ``start``
sees keys 0 .. start+i.  Chunking therefore only changes when prompt tokens
are processed, never the result.

For request r with ``q_len`` scheduled tokens and ``seq_len`` tokens in the
cache after this step's append, query token i sits at absolute position
p = seq_len - q_len + i and, for query head h,

    o[t, h] = sum_{j<=p} softmax_j(scale * q[t,h] . k_r[j, g]) * v_r[j, g]

with g = h // (Hq / Hkv) (grouped-query heads share KV head g in contiguous
groups; the pages do not discuss GQA) and scale = 1/sqrt(head_dim) (the
default of the example's ``scaled_dot_product_attention``).  K/V of request r
are read from the paged cache through its block table (*vLLM serving
internals*, "PagedAttention as a virtual memory system").

Sliding-window layers (*Continuous batching architecture*, the paragraph on
sliding attention under Memory management: such layers keep only a fixed
window of the most recent tokens): with window W > 0 the query at position
p sees only keys p-W+1 .. p (the W most recent tokens, its own included);
W = 0 means full attention.  Keys before a row's window are never read, so
their blocks may already have been recycled (-1 in the block table).

Arithmetic is float64 with the max subtracted before exponentiation.  A
matrix product per (request, head) is the only library step.

Parity: pinned by (i) the worked example (1000-token prompt in chunks of
256/256/256/232 equals one-shot), (ii) torch's scaled_dot_product_attention
on dense inputs (a special case), (iii) brute force loops on tiny inputs,
(iv) invariants (permuted blocks, chunk sizes, seq_len = 1 -> v[0],
identical keys -> mean of v).
"""
from __future__ import annotations

import numpy as np


def gather_kv(cache: np.ndarray, block_table: np.ndarray, seq_len: int,
              block_size: int, first: int = 0) -> np.ndarray:
    """Rows first..seq_len-1 of one request, [seq_len - first, Hkv, D], read
    through its block table."""
    pos = np.arange(first, seq_len)
    blocks = block_table[pos // block_size]
    if len(pos) and blocks.min() < 0:
        raise ValueError("block table shorter than seq_len")
    return cache[blocks, :, pos % block_size, :]


def attend_one_request(q: np.ndarray, K: np.ndarray, V: np.ndarray,
                       start: int, scale: float, window: int = 0,
                       first: int = 0) -> np.ndarray:
    """q [q_len, Hq, D]; K, V [n, Hkv, D] (float64) hold the keys at absolute
    positions first .. first+n-1; query i at absolute position start + i
    attends keys 0..start+i, or only start+i-window+1 .. start+i when
    window > 0.  Returns [q_len, Hq, D]."""
    q_len, Hq, D = q.shape
    seq_len, Hkv, _ = K.shape
    group = Hq // Hkv
    out = np.zeros((q_len, Hq, D), dtype=np.float64)
    qpos = start + np.arange(q_len)[:, None]
    kpos = first + np.arange(seq_len)[None, :]
    allowed = kpos <= qpos                                  # [q_len, seq_len]
    if window > 0:
        allowed &= kpos > qpos - window
    for h in range(Hq):
        g = h // group
        s = scale * (q[:, h, :] @ K[:, g, :].T)             # [q_len, seq_len]
        s = np.where(allowed, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        w = np.exp(s)
        w = w / w.sum(axis=1, keepdims=True)
        out[:, h, :] = w @ V[:, g, :]
    return out


def paged_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                    cu_seqlens_q: np.ndarray, seq_lens: np.ndarray,
                    block_tables: np.ndarray, block_size: int, scale: float,
                    requests=None, window: int = 0) -> np.ndarray:
    """q [T, Hq, D]; caches [num_blocks, Hkv, bs, D].  Returns float64
    [T, Hq, D].  ``requests`` optionally restricts the work to a subset of
    request indices (other rows are left zero); ``window`` > 0 selects
    sliding-window attention."""
    q = np.asarray(q, dtype=np.float64)
    T, Hq, D = q.shape
    out = np.zeros((T, Hq, D), dtype=np.float64)
    R = len(seq_lens)
    idx = range(R) if requests is None else requests
    for r in idx:
        t0, t1 = int(cu_seqlens_q[r]), int(cu_seqlens_q[r + 1])
        L = int(seq_lens[r])
        if t1 == t0:
            continue
        start = L - (t1 - t0)
        first = max(0, start - window + 1) if window > 0 else 0
        K = gather_kv(k_cache, block_tables[r], L, block_size, first).astype(np.float64)
        V = gather_kv(v_cache, block_tables[r], L, block_size, first).astype(np.float64)
        out[t0:t1] = attend_one_request(q[t0:t1], K, V, start, scale, window, first)
    return out


def dense_causal_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                           scale: float) -> np.ndarray:
    """One-shot prefill of a whole prompt: q, k, v [L, H, D] (MHA or GQA with
    k/v [L, Hkv, D]); query i attends keys 0..i."""
    return attend_one_request(np.asarray(q, np.float64), np.asarray(k, np.float64),
                              np.asarray(v, np.float64), 0, scale)
