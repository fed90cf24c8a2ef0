"""One serving step through the C ABI: upload the scheduler's metadata, append
the step's new K/V into the paged cache, run paged attention.

"vLLM serving internals", What the scheduler looks like: each iteration
schedules a batch of prefill chunks and decode tokens and runs them in one
forward pass.  This module is the attention part of that pass for one or
more stacked layers: ``StepRunner.upload`` moves a step's host metadata
(``cu_seqlens_q``, ``seq_lens``, ``block_tables``, ``slot_mapping``) to the
device in ONE copy from pinned memory; ``StepRunner.run`` calls
``cb_kv_append`` then ``cb_paged_attention`` on the current stream.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

from . import Workspace, kv_append, paged_attention


@dataclasses.dataclass
class DeviceStep:
    num_reqs: int
    num_tokens: int
    num_decodes: int
    max_q_len: int
    max_seq_len: int
    cu_seqlens_q: object    # device int32 views into one packed buffer
    seq_lens: object
    block_tables: object
    slot_mapping: object
    h2d_bytes: int


class StepRunner:
    def __init__(self, *, num_blocks: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                 dtype: str, max_reqs: int, max_tokens: int, max_blocks_per_seq: int,
                 num_layers: int = 1, block_size: int = 16, device: str = "cuda",
                 scale: Optional[float] = None, zero_cache: bool = True):
        import torch
        self.torch = torch
        self.dt = {"bf16": torch.bfloat16, "f32": torch.float32}[dtype]
        self.Hq, self.Hkv, self.D = num_q_heads, num_kv_heads, head_dim
        self.block_size = block_size
        self.num_blocks = num_blocks
        self.max_reqs, self.max_tokens = max_reqs, max_tokens
        self.W = max_blocks_per_seq
        self.scale = 1.0 / math.sqrt(head_dim) if scale is None else scale
        alloc = torch.zeros if zero_cache else torch.empty
        shape = (num_blocks, num_kv_heads, block_size, head_dim)
        self.k_cache = [alloc(shape, dtype=self.dt, device=device) for _ in range(num_layers)]
        self.v_cache = [alloc(shape, dtype=self.dt, device=device) for _ in range(num_layers)]
        self.workspace = Workspace(max_reqs, num_q_heads, num_kv_heads, head_dim, device=device)
        cap = (max_reqs + 1) + max_reqs + max_reqs * max_blocks_per_seq + max_tokens
        # two pinned staging buffers, used in turn: a buffer is refilled only
        # after the copy that last read it has executed (its event), since
        # the host may run steps ahead of the device
        self._host = [torch.empty(cap, dtype=torch.int32, pin_memory=True) for _ in range(2)]
        self._copied = [None, None]
        self._turn = 0
        self._dev = torch.empty(cap, dtype=torch.int32, device=device)

    def upload(self, step: dict, stream=None) -> DeviceStep:
        """Copy a step's metadata to the device (one pinned copy on the
        current stream).  The returned arrays stay valid until the next
        upload on this runner; kernels that use them must be queued on the
        same stream before that next upload."""
        R, T = int(step["num_reqs"]), int(step["num_tokens"])
        if R > self.max_reqs or T > self.max_tokens:
            raise ValueError("step larger than the runner was sized for")
        W = self.W
        bt = np.asarray(step["block_tables"], dtype=np.int32).reshape(R, -1)
        if bt.shape[1] != W:
            raise ValueError("block_tables width differs from max_blocks_per_seq")
        n = (R + 1) + R + R * W + T
        b = self._turn
        self._turn ^= 1
        if self._copied[b] is not None:
            self._copied[b].synchronize()
        h = self._host[b].numpy()
        o = 0
        h[o:o + R + 1] = step["cu_seqlens_q"]; o1 = o + R + 1
        h[o1:o1 + R] = step["seq_lens"]; o2 = o1 + R
        h[o2:o2 + R * W] = bt.reshape(-1); o3 = o2 + R * W
        h[o3:o3 + T] = step["slot_mapping"]
        self._dev[:n].copy_(self._host[b][:n], non_blocking=True)
        ev = self.torch.cuda.Event()
        ev.record()
        self._copied[b] = ev
        d = self._dev
        return DeviceStep(R, T, int(step["num_decodes"]), int(step["max_q_len"]) if "max_q_len" in step
                          else int(np.diff(step["cu_seqlens_q"]).max(initial=1)),
                          int(step["max_seq_len"]) if "max_seq_len" in step
                          else int(np.max(step["seq_lens"], initial=1)),
                          d[0:R + 1], d[o1:o1 + R], d[o2:o2 + R * W].view(R, W), d[o3:o3 + T],
                          4 * n)

    def run(self, ds: DeviceStep, q, k_new, v_new, layer: int = 0, out=None):
        """Append this step's K/V for ``layer`` and attend.  q [T, Hq, D],
        k_new/v_new [T, Hkv, D] on the device.  Returns out [T, Hq, D]."""
        kc, vc = self.k_cache[layer], self.v_cache[layer]
        kv_append(k_new, v_new, ds.slot_mapping, kc, vc)
        return paged_attention(q, kc, vc, ds.cu_seqlens_q, ds.seq_lens, ds.block_tables,
                               num_decodes=ds.num_decodes, max_q_len=ds.max_q_len,
                               max_seq_len=ds.max_seq_len, scale=self.scale,
                               workspace=self.workspace, out=out)


def bucket(n: int, lo: int = 1) -> int:
    """Smallest power of two >= n (>= lo); 0 for n <= 0."""
    if n <= 0:
        return 0
    b = lo
    while b < n:
        b *= 2
    return b


class GraphStepRunner:
    """A whole step -- every layer's cb_kv_append + cb_paged_attention --
    replayed from a CUDA graph.

    "Continuous batching architecture" (HF Transformers docs) pads a step's
    shapes to a few intervals so that captured graphs can be reused; here
    the step is padded up to power-of-two buckets of (tokens, decode rows,
    prefill rows, longest prefill chunk).  Padding rows have query length 0
    and seq_len 0 (the kernels skip them), padding tokens slot -1 (the append
    skips them), so one graph per bucket serves every step that fits it.  A
    graph is captured the first time its bucket is met, after one uncaptured
    run of the same launches.

    Per step: ``prepare(step)`` pads and uploads the metadata (one pinned
    copy into a static device buffer, two pinned buffers used in turn) and
    returns the bucket; the caller writes the step's q/k/v rows into
    ``q_buf[layer][:T]``, ``k_buf[layer][:T]``, ``v_buf[layer][:T]``; ``run(key)``
    replays the graph; the outputs are ``out_buf[layer][:T]``.
    """

    def __init__(self, *, num_blocks: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                 dtype: str, max_reqs: int, max_tokens: int, max_blocks_per_seq: int,
                 num_layers: int = 1, block_size: int = 16, device: str = "cuda",
                 scale: Optional[float] = None, zero_cache: bool = True):
        import torch
        self.torch = torch
        self.dt = {"bf16": torch.bfloat16, "f32": torch.float32}[dtype]
        self.Hq, self.Hkv, self.D = num_q_heads, num_kv_heads, head_dim
        self.block_size = block_size
        self.W = max_blocks_per_seq
        self.L = num_layers
        self.scale = 1.0 / math.sqrt(head_dim) if scale is None else scale
        self.R_cap = 2 * bucket(max_reqs)     # padded decode rows + padded prefill rows
        self.T_cap = bucket(max_tokens, 16)
        alloc = torch.zeros if zero_cache else torch.empty
        shape = (num_blocks, num_kv_heads, block_size, head_dim)
        self.k_cache = [alloc(shape, dtype=self.dt, device=device) for _ in range(num_layers)]
        self.v_cache = [alloc(shape, dtype=self.dt, device=device) for _ in range(num_layers)]
        self.workspace = Workspace(self.R_cap, num_q_heads, num_kv_heads, head_dim, device=device)
        mk = lambda h: [torch.zeros(self.T_cap, h, head_dim, dtype=self.dt, device=device)
                        for _ in range(num_layers)]
        self.q_buf, self.k_buf, self.v_buf = mk(num_q_heads), mk(num_kv_heads), mk(num_kv_heads)
        self.out_buf = mk(num_q_heads)
        cap = (self.R_cap + 1) + self.R_cap + self.R_cap * self.W + self.T_cap
        self._host = [torch.empty(cap, dtype=torch.int32, pin_memory=True) for _ in range(2)]
        self._copied = [None, None]
        self._turn = 0
        self._dev = torch.empty(cap, dtype=torch.int32, device=device)
        self.graphs = {}
        self.pool = None

    def prepare(self, step: dict):
        """Pad the step to its bucket and upload it; returns (key, T)."""
        R, T, nd = int(step["num_reqs"]), int(step["num_tokens"]), int(step["num_decodes"])
        npf = R - nd
        cu = np.asarray(step["cu_seqlens_q"], dtype=np.int64)
        max_q = int(np.diff(cu[nd:]).max(initial=0)) if npf else 0
        key = (bucket(T, 16), bucket(nd), bucket(npf), bucket(max_q))
        Tb, ndb, npb, _ = key
        Rb = ndb + npb
        if Tb > self.T_cap or Rb > self.R_cap:
            raise ValueError("step larger than the runner was sized for")
        W = self.W
        bt = np.asarray(step["block_tables"], dtype=np.int32).reshape(R, -1)
        if bt.shape[1] != W:
            raise ValueError("block_tables width differs from max_blocks_per_seq")
        b = self._turn
        self._turn ^= 1
        if self._copied[b] is not None:
            self._copied[b].synchronize()
        h = self._host[b].numpy()
        o_cu, o_sl, o_bt, o_sm = 0, Rb + 1, 2 * Rb + 1, 2 * Rb + 1 + Rb * W
        n = o_sm + Tb
        # rows: real decodes, decode padding, real prefills, prefill padding
        rows = list(range(nd)) + [-1] * (ndb - nd) + list(range(nd, R)) + [-1] * (npb - npf)
        cu_p = np.empty(Rb + 1, dtype=np.int32)
        sl_p = np.zeros(Rb, dtype=np.int32)
        bt_p = np.full((Rb, W), -1, dtype=np.int32)
        tok = 0
        for i, r in enumerate(rows):
            cu_p[i] = tok
            if r >= 0:
                tok = int(cu[r + 1])
                sl_p[i] = step["seq_lens"][r]
                bt_p[i] = bt[r]
        cu_p[Rb] = tok
        h[o_cu:o_cu + Rb + 1] = cu_p
        h[o_sl:o_sl + Rb] = sl_p
        h[o_bt:o_bt + Rb * W] = bt_p.reshape(-1)
        h[o_sm:o_sm + T] = step["slot_mapping"]
        h[o_sm + T:o_sm + Tb] = -1
        self._dev[:n].copy_(self._host[b][:n], non_blocking=True)
        ev = self.torch.cuda.Event()
        ev.record()
        self._copied[b] = ev
        return key, T

    def _launch(self, key):
        Tb, ndb, npb, mqb = key
        Rb = ndb + npb
        W = self.W
        d = self._dev
        cu, sl = d[0:Rb + 1], d[Rb + 1:2 * Rb + 1]
        bt = d[2 * Rb + 1:2 * Rb + 1 + Rb * W].view(Rb, W)
        sm = d[2 * Rb + 1 + Rb * W:2 * Rb + 1 + Rb * W + Tb]
        for layer in range(self.L):
            kc, vc = self.k_cache[layer], self.v_cache[layer]
            kv_append(self.k_buf[layer][:Tb], self.v_buf[layer][:Tb], sm, kc, vc)
            paged_attention(self.q_buf[layer][:Tb], kc, vc, cu, sl, bt, num_decodes=ndb,
                            max_q_len=max(mqb, 1), max_seq_len=W * self.block_size,
                            scale=self.scale, workspace=self.workspace,
                            out=self.out_buf[layer][:Tb])

    def run(self, key):
        """Run the step last prepared (key from prepare)."""
        torch = self.torch
        g = self.graphs.get(key)
        if g is not None:
            g.replay()
            return
        # first step of this bucket: run it uncaptured (this also does the
        # library's one-time set-up), then record the same launches; the
        # capture does not execute them, so the step runs once
        self._launch(key)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, pool=self.pool):
            self._launch(key)
        if self.pool is None:
            self.pool = g.pool()
        self.graphs[key] = g
