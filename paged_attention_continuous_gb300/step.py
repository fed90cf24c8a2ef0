"""One serving step through the C ABI: upload the scheduler's metadata, append
the step's new K/V into the paged cache, run paged attention.

"vLLM serving internals", What the scheduler looks like: each iteration
schedules a batch of prefill chunks and decode tokens and runs them in one
forward pass.  This module is the attention part of that pass for one or
more stacked layers: ``StepRunner.upload`` moves a step's host metadata
(``cu_seqlens_q``, ``seq_lens``, ``block_tables``, ``slot_mapping``) to the
device in ONE copy from pinned memory; ``StepRunner.run`` calls
``cb_kv_append`` then ``cb_paged_attention`` on the current stream.  With a
swap pool (``swap_blocks``) the scheduler's offload swaps are queued ahead
of each step (``SwapPool``).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

from . import SWAP_MAX_POOLS, Workspace, kv_append, kv_swap, paged_attention


class SwapPool:
    """Pinned host copies of offloaded requests' KV blocks.

    "Continuous batching architecture", Offloading: an offloaded request's
    blocks go to a preallocated pinned CPU pool and come back, without
    recomputation, when GPU blocks free up.  The pool holds ``swap_blocks``
    blocks per layer for K and for V, addressed by the scheduler's swap slot
    ids.  ``apply(step)`` queues on the current stream the step's swap-ins
    (slot -> cache block) and then its swap-outs (cache block -> slot), each
    as cb_kv_swap calls over every layer's K and V; it must run before the
    step's append and attention, and for every step the scheduler returns
    (a step that found no blocks still carries swap pairs).  The two
    directions are separate launches in that order because a slot a swap-in
    frees may be refilled by a swap-out of the same step.
    """

    def __init__(self, k_cache, v_cache, swap_blocks: int, device="cuda"):
        import torch
        self.torch = torch
        self.swap_blocks = int(swap_blocks)
        shape = (self.swap_blocks,) + tuple(k_cache[0].shape[1:])
        dt = k_cache[0].dtype
        self.k = [torch.zeros(shape, dtype=dt, pin_memory=True) for _ in k_cache]
        self.v = [torch.zeros(shape, dtype=dt, pin_memory=True) for _ in v_cache]
        self._cache = list(k_cache) + list(v_cache)
        self._pool = self.k + self.v
        self.block_bytes = k_cache[0][0].numel() * k_cache[0].element_size()
        cap = 4 * max(self.swap_blocks, 1)
        self._host = [torch.empty(cap, dtype=torch.int32, pin_memory=True) for _ in range(2)]
        self._copied = [None, None]
        self._turn = 0
        self._dev = torch.empty(cap, dtype=torch.int32, device=device)
        self.error_word = torch.zeros(1, dtype=torch.int32, device=device)

    def apply(self, step: dict) -> int:
        """Queue the step's swaps; returns the bytes moved over the CPU-GPU
        link (both directions)."""
        si = np.asarray(step.get("swap_in", np.zeros((0, 2))), dtype=np.int32).reshape(-1, 2)
        so = np.asarray(step.get("swap_out", np.zeros((0, 2))), dtype=np.int32).reshape(-1, 2)
        ni, no = len(si), len(so)
        if ni + no == 0:
            return 0
        if ni > self.swap_blocks or no > self.swap_blocks:
            raise ValueError("more swap pairs than swap slots")
        b = self._turn
        self._turn ^= 1
        if self._copied[b] is not None:
            self._copied[b].synchronize()
        h = self._host[b].numpy()
        h[0:ni] = si[:, 0]
        h[ni:2 * ni] = si[:, 1]
        h[2 * ni:2 * ni + no] = so[:, 0]
        h[2 * ni + no:2 * ni + 2 * no] = so[:, 1]
        n = 2 * (ni + no)
        self._dev[:n].copy_(self._host[b][:n], non_blocking=True)
        ev = self.torch.cuda.Event()
        ev.record()
        self._copied[b] = ev
        d = self._dev
        for lo in range(0, len(self._cache), SWAP_MAX_POOLS):
            hi = lo + SWAP_MAX_POOLS
            if ni:
                kv_swap(self._pool[lo:hi], self._cache[lo:hi], d[0:ni], d[ni:2 * ni],
                        error_word=self.error_word)
        for lo in range(0, len(self._cache), SWAP_MAX_POOLS):
            hi = lo + SWAP_MAX_POOLS
            if no:
                kv_swap(self._cache[lo:hi], self._pool[lo:hi], d[2 * ni:2 * ni + no],
                        d[2 * ni + no:n], error_word=self.error_word)
        return (ni + no) * len(self._cache) * self.block_bytes

    def read_errors(self) -> int:
        return int(self.error_word.item())


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
                 scale: Optional[float] = None, zero_cache: bool = True, swap_blocks: int = 0,
                 sliding_window: int = 0):
        import torch
        self.torch = torch
        self.dt = {"bf16": torch.bfloat16, "f32": torch.float32}[dtype]
        self.Hq, self.Hkv, self.D = num_q_heads, num_kv_heads, head_dim
        self.block_size = block_size
        self.num_blocks = num_blocks
        self.sliding_window = int(sliding_window)
        self.max_reqs, self.max_tokens = max_reqs, max_tokens
        self.W = max_blocks_per_seq
        self.scale = 1.0 / math.sqrt(head_dim) if scale is None else scale
        alloc = torch.zeros if zero_cache else torch.empty
        shape = (num_blocks, num_kv_heads, block_size, head_dim)
        self.k_cache = [alloc(shape, dtype=self.dt, device=device) for _ in range(num_layers)]
        self.v_cache = [alloc(shape, dtype=self.dt, device=device) for _ in range(num_layers)]
        self.workspace = Workspace(max_reqs, num_q_heads, num_kv_heads, head_dim, device=device)
        self.swap = SwapPool(self.k_cache, self.v_cache, swap_blocks, device) if swap_blocks else None
        cap = (max_reqs + 1) + max_reqs + max_reqs * max_blocks_per_seq + max_tokens
        # two pinned staging buffers, used in turn: a buffer is refilled only
        # after the copy that last read it has executed (its event), since
        # the host may run steps ahead of the device
        self._host = [torch.empty(cap, dtype=torch.int32, pin_memory=True) for _ in range(2)]
        self._copied = [None, None]
        self._turn = 0
        self._dev = torch.empty(cap, dtype=torch.int32, device=device)

    def apply_swaps(self, step: dict) -> int:
        """Queue the step's swap-ins and swap-outs (``SwapPool.apply``).
        ``upload`` calls it; call it directly for a step that found no
        blocks (it is not uploaded but may carry swap pairs)."""
        if self.swap is None:
            if len(step.get("swap_in", ())) or len(step.get("swap_out", ())):
                raise ValueError("step carries swaps but the runner has no swap pool")
            return 0
        return self.swap.apply(step)

    def _pack(self, step: dict, h: np.ndarray):
        """Write the step's metadata into the host int32 buffer ``h`` (one
        packed run: cu_seqlens_q, seq_lens, block_tables, slot_mapping);
        returns (words, offsets)."""
        R, T = int(step["num_reqs"]), int(step["num_tokens"])
        if R > self.max_reqs or T > self.max_tokens:
            raise ValueError("step larger than the runner was sized for")
        W = self.W
        bt = np.asarray(step["block_tables"], dtype=np.int32).reshape(R, -1 if R else W)
        if bt.shape[1] != W:
            raise ValueError("block_tables width differs from max_blocks_per_seq")
        o1 = R + 1
        o2 = o1 + R
        o3 = o2 + R * W
        h[0:o1] = step["cu_seqlens_q"]
        h[o1:o2] = step["seq_lens"]
        h[o2:o3] = bt.reshape(-1)
        h[o3:o3 + T] = step["slot_mapping"]
        return o3 + T, (o1, o2, o3)

    def _device_step(self, step: dict, d, n: int, offs) -> DeviceStep:
        R, T, W = int(step["num_reqs"]), int(step["num_tokens"]), self.W
        o1, o2, o3 = offs
        return DeviceStep(R, T, int(step["num_decodes"]), int(step["max_q_len"]) if "max_q_len" in step
                          else int(np.diff(step["cu_seqlens_q"]).max(initial=1)),
                          int(step["max_seq_len"]) if "max_seq_len" in step
                          else int(np.max(step["seq_lens"], initial=1)),
                          d[0:R + 1], d[o1:o2], d[o2:o3].view(R, W), d[o3:o3 + T], 4 * n)

    def upload(self, step: dict, stream=None) -> DeviceStep:
        """Queue the step's swaps, then copy its metadata to the device (one
        pinned copy on the current stream).  The returned arrays stay valid
        until the next upload on this runner; kernels that use them must be
        queued on the same stream before that next upload."""
        self.apply_swaps(step)
        b = self._turn
        self._turn ^= 1
        if self._copied[b] is not None:
            self._copied[b].synchronize()
        n, offs = self._pack(step, self._host[b].numpy())
        self._dev[:n].copy_(self._host[b][:n], non_blocking=True)
        ev = self.torch.cuda.Event()
        ev.record()
        self._copied[b] = ev
        return self._device_step(step, self._dev, n, offs)

    def run(self, ds: DeviceStep, q, k_new, v_new, layer: int = 0, out=None):
        """Append this step's K/V for ``layer`` and attend.  q [T, Hq, D],
        k_new/v_new [T, Hkv, D] on the device.  Returns out [T, Hq, D]."""
        kc, vc = self.k_cache[layer], self.v_cache[layer]
        kv_append(k_new, v_new, ds.slot_mapping, kc, vc)
        return paged_attention(q, kc, vc, ds.cu_seqlens_q, ds.seq_lens, ds.block_tables,
                               num_decodes=ds.num_decodes, max_q_len=ds.max_q_len,
                               max_seq_len=ds.max_seq_len, scale=self.scale,
                               workspace=self.workspace, out=out,
                               sliding_window=self.sliding_window, after_append=True)


class PipelinedStepRunner(StepRunner):
    """Async double-buffered batching ("Continuous batching architecture",
    Async batching): two sets of input/output buffers and separate streams
    for input copies, compute and output copies, so that while the device
    computes step N, step N+1's inputs are copied in and step N-1's output is
    copied out, and the host is free to schedule.

    ``submit(step, q, k, v, out)`` takes the step's inputs in pinned host
    memory -- per layer lists of q [T, Hq, D] and k/v [T, Hkv, D] (a single
    tensor for one layer) -- and a pinned host ``out`` (per layer list, or
    one tensor) that receives the attention output; it returns an event that
    completes once ``out`` holds the result.  The caller leaves the input
    tensors unchanged, and reads ``out`` only, after that event.  Steps use
    the two buffer sets in turn: a set's inputs are refilled only after the
    compute that read them (two steps back) finished, its output buffer is
    rewritten only after the copy-out that read it, and its host staging
    buffer only after the copy-in that read it.  Caches, workspace and swap
    pool are the StepRunner's; swaps run on the compute stream ahead of the
    step's kernels.  ``upload``/``run`` (current stream) may be used on the
    same runner only with the device synchronised in between.
    """

    def __init__(self, **kw):
        super().__init__(**kw)
        torch = self.torch
        dev = self.k_cache[0].device
        L = len(self.k_cache)
        T = self.max_tokens
        mk = lambda h: [torch.empty(T, h, self.D, dtype=self.dt, device=dev) for _ in range(L)]
        words = self._dev.shape[0]
        self._sets = [dict(q=mk(self.Hq), k=mk(self.Hkv), v=mk(self.Hkv), out=mk(self.Hq),
                           meta=torch.empty(words, dtype=torch.int32, device=dev),
                           stage=torch.empty(words, dtype=torch.int32, pin_memory=True))
                      for _ in range(2)]
        self.in_stream = torch.cuda.Stream(device=dev)
        self.compute_stream = torch.cuda.Stream(device=dev)
        self.out_stream = torch.cuda.Stream(device=dev)
        self._copied_in = [None, None]   # per set: copy-in finished
        self._computed = [None, None]    # per set: compute finished
        self._copied_out = [None, None]  # per set: copy-out finished
        self._slot = 0

    def submit(self, step: dict, q, k, v, out):
        torch = self.torch
        as_list = lambda x: list(x) if isinstance(x, (list, tuple)) else [x]
        q, k, v, out = as_list(q), as_list(k), as_list(v), as_list(out)
        L = len(self.k_cache)
        if not (len(q) == len(k) == len(v) == len(out) == L):
            raise ValueError("one q/k/v/out tensor per layer expected")
        T = int(step["num_tokens"])
        i = self._slot
        self._slot ^= 1
        st = self._sets[i]
        if self._copied_in[i] is not None:
            self._copied_in[i].synchronize()    # the set's host staging is free
        n, offs = self._pack(step, st["stage"].numpy())
        ins, ks, outs = self.in_stream, self.compute_stream, self.out_stream
        with torch.cuda.stream(ins):
            if self._computed[i] is not None:
                ins.wait_event(self._computed[i])
            st["meta"][:n].copy_(st["stage"][:n], non_blocking=True)
            for layer in range(L):
                st["q"][layer][:T].copy_(q[layer], non_blocking=True)
                st["k"][layer][:T].copy_(k[layer], non_blocking=True)
                st["v"][layer][:T].copy_(v[layer], non_blocking=True)
            copied_in = torch.cuda.Event()
            copied_in.record(ins)
        self._copied_in[i] = copied_in
        ds = self._device_step(step, st["meta"], n, offs)
        with torch.cuda.stream(ks):
            ks.wait_event(copied_in)
            if self._copied_out[i] is not None:
                ks.wait_event(self._copied_out[i])
            self.apply_swaps(step)
            for layer in range(L):
                self.run(ds, st["q"][layer][:T], st["k"][layer][:T], st["v"][layer][:T],
                         layer=layer, out=st["out"][layer][:T])
            computed = torch.cuda.Event()
            computed.record(ks)
        self._computed[i] = computed
        with torch.cuda.stream(outs):
            outs.wait_event(computed)
            for layer in range(L):
                out[layer].copy_(st["out"][layer][:T], non_blocking=True)
            copied_out = torch.cuda.Event()
            copied_out.record(outs)
        self._copied_out[i] = copied_out
        return copied_out

    def synchronize(self):
        for s_ in (self.in_stream, self.compute_stream, self.out_stream):
            s_.synchronize()


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
                 scale: Optional[float] = None, zero_cache: bool = True, swap_blocks: int = 0,
                 sliding_window: int = 0):
        import torch
        self.torch = torch
        self.dt = {"bf16": torch.bfloat16, "f32": torch.float32}[dtype]
        self.Hq, self.Hkv, self.D = num_q_heads, num_kv_heads, head_dim
        self.block_size = block_size
        self.W = max_blocks_per_seq
        self.sliding_window = int(sliding_window)
        self.L = num_layers
        self.scale = 1.0 / math.sqrt(head_dim) if scale is None else scale
        self.R_cap = 2 * bucket(max_reqs)     # padded decode rows + padded prefill rows
        self.T_cap = bucket(max_tokens, 16)
        alloc = torch.zeros if zero_cache else torch.empty
        shape = (num_blocks, num_kv_heads, block_size, head_dim)
        self.k_cache = [alloc(shape, dtype=self.dt, device=device) for _ in range(num_layers)]
        self.v_cache = [alloc(shape, dtype=self.dt, device=device) for _ in range(num_layers)]
        self.workspace = Workspace(self.R_cap, num_q_heads, num_kv_heads, head_dim, device=device)
        self.swap = SwapPool(self.k_cache, self.v_cache, swap_blocks, device) if swap_blocks else None
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

    apply_swaps = StepRunner.apply_swaps

    def prepare(self, step: dict):
        """Queue the step's swaps (uncaptured launches, ahead of the graph),
        pad the step to its bucket and upload it; returns (key, T)."""
        self.apply_swaps(step)
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
        bt = np.asarray(step["block_tables"], dtype=np.int32).reshape(R, -1 if R else W)
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
            # a chunk's bucket may pass the longest sequence the table spans;
            # no real chunk does
            paged_attention(self.q_buf[layer][:Tb], kc, vc, cu, sl, bt, num_decodes=ndb,
                            max_q_len=min(max(mqb, 1), W * self.block_size),
                            max_seq_len=W * self.block_size,
                            scale=self.scale, workspace=self.workspace,
                            out=self.out_buf[layer][:Tb], sliding_window=self.sliding_window)

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
