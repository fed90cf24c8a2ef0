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
