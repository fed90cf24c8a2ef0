"""Oracle paged KV append (TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__``).

*vLLM serving internals*, "PagedAttention as a virtual memory system": the
cache is a pool of fixed-size blocks of 16 token positions; a sequence's
block table maps its logical token positions to physical blocks.  A token's
slot is ``physical_block * block_size + offset_in_block``; slot -1 marks a
padding token that is not written.

Cache layout (the pages leave it open): ``[num_blocks, num_kv_heads,
block_size, head_dim]``, so the slot's (block, offset) picks one row per KV
head.

Parity: exact copy semantics, pinned in tests by a brute-force slot walk and
by the paging-invariance property (permuted physical blocks give identical
attention output).
"""
from __future__ import annotations

import numpy as np


def append(k_cache: np.ndarray, v_cache: np.ndarray, k_new: np.ndarray,
           v_new: np.ndarray, slot_mapping: np.ndarray, block_size: int) -> None:
    """In place: for each token t with slot s >= 0, write k_new[t] / v_new[t]
    (shape [num_kv_heads, head_dim]) at block s // bs, offset s % bs."""
    for t in range(len(slot_mapping)):
        s = int(slot_mapping[t])
        if s < 0:
            continue
        b, off = divmod(s, block_size)
        k_cache[b, :, off, :] = k_new[t]
        v_cache[b, :, off, :] = v_new[t]
