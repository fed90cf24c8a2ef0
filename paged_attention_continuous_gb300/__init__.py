"""GB300 continuous-batching paged attention: Python binding of ``libcb.so``.

A thin ctypes layer over the C ABI declared in ``include/cb.h``; it only
marshals arguments.  Every step of the path runs in the library: the host
FIFO scheduler (``Scheduler``, backed by ``cb_schedule_step``), the paged KV
append (``kv_append`` -> ``cb_kv_append``) and the paged attention
(``paged_attention`` -> ``cb_paged_attention``).  PyTorch is used for device
memory and streams only.  There is no CPU fallback: importing this package
fails if the library has not been built
(``python paged_attention_continuous_gb300/build.py``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

from ._lib_loader import LIB_PATH, load_library

_lib = load_library()

CB_OK = 0
CB_ERR_INVALID_ARG = 1
CB_ERR_NO_BLOCKS = 2
CB_ERR_CUDA = 3
CB_ERR_UNSUPPORTED = 4
CB_ERR_DEVICE_CHECK = 5
CB_ERR_STATE = 6

DTYPE_F32 = 0
DTYPE_BF16 = 1

DEVERR_BLOCK_RANGE = 0x1
DEVERR_SLOT_RANGE = 0x2
DEVERR_DECODE_QLEN = 0x4
DEVERR_SEQ_RANGE = 0x8
DEVERR_TIMEOUT = 0x10
DEVERR_PLAN = 0x20


class CBError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"cb status {status}: {message}")
        self.status = status


def _check(st: int) -> int:
    if st != CB_OK:
        raise CBError(st, _lib.cb_last_error().decode())
    return st


class cb_config(ctypes.Structure):
    _fields_ = [("block_size", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("max_batch_tokens", ctypes.c_int32),
                ("max_requests_per_batch", ctypes.c_int32),
                ("max_prefill_chunk", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32),
                ("safety_margin", ctypes.c_float),
                ("initial_free_list", ctypes.POINTER(ctypes.c_int32)),
                ("policy", ctypes.c_int32), ("max_prefill_reqs", ctypes.c_int32),
                ("long_prefill_tokens", ctypes.c_int32), ("max_long_prefills", ctypes.c_int32),
                ("offload", ctypes.c_int32), ("swap_blocks", ctypes.c_int32),
                ("prefix_caching", ctypes.c_int32), ("sliding_window", ctypes.c_int32)]


class cb_step(ctypes.Structure):
    _fields_ = [("num_reqs", ctypes.c_int32), ("num_tokens", ctypes.c_int32),
                ("num_decodes", ctypes.c_int32), ("max_q_len", ctypes.c_int32),
                ("max_seq_len", ctypes.c_int32), ("max_blocks_per_seq", ctypes.c_int32),
                ("req_ids", ctypes.POINTER(ctypes.c_int64)),
                ("cu_seqlens_q", ctypes.POINTER(ctypes.c_int32)),
                ("seq_lens", ctypes.POINTER(ctypes.c_int32)),
                ("block_tables", ctypes.POINTER(ctypes.c_int32)),
                ("slot_mapping", ctypes.POINTER(ctypes.c_int32)),
                ("num_stalled", ctypes.c_int32),
                ("stalled_ids", ctypes.POINTER(ctypes.c_int64)),
                ("stalled_demand", ctypes.POINTER(ctypes.c_int32)),
                ("num_swap_in", ctypes.c_int32),
                ("swap_in_slots", ctypes.POINTER(ctypes.c_int32)),
                ("swap_in_blocks", ctypes.POINTER(ctypes.c_int32)),
                ("num_swap_out", ctypes.c_int32),
                ("swap_out_blocks", ctypes.POINTER(ctypes.c_int32)),
                ("swap_out_slots", ctypes.POINTER(ctypes.c_int32))]


class cb_attention_args(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("out", ctypes.c_void_p),
                ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("cu_seqlens_q", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
                ("block_tables", ctypes.c_void_p),
                ("num_reqs", ctypes.c_int32), ("num_decodes", ctypes.c_int32),
                ("num_tokens", ctypes.c_int32), ("max_q_len", ctypes.c_int32),
                ("max_seq_len", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("scale", ctypes.c_float),
                ("dtype", ctypes.c_int32), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("sliding_window", ctypes.c_int32),
                ("after_append", ctypes.c_int32)]


class cb_executor_config(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("k_caches", ctypes.POINTER(ctypes.c_void_p)),
                ("v_caches", ctypes.POINTER(ctypes.c_void_p)), ("num_blocks", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("scale", ctypes.c_float),
                ("sliding_window", ctypes.c_int32), ("max_reqs", ctypes.c_int32),
                ("max_tokens", ctypes.c_int32), ("max_blocks_per_seq", ctypes.c_int32)]


SWAP_MAX_POOLS = 128


class cb_swap_args(ctypes.Structure):
    _fields_ = [("num_pairs", ctypes.c_int32), ("src_ids", ctypes.c_void_p),
                ("dst_ids", ctypes.c_void_p), ("num_pools", ctypes.c_int32),
                ("src_pools", ctypes.POINTER(ctypes.c_void_p)),
                ("dst_pools", ctypes.POINTER(ctypes.c_void_p)),
                ("src_capacity", ctypes.c_int64), ("dst_capacity", ctypes.c_int64),
                ("block_bytes", ctypes.c_int64), ("error_word", ctypes.c_void_p)]


def _declare():
    L = _lib
    P = ctypes.POINTER
    i32, i64, vp, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
    L.cb_last_error.restype = ctypes.c_char_p
    L.cb_version.restype = i32
    L.cb_sched_create.argtypes = [P(cb_config), P(vp)]
    L.cb_sched_destroy.argtypes = [vp]
    L.cb_sched_destroy.restype = None
    L.cb_add_request.argtypes = [vp, i64, i32, i32]
    L.cb_add_request_tokens.argtypes = [vp, i64, i32, i32, P(i32), i32]
    L.cb_sched_prefix_stats.argtypes = [vp, P(i64), P(i32), P(i32)]
    L.cb_sched_hold_blocks.argtypes = [vp, i32, P(i32), P(i32)]
    L.cb_sched_release_blocks.argtypes = [vp, P(i32), i32]
    L.cb_add_running_request.argtypes = [vp, i64, i32, i32, i32]
    L.cb_schedule_step.argtypes = [vp, P(cb_step)]
    L.cb_step_done.argtypes = [vp, P(i32), P(P(i64))]
    L.cb_request_slots.argtypes = [vp, i64, i32, i32, P(i32)]
    L.cb_sched_counts.argtypes = [vp, P(i32), P(i32), P(i32)]
    L.cb_sched_free_list.argtypes = [vp, P(i32), i32, P(i32)]
    L.cb_sched_swapped.argtypes = [vp, P(ctypes.c_int64), i32, P(i32), P(i32)]
    L.cb_kv_append.argtypes = [vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, vp, vp]
    L.cb_kv_swap.argtypes = [P(cb_swap_args), vp]
    L.cb_validate_step.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32]
    L.cb_attention_workspace_size.argtypes = [i32, i32, i32, i32]
    L.cb_attention_workspace_size.restype = sz
    L.cb_attention_workspace_init.argtypes = [vp, sz, vp]
    L.cb_paged_attention.argtypes = [P(cb_attention_args), vp]
    L.cb_attention_read_errors.argtypes = [vp, sz, vp, P(ctypes.c_uint32)]
    L.cb_debug_inject_wait_timeout.argtypes = [ctypes.c_uint64, i32, i32]
    PV = P(vp)
    L.cb_executor_create.argtypes = [P(cb_executor_config), P(vp)]
    L.cb_executor_destroy.argtypes = [vp]
    L.cb_executor_destroy.restype = None
    L.cb_executor_submit.argtypes = [vp, P(cb_step), PV, PV, PV, PV]
    L.cb_executor_run_step.argtypes = [vp, vp, PV, PV, PV, PV, P(i32), P(i32)]
    L.cb_executor_synchronize.argtypes = [vp]
    L.cb_executor_stats.argtypes = [vp, P(i64), P(i64), P(ctypes.c_double)]
    L.cb_executor_reset_stats.argtypes = [vp]
    L.cb_executor_read_errors.argtypes = [vp, P(ctypes.c_uint32)]
    for name in ("cb_sched_create", "cb_add_request", "cb_add_request_tokens",
                 "cb_sched_prefix_stats", "cb_sched_hold_blocks", "cb_sched_release_blocks",
                 "cb_add_running_request",
                 "cb_schedule_step", "cb_step_done", "cb_request_slots", "cb_sched_counts",
                 "cb_sched_free_list", "cb_sched_swapped", "cb_kv_append", "cb_kv_swap",
                 "cb_validate_step",
                 "cb_attention_workspace_init",
                 "cb_paged_attention", "cb_attention_read_errors",
                 "cb_debug_inject_wait_timeout", "cb_executor_create", "cb_executor_submit",
                 "cb_executor_run_step", "cb_executor_synchronize", "cb_executor_stats",
                 "cb_executor_reset_stats", "cb_executor_read_errors"):
        getattr(L, name).restype = ctypes.c_int


_declare()


def version() -> int:
    return int(_lib.cb_version())


def library():
    """The loaded ctypes handle of libcb.so."""
    return _lib


# --------------------------------------------------------------- scheduler
def _arr(ptr, n, dtype):
    """A numpy copy of n elements of `dtype` (the C element type) at ptr:
    one memmove into a fresh array (cheaper per call than building a ctypes
    array view)."""
    out = np.empty(n, dtype=dtype)
    if n:
        ctypes.memmove(out.__array_interface__["data"][0], ptr, n * out.itemsize)
    return out


def _pairs(a_ptr, b_ptr, n):
    """[n, 2] int32 of two C int32 arrays side by side."""
    if n == 0:
        return np.zeros((0, 2), dtype=np.int32)
    return np.stack([_arr(a_ptr, n, np.int32), _arr(b_ptr, n, np.int32)], axis=1)


POLICY_FIFO, POLICY_PREFILL_FIRST = 0, 1


class Scheduler:
    """Continuous-batching scheduler (C++), see ``cb_schedule_step``:
    policy FIFO (default) or PREFILL_FIRST, optional prefill-row and
    long-prefill caps, offloading, prefix caching, sliding-window page
    recycling."""

    def __init__(self, *, block_size: int, num_blocks: int, max_batch_tokens: int,
                 max_requests_per_batch: int, max_blocks_per_seq: int,
                 max_prefill_chunk: int = 0, safety_margin: float = 0.15,
                 free_list: Optional[Sequence[int]] = None, policy: int = POLICY_FIFO,
                 max_prefill_reqs: int = 0, long_prefill_tokens: int = 0,
                 max_long_prefills: int = 1, offload: bool = False, swap_blocks: int = 0,
                 prefix_caching: bool = False, sliding_window: int = 0):
        self.max_blocks_per_seq = int(max_blocks_per_seq)
        cfg = cb_config(block_size, num_blocks, max_batch_tokens, max_requests_per_batch,
                        max_prefill_chunk, max_blocks_per_seq, float(safety_margin), None,
                        int(policy), int(max_prefill_reqs), int(long_prefill_tokens),
                        int(max_long_prefills), int(bool(offload)), int(swap_blocks),
                        int(bool(prefix_caching)), int(sliding_window))
        keep = None
        if free_list is not None:
            keep = np.ascontiguousarray(np.asarray(free_list, dtype=np.int32))
            if keep.shape != (num_blocks,):
                raise ValueError("free_list must hold num_blocks ids")
            cfg.initial_free_list = keep.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        h = ctypes.c_void_p()
        _check(_lib.cb_sched_create(ctypes.byref(cfg), ctypes.byref(h)))
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            _lib.cb_sched_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def add_request(self, req_id: int, prompt_len: int, output_len: int,
                    tokens: Optional[Sequence[int]] = None) -> None:
        """``tokens``: ids of the first len(tokens) prompt tokens, for prefix
        caching (``cb_add_request_tokens``)."""
        if tokens is None:
            _check(_lib.cb_add_request(self._h, req_id, prompt_len, output_len))
            return
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32).reshape(-1))
        _check(_lib.cb_add_request_tokens(self._h, req_id, prompt_len, output_len,
                                          t.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                          int(t.shape[0])))

    def hold_blocks(self, n: int) -> list:
        """Fault injection: take up to n blocks out of the allocatable pool
        (``cb_sched_hold_blocks``); returns their ids."""
        out = np.zeros(max(int(n), 1), dtype=np.int32)
        k = ctypes.c_int32()
        _check(_lib.cb_sched_hold_blocks(self._h, int(n),
                                         out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                         ctypes.byref(k)))
        return out[:k.value].tolist()

    def release_blocks(self, ids) -> None:
        """Return held blocks to the free queue's tail, in order."""
        a = np.ascontiguousarray(np.asarray(list(ids), dtype=np.int32))
        _check(_lib.cb_sched_release_blocks(self._h, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                            int(a.shape[0])))

    def prefix_stats(self):
        """(prompt tokens reused so far, keyed blocks, keyed blocks in the
        initialized pool)."""
        h, k, p = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
        _check(_lib.cb_sched_prefix_stats(self._h, ctypes.byref(h), ctypes.byref(k),
                                          ctypes.byref(p)))
        return h.value, k.value, p.value

    def add_running_request(self, req_id: int, prompt_len: int, output_len: int,
                            num_cached: int) -> None:
        _check(_lib.cb_add_running_request(self._h, req_id, prompt_len, output_len, num_cached))

    def schedule_step(self) -> dict:
        """Returns the step as numpy arrays (copies) plus 'status'
        (0 = OK, 2 = NO_BLOCKS); other statuses raise CBError."""
        s = cb_step()
        st = _lib.cb_schedule_step(self._h, ctypes.byref(s))
        if st not in (CB_OK, CB_ERR_NO_BLOCKS):
            _check(st)
        R, T, W = s.num_reqs, s.num_tokens, s.max_blocks_per_seq
        return {
            "status": int(st), "num_reqs": R, "num_tokens": T, "num_decodes": s.num_decodes,
            "max_q_len": s.max_q_len, "max_seq_len": s.max_seq_len,
            "req_ids": _arr(s.req_ids, R, np.int64),
            "cu_seqlens_q": _arr(s.cu_seqlens_q, R + 1, np.int32),
            "seq_lens": _arr(s.seq_lens, R, np.int32),
            "block_tables": _arr(s.block_tables, R * W, np.int32).reshape(R, W),
            "slot_mapping": _arr(s.slot_mapping, T, np.int32),
            "stalled_ids": _arr(s.stalled_ids, s.num_stalled, np.int64),
            "stalled_demand": _arr(s.stalled_demand, s.num_stalled, np.int32),
            "swap_in": _pairs(s.swap_in_slots, s.swap_in_blocks, s.num_swap_in),
            "swap_out": _pairs(s.swap_out_blocks, s.swap_out_slots, s.num_swap_out),
        }

    def swapped(self):
        """(ids of requests in the swap pool in offload order, free slots)."""
        n, f = ctypes.c_int32(), ctypes.c_int32()
        _check(_lib.cb_sched_swapped(self._h, None, 0, ctypes.byref(n), ctypes.byref(f)))
        out = np.zeros(max(n.value, 1), dtype=np.int64)
        _check(_lib.cb_sched_swapped(self._h, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                     n.value, ctypes.byref(n), ctypes.byref(f)))
        return [int(x) for x in out[:n.value]], f.value

    def step_done(self) -> list:
        n = ctypes.c_int32()
        ids = ctypes.POINTER(ctypes.c_int64)()
        _check(_lib.cb_step_done(self._h, ctypes.byref(n), ctypes.byref(ids)))
        return [int(x) for x in _arr(ids, n.value, np.int64)]

    def slots(self, req_id: int, start: int, count: int) -> np.ndarray:
        out = np.zeros(count, dtype=np.int32)
        _check(_lib.cb_request_slots(self._h, req_id, start, count,
                                     out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))))
        return out

    def counts(self):
        f, w, r = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        _check(_lib.cb_sched_counts(self._h, ctypes.byref(f), ctypes.byref(w), ctypes.byref(r)))
        return f.value, w.value, r.value

    @property
    def free(self) -> list:
        n = ctypes.c_int32()
        _check(_lib.cb_sched_free_list(self._h, None, 0, ctypes.byref(n)))
        out = np.zeros(max(n.value, 1), dtype=np.int32)
        _check(_lib.cb_sched_free_list(self._h, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                       n.value, ctypes.byref(n)))
        return out[:n.value].tolist()


# ------------------------------------------------------------------ GPU ops
def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float32:
        return DTYPE_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream_ptr(stream) -> int:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if not t.is_cuda:
            raise ValueError("tensors must live on the GPU (no CPU path)")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def kv_append(k_new, v_new, slot_mapping, k_cache, v_cache, *, error_word=None,
              stream=None) -> None:
    """cb_kv_append: k_new/v_new [T, Hkv, D]; slot_mapping int32 [T];
    caches [num_blocks, Hkv, block_size, D]."""
    _need_cuda(k_new, v_new, slot_mapping, k_cache, v_cache)
    T = slot_mapping.shape[0]
    nb, hkv, bs, d = k_cache.shape
    ew = error_word.data_ptr() if error_word is not None else None
    _check(_lib.cb_kv_append(k_new.data_ptr(), v_new.data_ptr(), slot_mapping.data_ptr(), T,
                             k_cache.data_ptr(), v_cache.data_ptr(), nb, hkv, d, bs,
                             _dtype_code(k_cache), ew, _stream_ptr(stream)))


def kv_swap(src_pools, dst_pools, src_ids, dst_ids, *, error_word=None, stream=None) -> None:
    """cb_kv_swap: for every pair i and pool k, block ``src_ids[i]`` of
    ``src_pools[k]`` is copied to block ``dst_ids[i]`` of ``dst_pools[k]``.
    Pools are contiguous tensors [capacity, ...] of one block shape, each on
    the GPU or in pinned host memory; ids are int32 device tensors."""
    if len(src_pools) != len(dst_pools):
        raise ValueError("src_pools and dst_pools differ in length")
    if len(src_pools) > SWAP_MAX_POOLS:
        raise ValueError(f"at most {SWAP_MAX_POOLS} pools per call")
    _need_cuda(src_ids, dst_ids)
    n = int(src_ids.shape[0])
    if int(dst_ids.shape[0]) != n:
        raise ValueError("src_ids and dst_ids differ in length")
    if n == 0 or not src_pools:
        return
    torch = _torch()
    if src_ids.dtype != torch.int32 or dst_ids.dtype != torch.int32:
        raise TypeError("ids must be int32")
    blk = src_pools[0][0].numel() * src_pools[0].element_size()
    for t in list(src_pools) + list(dst_pools):
        if not t.is_contiguous():
            raise ValueError("pools must be contiguous")
        if not (t.is_cuda or t.is_pinned()):
            raise ValueError("pools must live on the GPU or in pinned host memory")
        if t[0].numel() * t.element_size() != blk:
            raise ValueError("pools differ in block size")
    for grp in (src_pools, dst_pools):
        if len({int(t.shape[0]) for t in grp}) != 1:
            raise ValueError("pools on one side differ in capacity")
    P = ctypes.c_void_p * len(src_pools)
    sp = P(*[t.data_ptr() for t in src_pools])
    dp = P(*[t.data_ptr() for t in dst_pools])
    a = cb_swap_args(n, src_ids.data_ptr(), dst_ids.data_ptr(), len(src_pools),
                     ctypes.cast(sp, ctypes.POINTER(ctypes.c_void_p)),
                     ctypes.cast(dp, ctypes.POINTER(ctypes.c_void_p)),
                     int(src_pools[0].shape[0]), int(dst_pools[0].shape[0]), blk,
                     error_word.data_ptr() if error_word is not None else None)
    _check(_lib.cb_kv_swap(ctypes.byref(a), _stream_ptr(stream)))


def validate_step(step: dict, *, num_blocks: int, block_size: int = 16,
                  sliding_window: int = 0) -> None:
    """cb_validate_step on a scheduler step's host arrays (numpy); raises
    CBError naming the first broken rule."""
    R = int(step["num_reqs"])
    keep = [np.ascontiguousarray(np.asarray(step[k], dtype=np.int32).reshape(-1))
            for k in ("cu_seqlens_q", "seq_lens", "block_tables")]
    bt = np.asarray(step["block_tables"]).reshape(R, -1) if R else np.zeros((0, 1))
    W = int(bt.shape[1]) if R else int(step.get("max_blocks_per_seq", 1) or 1)
    sm = step.get("slot_mapping")
    sm = None if sm is None else np.ascontiguousarray(np.asarray(sm, dtype=np.int32))
    T = int(step["num_tokens"])
    _check(_lib.cb_validate_step(keep[0].ctypes.data, keep[1].ctypes.data, keep[2].ctypes.data,
                                 None if sm is None else sm.ctypes.data, R,
                                 int(step["num_decodes"]), T, W, int(num_blocks),
                                 int(block_size), int(sliding_window)))


def workspace_size(num_reqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int) -> int:
    return int(_lib.cb_attention_workspace_size(num_reqs, num_q_heads, num_kv_heads, head_dim))


class Workspace:
    """Device scratch for cb_paged_attention (zeroed once on creation)."""

    def __init__(self, max_reqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                 device="cuda", stream=None):
        torch = _torch()
        self.nbytes = workspace_size(max_reqs, num_q_heads, num_kv_heads, head_dim)
        self.max_reqs = max_reqs
        self.buf = torch.empty(self.nbytes + 256, dtype=torch.uint8, device=device)
        off = (-self.buf.data_ptr()) % 256
        self.ptr = self.buf.data_ptr() + off
        _check(_lib.cb_attention_workspace_init(self.ptr, self.nbytes, _stream_ptr(stream)))

    def read_errors(self, stream=None) -> int:
        bits = ctypes.c_uint32()
        st = _lib.cb_attention_read_errors(self.ptr, self.nbytes, _stream_ptr(stream),
                                           ctypes.byref(bits))
        if st not in (CB_OK, CB_ERR_DEVICE_CHECK):
            _check(st)
        return int(bits.value)

    def reinit(self, stream=None):
        _check(_lib.cb_attention_workspace_init(self.ptr, self.nbytes, _stream_ptr(stream)))


def paged_attention(q, k_cache, v_cache, cu_seqlens_q, seq_lens, block_tables, *,
                    num_decodes: int, max_q_len: int, max_seq_len: int, scale: float,
                    workspace: Workspace, out=None, stream=None, sliding_window: int = 0,
                    after_append: bool = False):
    """cb_paged_attention.  q [T, Hq, D]; caches [num_blocks, Hkv, bs, D];
    metadata int32 device tensors; ``sliding_window`` > 0 for a
    sliding-window layer; ``after_append``: the launch just before on the
    stream was this step's kv_append (the decode kernel then overlaps its
    end).  Returns out [T, Hq, D]."""
    torch = _torch()
    _need_cuda(q, k_cache, v_cache, cu_seqlens_q, seq_lens, block_tables)
    if out is None:
        out = torch.empty_like(q)
    T, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    R = seq_lens.shape[0]
    if R > workspace.max_reqs:
        raise ValueError("workspace sized for fewer requests")
    a = cb_attention_args(q.data_ptr(), out.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                          cu_seqlens_q.data_ptr(), seq_lens.data_ptr(), block_tables.data_ptr(),
                          R, num_decodes, T, max_q_len, max_seq_len, nb, block_tables.shape[1],
                          bs, hq, hkv, d, float(scale), _dtype_code(q), workspace.ptr,
                          workspace.nbytes, int(sliding_window), int(bool(after_append)))
    _check(_lib.cb_paged_attention(ctypes.byref(a), _stream_ptr(stream)))
    return out


def inject_wait_timeout(wait_ns: int = 0, decode_item: int = -1, prefill_tile: int = -1) -> None:
    """cb_debug_inject_wait_timeout (test hook): shorten every bounded device
    wait of later launches to ``wait_ns`` (0 restores 1 s) and withhold the
    copies of one decode work item / one prefill K tile (-1: none)."""
    _check(_lib.cb_debug_inject_wait_timeout(int(wait_ns), int(decode_item), int(prefill_tile)))


def _ptrs(ts):
    ts = list(ts) if isinstance(ts, (list, tuple)) else [ts]
    return (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts]), ts


class Executor:
    """cb_executor: a whole serving step behind one C call, double-buffered
    over copy-in / compute / copy-out streams.  ``k_caches``/``v_caches``:
    per layer device tensors [num_blocks, Hkv, 16, D] (the caller keeps
    them).  ``run_step(sched, q, k, v, out)`` schedules the next step of a
    ``Scheduler``, queues its copies and kernels and commits it; q/k/v/out
    are per layer pinned host tensors with at least the step's T rows (one
    tensor for a single layer).  Results are in ``out`` after
    ``synchronize()``."""

    def __init__(self, k_caches, v_caches, *, num_q_heads: int, max_reqs: int, max_tokens: int,
                 max_blocks_per_seq: int, scale: float, sliding_window: int = 0):
        kc = list(k_caches) if isinstance(k_caches, (list, tuple)) else [k_caches]
        vc = list(v_caches) if isinstance(v_caches, (list, tuple)) else [v_caches]
        _need_cuda(*kc, *vc)
        nb, hkv, bs, d = kc[0].shape
        self._kp = (ctypes.c_void_p * len(kc))(*[t.data_ptr() for t in kc])
        self._vp = (ctypes.c_void_p * len(vc))(*[t.data_ptr() for t in vc])
        self._caches = (kc, vc)
        cfg = cb_executor_config(len(kc), ctypes.cast(self._kp, ctypes.POINTER(ctypes.c_void_p)),
                                 ctypes.cast(self._vp, ctypes.POINTER(ctypes.c_void_p)), nb, bs,
                                 num_q_heads, hkv, d, _dtype_code(kc[0]), float(scale),
                                 int(sliding_window), max_reqs, max_tokens, max_blocks_per_seq)
        h = ctypes.c_void_p()
        _check(_lib.cb_executor_create(ctypes.byref(cfg), ctypes.byref(h)))
        self._h = h
        self.num_layers = len(kc)

    def close(self):
        if getattr(self, "_h", None):
            _lib.cb_executor_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def _bufs(self, q, k, v, out):
        (qp, qs), (kp, ks), (vp, vs), (op, os_) = _ptrs(q), _ptrs(k), _ptrs(v), _ptrs(out)
        if not (len(qs) == len(ks) == len(vs) == len(os_) == self.num_layers):
            raise ValueError("one q/k/v/out tensor per layer expected")
        for t in qs + ks + vs + os_:
            if t.is_cuda or not t.is_contiguous():
                raise ValueError("executor inputs and outputs are contiguous host tensors")
        P = ctypes.POINTER(ctypes.c_void_p)
        return [ctypes.cast(x, P) for x in (qp, kp, vp, op)]

    def run_step(self, sched, q, k, v, out):
        """One serving step of ``sched`` (schedule + submit + commit); returns
        (tokens, rows) of the step.  Raises CBError(CB_ERR_NO_BLOCKS) when
        nothing could be scheduled."""
        bufs = self._bufs(q, k, v, out)
        n, r = ctypes.c_int32(), ctypes.c_int32()
        _check(_lib.cb_executor_run_step(self._h, sched._h, *bufs, ctypes.byref(n), ctypes.byref(r)))
        return int(n.value), int(r.value)

    def submit(self, step: dict, q, k, v, out) -> None:
        """Queue a step already scheduled (the dict ``Scheduler.schedule_step``
        returns); its arrays are packed before this returns."""
        bufs = self._bufs(q, k, v, out)
        R, T = int(step["num_reqs"]), int(step["num_tokens"])
        i32p = ctypes.POINTER(ctypes.c_int32)
        arrs = [np.ascontiguousarray(step[k_], dtype=np.int32)
                for k_ in ("cu_seqlens_q", "seq_lens", "block_tables", "slot_mapping")]
        bt = arrs[2].reshape(R, -1) if R else arrs[2].reshape(0, 1)
        c = cb_step()
        c.num_reqs, c.num_tokens, c.num_decodes = R, T, int(step["num_decodes"])
        c.max_q_len = int(step.get("max_q_len", 1))
        c.max_seq_len = int(step.get("max_seq_len", 1))
        c.max_blocks_per_seq = int(bt.shape[1])
        c.cu_seqlens_q = arrs[0].ctypes.data_as(i32p)
        c.seq_lens = arrs[1].ctypes.data_as(i32p)
        c.block_tables = arrs[2].ctypes.data_as(i32p)
        c.slot_mapping = arrs[3].ctypes.data_as(i32p)
        c.num_swap_in = len(step.get("swap_in", ()))
        c.num_swap_out = len(step.get("swap_out", ()))
        _check(_lib.cb_executor_submit(self._h, ctypes.byref(c), *bufs))

    def synchronize(self) -> None:
        _check(_lib.cb_executor_synchronize(self._h))

    def stats(self):
        """(steps, tokens, compute milliseconds) since creation or reset."""
        a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_double()
        _check(_lib.cb_executor_stats(self._h, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)))
        return int(a.value), int(b.value), float(c.value)

    def reset_stats(self) -> None:
        _check(_lib.cb_executor_reset_stats(self._h))

    def read_errors(self) -> int:
        bits = ctypes.c_uint32()
        st = _lib.cb_executor_read_errors(self._h, ctypes.byref(bits))
        if st not in (CB_OK, CB_ERR_DEVICE_CHECK):
            _check(st)
        return int(bits.value)


def paged_attention_args(**kw) -> cb_attention_args:
    """Build a raw cb_attention_args (for callers that drive the C ABI
    directly, e.g. with CUDA graphs)."""
    return cb_attention_args(**kw)


__all__ = ["Scheduler", "kv_append", "kv_swap", "validate_step", "paged_attention", "Workspace", "workspace_size",
           "Executor",
           "CBError", "version", "library", "LIB_PATH"]
