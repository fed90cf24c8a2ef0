"""cb_paged_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (a plugin running inside a host framework that owns
the memory budget, or a loop that cannot pay for cudaMalloc's implicit
synchronisation).  It takes no workspace and keeps its scratch in a fixed
array inside the library.

The GPU test calls it through the C ABI twice in a row, on two different
decode batches, and checks each output against cb_paged_attention (which
uses a caller-allocated workspace) within the bf16 tolerance used by every
parity test.  This file is collected last so that, in a run that stops at
the first failure, every other test has already run.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads

BF16_ATOL, BF16_RTOL = 2e-2, 1e-2


def _lib():
    import paged_attention_continuous_gb300 as cb
    lib = cb.library()
    lib.cb_paged_decode_noalloc.argtypes = [ctypes.POINTER(cb.cb_attention_args),
                                            ctypes.c_void_p, ctypes.c_void_p]
    lib.cb_paged_decode_noalloc.restype = ctypes.c_int
    return cb, lib


def _args(cb, q, out, kc, vc, cu, sl, bt, max_seq_len):
    T, Hq, D = q.shape
    nb, Hkv, bs, _ = kc.shape
    return cb.cb_attention_args(
        q=q.data_ptr(), out=out.data_ptr(), k_cache=kc.data_ptr(), v_cache=vc.data_ptr(),
        cu_seqlens_q=cu.data_ptr(), seq_lens=sl.data_ptr(), block_tables=bt.data_ptr(),
        num_reqs=T, num_decodes=T, num_tokens=T, max_q_len=1, max_seq_len=max_seq_len,
        num_blocks=nb, max_blocks_per_seq=bt.shape[1], block_size=bs, num_q_heads=Hq,
        num_kv_heads=Hkv, head_dim=D, scale=float(D) ** -0.5, dtype=cb.DTYPE_BF16,
        workspace=None, workspace_bytes=0)


def test_rejects_sizes_beyond_the_fixed_scratch():
    cb, lib = _lib()
    # 1024 rows x 64 query heads x (128 + 2) floats x 2 slots per row > 64 MiB
    a = cb.cb_attention_args(q=16, out=16, k_cache=16, v_cache=16, cu_seqlens_q=16,
                             seq_lens=16, block_tables=16, num_reqs=1024, num_decodes=1024,
                             num_tokens=1024, max_q_len=1, max_seq_len=16, num_blocks=10,
                             max_blocks_per_seq=4, block_size=16, num_q_heads=64,
                             num_kv_heads=8, head_dim=128, scale=0.1, dtype=cb.DTYPE_BF16)
    st = lib.cb_paged_decode_noalloc(ctypes.byref(a), None, None)
    assert st == cb.CB_ERR_INVALID_ARG
    assert "scratch" in lib.cb_last_error().decode()
    a.num_decodes = 1023  # a prefill row present: refused, it serves decodes only
    assert lib.cb_paged_decode_noalloc(ctypes.byref(a), None, None) == cb.CB_ERR_INVALID_ARG


@pytest.mark.gpu
def test_no_alloc_decode_matches_workspace_entry_point_twice():
    cb, lib = _lib()
    dev = "cuda"
    Hq, Hkv, D, bs = 32, 8, 128, 16
    rng = np.random.default_rng(21)
    nb = 8000
    kc = workloads.cache_fill(nb, Hkv, bs, D, seed=31, dtype="bf16", scale=0.5, device=dev)
    vc = workloads.cache_fill(nb, Hkv, bs, D, seed=32, dtype="bf16", scale=0.5, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    for call, R in enumerate((37, 19)):
        seq = rng.integers(2, 2500, size=R).astype(np.int32)
        W = int(-(-seq.max() // bs))
        perm = rng.permutation(nb).astype(np.int32)
        bt = np.full((R, W), -1, dtype=np.int32)
        o = 0
        for r in range(R):
            n = int(-(-seq[r] // bs))
            bt[r, :n] = perm[o:o + n]
            o += n
        cu = torch.arange(R + 1, dtype=torch.int32, device=dev)
        sl = torch.from_numpy(seq).to(dev)
        btd = torch.from_numpy(bt).to(dev)
        q = workloads.token_tensors(R, Hq, D, seed=40 + call, dtype="bf16", scale=0.5, device=dev)
        ref = cb.paged_attention(q, kc, vc, cu, sl, btd, num_decodes=R, max_q_len=1,
                                 max_seq_len=int(seq.max()), scale=D ** -0.5,
                                 workspace=cb.Workspace(R, Hq, Hkv, D))
        out = torch.full_like(q, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        a = _args(cb, q, out, kc, vc, cu, sl, btd, int(seq.max()))
        st = lib.cb_paged_decode_noalloc(ctypes.byref(a), err.data_ptr(), stream)
        assert st == cb.CB_OK, lib.cb_last_error().decode()
        torch.cuda.synchronize()
        assert err.item() == 0
        g = out.double().cpu().numpy()
        rf = ref.double().cpu().numpy()
        assert np.isfinite(g).all()
        assert (np.abs(g - rf) <= BF16_ATOL + BF16_RTOL * np.abs(rf)).all(), f"call {call}"


@pytest.mark.gpu
def test_no_alloc_many_rows_plans_larger_splits():
    """800 rows x 64 query heads leave the fixed scratch room for fewer
    partial slots than the plan first asks for; the kernel then plans larger
    splits and must still agree with the workspace entry point."""
    cb, lib = _lib()
    dev = "cuda"
    Hq, Hkv, D, bs, R = 64, 8, 128, 16, 800
    rng = np.random.default_rng(5)
    nb = 3000
    kc = workloads.cache_fill(nb, Hkv, bs, D, seed=51, dtype="bf16", scale=0.5, device=dev)
    vc = workloads.cache_fill(nb, Hkv, bs, D, seed=52, dtype="bf16", scale=0.5, device=dev)
    seq = rng.integers(2, 600, size=R).astype(np.int32)
    W = int(-(-seq.max() // bs))
    bt = np.full((R, W), -1, dtype=np.int32)
    for r in range(R):
        n = int(-(-seq[r] // bs))
        bt[r, :n] = rng.choice(nb, size=n, replace=False)  # rows may share blocks
    cu = torch.arange(R + 1, dtype=torch.int32, device=dev)
    sl = torch.from_numpy(seq).to(dev)
    btd = torch.from_numpy(bt).to(dev)
    q = workloads.token_tensors(R, Hq, D, seed=60, dtype="bf16", scale=0.5, device=dev)
    ref = cb.paged_attention(q, kc, vc, cu, sl, btd, num_decodes=R, max_q_len=1,
                             max_seq_len=int(seq.max()), scale=D ** -0.5,
                             workspace=cb.Workspace(R, Hq, Hkv, D))
    out = torch.full_like(q, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    a = _args(cb, q, out, kc, vc, cu, sl, btd, int(seq.max()))
    st = lib.cb_paged_decode_noalloc(ctypes.byref(a), err.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream)
    assert st == cb.CB_OK, lib.cb_last_error().decode()
    torch.cuda.synchronize()
    assert err.item() == 0
    g = out.double().cpu().numpy()
    rf = ref.double().cpu().numpy()
    assert np.isfinite(g).all()
    assert (np.abs(g - rf) <= BF16_ATOL + BF16_RTOL * np.abs(rf)).all()
