"""cb_paged_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (a plugin running inside a host framework that owns
the memory budget, or a loop that cannot pay for cudaMalloc's implicit
synchronisation).  It takes no workspace and keeps its scratch in a fixed
array inside the library.

The GPU tests call it through the C ABI twice in a row, on two different
decode batches, and check each output against cb_paged_attention (which
uses a caller-allocated workspace and so plans different splits) within the
bf16 tolerance used by every parity test, and both outputs against the
oracle.  A windowed batch and an fp32 batch go through the same checks.
This file is collected last so that, in a run that stops at the first
failure, every other test has already run.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from oracle import attention as oatt

TOL = {"bf16": (2e-2, 1e-2), "f32": (1e-4, 0.0)}


def _lib():
    import paged_attention_continuous_gb300 as cb
    lib = cb.library()
    lib.cb_paged_decode_noalloc.argtypes = [ctypes.POINTER(cb.cb_attention_args),
                                            ctypes.c_void_p, ctypes.c_void_p]
    lib.cb_paged_decode_noalloc.restype = ctypes.c_int
    return cb, lib


def _args(cb, q, out, kc, vc, cu, sl, bt, max_seq_len, window=0):
    T, Hq, D = q.shape
    nb, Hkv, bs, _ = kc.shape
    return cb.cb_attention_args(
        q=q.data_ptr(), out=out.data_ptr(), k_cache=kc.data_ptr(), v_cache=vc.data_ptr(),
        cu_seqlens_q=cu.data_ptr(), seq_lens=sl.data_ptr(), block_tables=bt.data_ptr(),
        num_reqs=T, num_decodes=T, num_tokens=T, max_q_len=1, max_seq_len=max_seq_len,
        num_blocks=nb, max_blocks_per_seq=bt.shape[1], block_size=bs, num_q_heads=Hq,
        num_kv_heads=Hkv, head_dim=D, scale=float(D) ** -0.5,
        dtype=cb.DTYPE_BF16 if q.dtype == torch.bfloat16 else cb.DTYPE_F32,
        workspace=None, workspace_bytes=0, sliding_window=window)


def _close(g, r, dtype):
    atol, rtol = TOL[dtype]
    return bool((np.abs(g - r) <= atol + rtol * np.abs(r)).all()), float(np.abs(g - r).max())


def _oracle(q, kc, vc, seq, bt, window):
    """The oracle on a compact copy of the blocks the table references."""
    used = sorted({int(b) for b in bt.reshape(-1) if b >= 0})
    sel = torch.tensor(used, dtype=torch.long, device=kc.device)
    k = kc.index_select(0, sel).double().cpu().numpy()
    v = vc.index_select(0, sel).double().cpu().numpy()
    remap = {b: i for i, b in enumerate(used)}
    tab = np.vectorize(lambda b: remap.get(int(b), -1))(bt) if bt.size else bt
    R = len(seq)
    return oatt.paged_attention(q.double().cpu().numpy(), k, v, np.arange(R + 1), seq, tab,
                                kc.shape[2], float(q.shape[2]) ** -0.5, window=window)


def _batch(rng, R, nb, bs, lo, hi, window=0):
    """Sequence lengths and a block table over a permuted pool; with a
    window, table entries of pages wholly before each row's window are -1
    (pages recycled by the scheduler) and never read."""
    seq = rng.integers(lo, hi, size=R).astype(np.int32)
    W = int(-(-seq.max() // bs))
    perm = rng.permutation(nb).astype(np.int32)
    bt = np.full((R, W), -1, dtype=np.int32)
    o = 0
    for r in range(R):
        n = int(-(-seq[r] // bs))
        first = (max(0, int(seq[r]) - window) // bs) if window else 0
        bt[r, first:n] = perm[o:o + n - first]
        o += n - first
    return seq, bt


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
    # a head size the kernels do not have is refused before any sizing
    for hd in (-2, 0, 96):
        a = cb.cb_attention_args(q=16, out=16, k_cache=16, v_cache=16, cu_seqlens_q=16,
                                 seq_lens=16, block_tables=16, num_reqs=4, num_decodes=4,
                                 num_tokens=4, max_q_len=1, max_seq_len=16, num_blocks=10,
                                 max_blocks_per_seq=4, block_size=16, num_q_heads=8,
                                 num_kv_heads=8, head_dim=hd, scale=0.1, dtype=cb.DTYPE_BF16)
        assert lib.cb_paged_decode_noalloc(ctypes.byref(a), None, None) == cb.CB_ERR_UNSUPPORTED
    # a GQA group the kernels do not have
    a.head_dim, a.num_q_heads, a.num_kv_heads = 128, 24, 8
    assert lib.cb_paged_decode_noalloc(ctypes.byref(a), None, None) == cb.CB_ERR_UNSUPPORTED


def _run_pair(cb, lib, kc, vc, seq, bt, q, window=0):
    """The no-alloc call and cb_paged_attention on the same batch."""
    dev = kc.device
    R = len(seq)
    Hq, D = q.shape[1], q.shape[2]
    Hkv = kc.shape[1]
    cu = torch.arange(R + 1, dtype=torch.int32, device=dev)
    sl = torch.from_numpy(seq).to(dev)
    btd = torch.from_numpy(bt).to(dev)
    ref = cb.paged_attention(q, kc, vc, cu, sl, btd, num_decodes=R, max_q_len=1,
                             max_seq_len=int(seq.max()), scale=D ** -0.5,
                             workspace=cb.Workspace(R, Hq, Hkv, D), sliding_window=window)
    out = torch.full_like(q, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    a = _args(cb, q, out, kc, vc, cu, sl, btd, int(seq.max()), window)
    st = lib.cb_paged_decode_noalloc(ctypes.byref(a), err.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream)
    assert st == cb.CB_OK, lib.cb_last_error().decode()
    torch.cuda.synchronize()
    assert err.item() == 0
    return out, ref


@pytest.mark.gpu
def test_no_alloc_decode_matches_workspace_entry_point_twice():
    cb, lib = _lib()
    dev = "cuda"
    Hq, Hkv, D, bs = 32, 8, 128, 16
    rng = np.random.default_rng(21)
    nb = 8000
    kc = workloads.cache_fill(nb, Hkv, bs, D, seed=31, dtype="bf16", scale=0.5, device=dev)
    vc = workloads.cache_fill(nb, Hkv, bs, D, seed=32, dtype="bf16", scale=0.5, device=dev)
    for call, R in enumerate((37, 19)):
        seq, bt = _batch(rng, R, nb, bs, 2, 2500)
        q = workloads.token_tensors(R, Hq, D, seed=40 + call, dtype="bf16", scale=0.5, device=dev)
        out, ref = _run_pair(cb, lib, kc, vc, seq, bt, q)
        g = out.double().cpu().numpy()
        rf = ref.double().cpu().numpy()
        assert np.isfinite(g).all()
        ok, e = _close(g, rf, "bf16")
        assert ok, f"call {call}: no-alloc vs workspace entry point, max err {e:.3e}"
        orc = _oracle(q, kc, vc, seq, bt, 0)
        for name, x in (("no-alloc", g), ("workspace", rf)):
            ok, e = _close(x, orc, "bf16")
            assert ok, f"call {call}: {name} vs oracle, max err {e:.3e}"


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,Hq,Hkv,D,window", [("bf16", 64, 8, 128, 300),
                                                   ("f32", 16, 4, 64, 0),
                                                   ("f32", 8, 8, 128, 77)])
def test_no_alloc_window_and_fp32_match_oracle(dtype, Hq, Hkv, D, window):
    """A sliding-window batch (tables hold -1 before each window) and fp32
    caches (the CUDA-core instantiations), each checked against the
    workspace entry point and the oracle at the tolerance of their dtype."""
    cb, lib = _lib()
    dev = "cuda"
    bs, R, nb = 16, 23, 3000
    rng = np.random.default_rng(9)
    kc = workloads.cache_fill(nb, Hkv, bs, D, seed=71, dtype=dtype, scale=0.5, device=dev)
    vc = workloads.cache_fill(nb, Hkv, bs, D, seed=72, dtype=dtype, scale=0.5, device=dev)
    seq, bt = _batch(rng, R, nb, bs, 1, 1500, window)
    q = workloads.token_tensors(R, Hq, D, seed=73, dtype=dtype, scale=0.5, device=dev)
    out, ref = _run_pair(cb, lib, kc, vc, seq, bt, q, window)
    g = out.double().cpu().numpy()
    rf = ref.double().cpu().numpy()
    assert np.isfinite(g).all()
    orc = _oracle(q, kc, vc, seq, bt, window)
    for name, x in (("no-alloc", g), ("workspace", rf)):
        ok, e = _close(x, orc, dtype)
        assert ok, f"{name} vs oracle, max err {e:.3e}"
    ok, e = _close(g, rf, dtype)
    assert ok, f"no-alloc vs workspace entry point, max err {e:.3e}"


@pytest.mark.gpu
def test_no_alloc_many_rows_plans_larger_splits():
    """800 rows x 64 query heads leave the fixed scratch room for fewer
    partial slots than the plan first asks for; the kernel then plans larger
    splits and must still agree with the workspace entry point and, on a
    sample of rows, with the oracle."""
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
    q = workloads.token_tensors(R, Hq, D, seed=60, dtype="bf16", scale=0.5, device=dev)
    out, ref = _run_pair(cb, lib, kc, vc, seq, bt, q)
    g = out.double().cpu().numpy()
    rf = ref.double().cpu().numpy()
    assert np.isfinite(g).all()
    ok, e = _close(g, rf, "bf16")
    assert ok, f"no-alloc vs workspace entry point, max err {e:.3e}"
    rows = np.arange(0, R, 37)
    orc = _oracle(q[torch.as_tensor(rows, device=dev)], kc, vc, seq[rows], bt[rows], 0)
    ok, e = _close(g[rows], orc, "bf16")
    assert ok, f"no-alloc vs oracle, max err {e:.3e}"
