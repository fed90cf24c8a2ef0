"""GPU parity: the CUDA path (through the C ABI) against the oracle.

Bars: KV cache contents and scheduler metadata bit-exact; fp32 outputs
max-abs <= 1e-4; bf16 outputs |gpu - oracle| <= 2e-2 + 1e-2 * |oracle|
elementwise.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import attention as oatt
from oracle import paged_kv
from tests.gpu_harness import ParityRun, tolerance_ok

pytestmark = pytest.mark.gpu


def _cb():
    import paged_attention_continuous_gb300 as cb
    return cb


def _check(gpu, ref, dtype, what=""):
    ok, err, excess = tolerance_ok(gpu, ref, dtype)
    assert ok, f"{what}: max err {err:.3e}, worst excess over bound {excess:.3e}"
    return err


# ---------------------------------------------------------------- append
@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f32", 64), ("bf16", 64)])
def test_kv_append_bit_exact(dtype, D):
    cb = _cb()
    nb, Hkv, bs, T = 40, 4, 16, 77
    rng = np.random.default_rng(3)
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int32)
    slots[[5, 17, 40]] = -1
    k0 = workloads.cache_fill(nb, Hkv, bs, D, seed=1, dtype=dtype, device="cuda")
    v0 = workloads.cache_fill(nb, Hkv, bs, D, seed=2, dtype=dtype, device="cuda")
    kn = workloads.token_tensors(T, Hkv, D, seed=3, dtype=dtype, device="cuda")
    vn = workloads.token_tensors(T, Hkv, D, seed=4, dtype=dtype, device="cuda")
    ko = k0.double().cpu().numpy(); vo = v0.double().cpu().numpy()
    paged_kv.append(ko, vo, kn.double().cpu().numpy(), vn.double().cpu().numpy(), slots, bs)
    kc, vc = k0.clone(), v0.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cb.kv_append(kn, vn, torch.from_numpy(slots).cuda(), kc, vc, error_word=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    tdt = kc.dtype
    assert torch.equal(kc.cpu(), torch.from_numpy(ko).to(tdt))
    assert torch.equal(vc.cpu(), torch.from_numpy(vo).to(tdt))


def test_kv_append_out_of_range_slot_is_flagged_not_written():
    cb = _cb()
    nb, Hkv, bs, D = 4, 2, 16, 128
    kc = torch.zeros(nb, Hkv, bs, D, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    kn = torch.ones(2, Hkv, D, dtype=torch.bfloat16, device="cuda")
    slots = torch.tensor([3, nb * bs + 5], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cb.kv_append(kn, kn, slots, kc, vc, error_word=err)
    torch.cuda.synchronize()
    assert err.item() == cb.DEVERR_SLOT_RANGE
    assert kc.float().sum().item() == Hkv * D      # only slot 3 written


# ---------------------------------------------------------------- decode
def _decode_scenario(ctx, Hq, Hkv, D, dtype, seed=0, extra_blocks=7):
    running = [workloads.RunningRequest(req_id=i, prompt_len=c - 1, output_len=8, num_cached=c - 1)
               for i, c in enumerate(ctx)]
    nb = sum(-(-c // 16) for c in ctx) + extra_blocks
    return workloads.Scenario(
        name="decode_edges", num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, dtype=dtype,
        num_blocks=nb, max_batch_tokens=len(ctx), max_requests_per_batch=len(ctx),
        max_prefill_chunk=0, safety_margin=0.0, max_blocks_per_seq=0,
        free_list=workloads.permuted_free_list(nb, seed + 5), running=running, waiting=[],
        value_scale=0.5 if dtype == "bf16" else 1.0, seed=seed)


EDGE_CTX = [2, 3, 15, 16, 17, 31, 32, 33, 100, 255, 256, 257, 1000, 2049]


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f32", 64), ("f32", 128), ("bf16", 64)])
@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 4), (32, 8), (16, 2), (64, 4)])
def test_decode_edges(dtype, D, Hq, Hkv):
    """GQA 1, 2, 4, 8 and 16 (bf16: the matrix-instruction instantiations,
    seven warps per CTA at 16; fp32 at 16: the CUDA-core fallback)."""
    sc = _decode_scenario(EDGE_CTX, Hq, Hkv, D, dtype)
    run = ParityRun(sc)
    st, g, r, _ = run.step()
    assert st == 0
    _check(g[0], r[0], dtype, "decode")
    # a second step (every context one longer) reuses the workspace
    st, g, r, _ = run.step()
    _check(g[0], r[0], dtype, "decode step 2")


def test_decode_many_splits_and_rows():
    ctx = list(np.random.default_rng(0).integers(2, 9000, size=70))
    sc = _decode_scenario(ctx, 32, 8, 128, "bf16")
    run = ParityRun(sc)
    st, g, r, _ = run.step()
    _check(g[0], r[0], "bf16", "decode 70 rows")


@pytest.mark.parametrize("dtype,Hq,Hkv,D", [("bf16", 32, 8, 128), ("bf16", 64, 8, 128),
                                            ("bf16", 64, 4, 128), ("f32", 16, 4, 128)])
def test_decode_few_long_rows(dtype, Hq, Hkv, D):
    """A handful of very long caches next to tiny ones: each long row is cut
    into hundreds of splits (both phases), merged in the same kernel by the
    warps that run out of items."""
    sc = _decode_scenario([40001, 32768, 17, 2], Hq, Hkv, D, dtype)
    run = ParityRun(sc)
    st, g, r, _ = run.step()
    assert st == 0
    _check(g[0], r[0], dtype, "decode few long rows")


def test_paging_invisible_on_gpu():
    """Different physical placements of the same logical cache give
    bit-identical GPU outputs."""
    outs = []
    for seed in (0, 11):
        sc = _decode_scenario(EDGE_CTX, 32, 8, 128, "bf16", seed=0)
        sc.free_list = workloads.permuted_free_list(sc.num_blocks, seed + 100)
        run = ParityRun(sc)
        # the initial pool contents follow the logical positions: rewrite the
        # context tokens of every request identically for both placements
        for r in sc.running:
            slots = run.c.slots(r.req_id, 0, r.num_cached)
            kv = workloads.token_tensors(r.num_cached, sc.num_kv_heads, sc.head_dim,
                                         seed=1000 + r.req_id, dtype="bf16", scale=0.5, device="cuda")
            vv = workloads.token_tensors(r.num_cached, sc.num_kv_heads, sc.head_dim,
                                         seed=2000 + r.req_id, dtype="bf16", scale=0.5, device="cuda")
            _cb().kv_append(kv, vv, torch.from_numpy(slots).cuda(), run.runner.k_cache[0],
                            run.runner.v_cache[0])
        step = run.c.schedule_step()
        ds = run.runner.upload(step)
        T = step["num_tokens"]
        q = workloads.token_tensors(T, 32, 128, seed=7, dtype="bf16", scale=0.5, device="cuda")
        k = workloads.token_tensors(T, 8, 128, seed=8, dtype="bf16", scale=0.5, device="cuda")
        v = workloads.token_tensors(T, 8, 128, seed=9, dtype="bf16", scale=0.5, device="cuda")
        outs.append(run.runner.run(ds, q, k, v).cpu())
    assert torch.equal(outs[0], outs[1])


# --------------------------------------------------------------- prefill
def test_worked_example_fp32_chunked():
    """The Chunked Prefill page's example through the whole path: 1000-token
    prompt, 8 heads x 64 dims, fp32, budget 256 -> 256/256/256/232, block
    size 16, permuted physical blocks; compared with one-shot attention."""
    cb = _cb()
    from paged_attention_continuous_gb300.step import StepRunner
    q, k, v = workloads.worked_example_qkv()                 # [1, 8, 1000, 64]
    qt = q[0].permute(1, 0, 2).contiguous()                 # [1000, 8, 64]
    kt = k[0].permute(1, 0, 2).contiguous()
    vt = v[0].permute(1, 0, 2).contiguous()
    sc = workloads.chunked_prefill_1000()
    s = cb.Scheduler(block_size=16, num_blocks=sc.num_blocks, max_batch_tokens=256,
                     max_requests_per_batch=8, max_blocks_per_seq=sc.max_blocks_per_seq,
                     safety_margin=0.0, free_list=sc.free_list)
    s.add_request(0, 1000, 1)
    runner = StepRunner(num_blocks=sc.num_blocks, num_q_heads=8, num_kv_heads=8, head_dim=64,
                        dtype="f32", max_reqs=8, max_tokens=256,
                        max_blocks_per_seq=sc.max_blocks_per_seq)
    outs, chunks = [], []
    while True:
        st = s.schedule_step()
        if st["num_reqs"] == 0:
            break
        p1 = int(st["seq_lens"][0]); n = int(st["cu_seqlens_q"][1]); p0 = p1 - n
        chunks.append(n)
        ds = runner.upload(st)
        o = runner.run(ds, qt[p0:p1].cuda(), kt[p0:p1].cuda(), vt[p0:p1].cuda())
        outs.append(o.double().cpu().numpy())
        s.step_done()
    assert chunks == [256, 256, 256, 232]
    gpu = np.concatenate(outs)
    ref = oatt.dense_causal_attention(qt.double().numpy(), kt.double().numpy(),
                                      vt.double().numpy(), 1 / 8.0)
    assert np.max(np.abs(gpu - ref)) <= 1e-4


def _mixed_small(dtype="bf16", Hq=32, Hkv=8, D=128, seed=0):
    rng = np.random.default_rng(seed)
    ctx = rng.integers(20, 600, size=10)
    running = [workloads.RunningRequest(i, int(c) - 1, 40, int(c) - 1) for i, c in enumerate(ctx)]
    running.append(workloads.RunningRequest(10, 300, 4, 64))
    waiting = [workloads.WaitingRequest(11 + i, int(p), 3)
               for i, p in enumerate(rng.integers(1, 200, size=8))]
    nb = 1200
    return workloads.Scenario(
        name="mixed_small", num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, dtype=dtype,
        num_blocks=nb, max_batch_tokens=256, max_requests_per_batch=24, max_prefill_chunk=128,
        safety_margin=0.15, max_blocks_per_seq=0,
        free_list=workloads.permuted_free_list(nb, seed + 1), running=running, waiting=waiting,
        value_scale=0.5 if dtype == "bf16" else 1.0, seed=seed)


@pytest.mark.parametrize("dtype,Hq,Hkv,D", [("bf16", 32, 8, 128), ("bf16", 16, 16, 128),
                                           ("bf16", 64, 8, 128), ("f32", 8, 2, 64),
                                           ("bf16", 8, 4, 64)])
def test_mixed_steps_small(dtype, Hq, Hkv, D):
    sc = _mixed_small(dtype, Hq, Hkv, D)
    run = ParityRun(sc)
    for step in range(5):
        st, g, r, _ = run.step()
        assert st == 0
        _check(g[0], r[0], dtype, f"mixed step {step}")


def test_prefill_chunk_of_one_and_seq_len_one():
    """A chunk of length 1 that is not a decode, and a first chunk of 1 token
    (seq_len 1, output must equal v[0])."""
    waiting = [workloads.WaitingRequest(0, 1, 2), workloads.WaitingRequest(1, 17, 2),
               workloads.WaitingRequest(2, 40, 2)]
    sc = workloads.Scenario(
        name="tiny", num_q_heads=8, num_kv_heads=2, head_dim=128, dtype="bf16",
        num_blocks=64, max_batch_tokens=18, max_requests_per_batch=4, max_prefill_chunk=0,
        safety_margin=0.0, max_blocks_per_seq=0, free_list=workloads.permuted_free_list(64, 2),
        running=[], waiting=waiting, value_scale=0.5)
    run = ParityRun(sc)
    for _ in range(4):
        st, g, r, _ = run.step()
        if st != 0 or g[0].shape[0] == 0:
            break
        _check(g[0], r[0], "bf16", "tiny prefill")


# ------------------------------------------------------- full-size configs
def test_full_decode_64_sampled():
    sc = workloads.decode_64()
    run = ParityRun(sc, sample=[0, 1, 17, 33, 62, 63])
    st, g, r, toks = run.step()
    assert st == 0 and len(toks) == 6
    _check(g[0], r[0], "bf16", "decode_64")


def test_full_mixed_2048_sampled():
    sc = workloads.mixed_2048()
    sample = [0, 5, 50, 95, 96, 97, 98]     # decodes, the in-flight prefill, new prompts
    run = ParityRun(sc, sample=sample)
    st, g, r, toks = run.step()
    assert st == 0
    _check(g[0], r[0], "bf16", "mixed_2048")
    st, g, r, toks = run.step()
    _check(g[0], r[0], "bf16", "mixed_2048 step 2")


def test_full_long_prompt_late_step_sampled():
    """Long-prompt interleave at full shape (64 Q / 8 KV heads, 128 decodes);
    steps 0..5 run, the oracle follows 3 decodes and the long prompt."""
    sc = workloads.long_prompt_32k()
    run = ParityRun(sc, sample=[0, 64, 127, 128])
    for step in range(6):
        st, g, r, toks = run.step()
        assert st == 0
    _check(g[0], r[0], "bf16", "long prompt step 6")


def test_full_long_prompt_late_chunks():
    """The long-prompt interleave through its whole 32,768-token prompt: 64
    steps of 512-token chunks at offsets 0 .. 32,256 next to 128 growing
    decodes (64 Q / 8 KV heads).  The oracle follows decode row 0 and the
    prompt; every query of chunks 16, 32 and 63 (keys up to 8,704, 16,896
    and 32,768) is compared element by element."""
    sc = workloads.long_prompt_32k()
    run = ParityRun(sc, sample=[0, 128])
    checks = {16, 32, 63}
    for step in range(64):
        st, g, r, toks = run.step(check=step in checks)
        assert st == 0
        if step in checks:
            assert len(toks) == 513
            _check(g[0], r[0], "bf16", f"long prompt chunk {step}")
    assert int(run.last["seq_lens"][-1]) == 32768


def test_full_prefill_chunk_16k():
    """The 512-token chunk at offset 16,384 (64 Q / 8 KV heads) that the
    prefill kernel's counters are quoted on, every query and head."""
    sc = workloads.prefill_chunk_16k()
    run = ParityRun(sc)
    st, g, r, toks = run.step()
    assert st == 0 and len(toks) == 512
    _check(g[0], r[0], "bf16", "prefill_chunk_16k")


def test_prefill_short_chunks_long_context():
    """Short chunks of long requests: few query tiles, each against
    hundreds of KV tiles -- two requests with 192- and 64-token chunks at
    offsets 30,000 and 12,000 (64 Q / 8 KV heads), every query compared."""
    running = [workloads.RunningRequest(0, 30192, 4, 30000),
               workloads.RunningRequest(1, 12064, 4, 12000)]
    nb = 3000
    sc = workloads.Scenario(
        name="short_chunks", num_q_heads=64, num_kv_heads=8, head_dim=128, dtype="bf16",
        num_blocks=nb, max_batch_tokens=256, max_requests_per_batch=4, max_prefill_chunk=0,
        safety_margin=0.0, max_blocks_per_seq=0, free_list=workloads.permuted_free_list(nb, 9),
        running=running, waiting=[], value_scale=0.5)
    run = ParityRun(sc)
    st, g, r, toks = run.step()
    assert st == 0 and len(toks) == 256
    _check(g[0], r[0], "bf16", "short chunks, long context")


def test_trace_first_steps_sampled_all_layers():
    """The request trace (Poisson arrivals, lognormal lengths, 4 layers with
    their own pools): its first 10 steps with arrivals added per step; the
    oracle follows four short requests (two arriving at step 0, one at 1,
    one at 2) through prefill and decode on every layer."""
    sc = workloads.trace_2000()
    run = ParityRun(sc, sample=[1, 5, 25, 39], arrivals=True)
    seen = 0
    for step in range(10):
        st, g, r, toks = run.step()
        assert st == 0
        for layer in range(sc.num_layers):
            if len(toks):
                _check(g[layer], r[layer], "bf16", f"trace step {step} layer {layer}")
        seen += len(toks)
    assert seen > 0


def test_empty_batch_is_a_noop():
    cb = _cb()
    ws = cb.Workspace(4, 8, 8, 128)
    a = cb.cb_attention_args()
    a.num_reqs = 0
    assert cb.library().cb_paged_attention(__import__("ctypes").byref(a), None) == 0


def test_bad_block_id_is_flagged_not_read():
    cb = _cb()
    sc = _decode_scenario([40, 50], 8, 2, 128, "bf16")
    run = ParityRun(sc)
    step = run.c.schedule_step()
    step["block_tables"][1, 1] = sc.num_blocks + 7        # corrupt one entry
    ds = run.runner.upload(step)
    T = step["num_tokens"]
    q = torch.zeros(T, 8, 128, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(T, 2, 128, dtype=torch.bfloat16, device="cuda")
    run.runner.run(ds, q, kv, kv)
    bits = run.runner.workspace.read_errors()
    assert bits & cb.DEVERR_BLOCK_RANGE
    run.runner.workspace.reinit()
    torch.cuda.synchronize()


def test_workspace_reused_across_calls_of_different_sizes():
    """One workspace serves calls with different row counts: a decode-only
    call with few rows, then the full mixed step, must give the same bytes as
    the full step on a fresh workspace."""
    cb = _cb()
    sc = _mixed_small("bf16", 16, 16, 128)
    run = ParityRun(sc)
    st = run.c.schedule_step()
    ds = run.runner.upload(st)
    T, nd = st["num_tokens"], st["num_decodes"]
    q = workloads.token_tensors(T, 16, 128, seed=1, dtype="bf16", scale=0.5, device="cuda")
    k = workloads.token_tensors(T, 16, 128, seed=2, dtype="bf16", scale=0.5, device="cuda")
    kc, vc = run.runner.k_cache[0], run.runner.v_cache[0]
    cb.kv_append(k, k, ds.slot_mapping, kc, vc)
    kw = dict(scale=0.0884, out=None)
    full = dict(num_decodes=nd, max_q_len=st["max_q_len"], max_seq_len=st["max_seq_len"])
    ws = run.runner.workspace
    for n in (3, nd):
        cb.paged_attention(q[:n], kc, vc, ds.cu_seqlens_q[:n + 1], ds.seq_lens[:n],
                           ds.block_tables[:n], num_decodes=n, max_q_len=1,
                           max_seq_len=int(st["seq_lens"][:n].max()), workspace=ws, **kw)
    a = cb.paged_attention(q, kc, vc, ds.cu_seqlens_q, ds.seq_lens, ds.block_tables,
                           workspace=ws, **full, **kw)
    fresh = cb.Workspace(sc.max_requests_per_batch, 16, 16, 128)
    b = cb.paged_attention(q, kc, vc, ds.cu_seqlens_q, ds.seq_lens, ds.block_tables,
                           workspace=fresh, **full, **kw)
    torch.cuda.synchronize()
    assert ws.read_errors() == 0
    assert torch.equal(a, b)


def test_attention_after_append_overlap_is_bit_identical():
    """after_append=True lets the decode kernel start while the step's
    append finishes (it waits for it before reading the cache); the output
    must be the same bytes as with plain stream order, over several mixed
    steps on their own pools, with the append re-run right before each."""
    cb = _cb()
    sc = _mixed_small("bf16", 32, 8, 128, seed=3)
    outs = {}
    for flag in (False, True):
        run = ParityRun(sc)
        res = []
        for step_i in range(3):
            st = run.c.schedule_step()
            assert st["status"] == 0
            ds = run.runner.upload(st)
            T = st["num_tokens"]
            q = workloads.token_tensors(T, 32, 128, seed=10 + step_i, dtype="bf16", scale=0.5,
                                        device="cuda")
            k = workloads.token_tensors(T, 8, 128, seed=20 + step_i, dtype="bf16", scale=0.5,
                                        device="cuda")
            v = workloads.token_tensors(T, 8, 128, seed=30 + step_i, dtype="bf16", scale=0.5,
                                        device="cuda")
            kc, vc = run.runner.k_cache[0], run.runner.v_cache[0]
            cb.kv_append(k, v, ds.slot_mapping, kc, vc)
            o = cb.paged_attention(q, kc, vc, ds.cu_seqlens_q, ds.seq_lens, ds.block_tables,
                                   num_decodes=st["num_decodes"], max_q_len=st["max_q_len"],
                                   max_seq_len=st["max_seq_len"], scale=sc.softmax_scale,
                                   workspace=run.runner.workspace, after_append=flag)
            res.append(o.clone())
            run.c.step_done()
        torch.cuda.synchronize()
        assert run.runner.workspace.read_errors() == 0
        outs[flag] = res
    for a, b in zip(outs[False], outs[True]):
        assert torch.equal(a, b)


def test_trace_late_steps_sampled_all_layers():
    """The request trace far past its start: every request runs on the GPU
    (4 layers), while the oracle follows two long-lived requests that
    arrive at steps 40 and 60 and, behind the queue, run from about step
    460 and 720 to 930 and 1140 -- prefill through hundreds of decode steps
    at sequence lengths up to ~1,900, on every layer."""
    sc = workloads.trace_2000()
    picks = []
    for w in sc.waiting:
        if w.arrival_step >= 40 + 20 * len(picks) and w.output_len >= 250 and w.prompt_len <= 3000:
            picks.append(w.req_id)
        if len(picks) == 2:
            break
    run = ParityRun(sc, sample=picks, arrivals=True)
    seen_steps, longest = 0, 0
    for step in range(1300):
        st, g, r, toks = run.step()
        assert st == 0
        if len(toks):
            for layer in range(sc.num_layers):
                _check(g[layer], r[layer], "bf16", f"trace step {step} layer {layer}")
            seen_steps += 1
            rows = [i for i, rid in enumerate(run.last["req_ids"]) if int(rid) in picks]
            longest = max([longest] + [int(run.last["seq_lens"][i]) for i in rows])
        if all(p in run.o.requests and run.o.requests[p].state == "finished" for p in picks):
            break
    assert all(run.o.requests[p].state == "finished" for p in picks)
    assert seen_steps > 600 and longest > 1500
