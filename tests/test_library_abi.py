"""The C-ABI library loads and exports every function include/cb.h declares;
host-side argument checks reject bad calls before anything is launched.
No compute call here needs a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[\w\s\*]+?\b(cb_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_three_calls():
    names = _declared_functions()
    for required in ("cb_schedule_step", "cb_kv_append", "cb_paged_attention"):
        assert required in names


def test_library_exports_every_declared_symbol():
    import paged_attention_continuous_gb300 as cb
    lib = cb.library()
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_version_and_no_cpu_fallback():
    import paged_attention_continuous_gb300 as cb
    assert cb.version() >= (1 << 16)
    src = open(os.path.join(ROOT, "paged_attention_continuous_gb300", "__init__.py")).read()
    assert "oracle" not in src
    for fn in os.listdir(os.path.join(ROOT, "paged_attention_continuous_gb300")):
        if fn.endswith(".py"):
            text = open(os.path.join(ROOT, "paged_attention_continuous_gb300", fn)).read()
            assert "import oracle" not in text and "from oracle" not in text


def test_argument_errors_without_gpu():
    import paged_attention_continuous_gb300 as cb
    lib = cb.library()
    # NULL pointers are rejected on the host
    st = lib.cb_kv_append(None, None, None, 4, None, None, 10, 8, 128, 16, 1, None, None)
    assert st == cb.CB_ERR_INVALID_ARG
    st = lib.cb_kv_append(16, 16, 16, 4, 16, 16, 10, 8, 128, 12, 1, None, None)
    assert st == cb.CB_ERR_UNSUPPORTED            # block size not a power of two
    st = lib.cb_kv_append(16, 16, 16, 4, 16, 16, 10, 8, 96, 16, 1, None, None)
    assert st == cb.CB_ERR_UNSUPPORTED            # 12 vectors of 16 bytes per row
    a = cb.cb_attention_args()
    a.num_reqs, a.num_tokens, a.num_decodes = 2, 3, 3
    assert lib.cb_paged_attention(ctypes.byref(a), None) == cb.CB_ERR_INVALID_ARG
    a = cb.cb_attention_args(q=16, out=16, k_cache=16, v_cache=16, cu_seqlens_q=16,
                             seq_lens=16, block_tables=16, num_reqs=1, num_decodes=0,
                             num_tokens=1, max_q_len=1, max_seq_len=1, num_blocks=1,
                             max_blocks_per_seq=1, block_size=8, num_q_heads=4,
                             num_kv_heads=2, head_dim=128, scale=0.1, dtype=1,
                             workspace=256, workspace_bytes=1 << 30)
    assert lib.cb_paged_attention(ctypes.byref(a), None) == cb.CB_ERR_UNSUPPORTED
    a.block_size = 16
    a.num_kv_heads = 3
    assert lib.cb_paged_attention(ctypes.byref(a), None) == cb.CB_ERR_INVALID_ARG
    assert "multiple" in lib.cb_last_error().decode()
    assert cb.workspace_size(0, 0, 1, 1) == 0
    assert cb.workspace_size(96, 32, 8, 128) > 0


def test_scheduler_errors():
    import paged_attention_continuous_gb300 as cb
    with pytest.raises(cb.CBError):
        cb.Scheduler(block_size=16, num_blocks=0, max_batch_tokens=8,
                     max_requests_per_batch=2, max_blocks_per_seq=2)
    with pytest.raises(cb.CBError):
        cb.Scheduler(block_size=16, num_blocks=4, max_batch_tokens=8,
                     max_requests_per_batch=2, max_blocks_per_seq=2, free_list=[0, 1, 1, 2])
    s = cb.Scheduler(block_size=4, num_blocks=4, max_batch_tokens=8, max_requests_per_batch=2,
                     max_blocks_per_seq=2, safety_margin=0.0)
    with pytest.raises(cb.CBError):
        s.add_request(1, 8, 2)          # needs 3 blocks > max_blocks_per_seq
    s.add_request(1, 4, 2)
    with pytest.raises(cb.CBError):
        s.add_request(1, 4, 2)          # duplicate id
    with pytest.raises(cb.CBError) as e:
        s.step_done()                   # no open step
    assert e.value.status == cb.CB_ERR_STATE
    s.schedule_step()
    with pytest.raises(cb.CBError) as e:
        s.schedule_step()               # previous step not committed
    assert e.value.status == cb.CB_ERR_STATE
    s.step_done()


def test_kv_swap_argument_errors_without_gpu():
    import paged_attention_continuous_gb300 as cb
    lib = cb.library()
    assert lib.cb_kv_swap(None, None) == cb.CB_ERR_INVALID_ARG
    pools = (ctypes.c_void_p * 2)(256, 512)
    P = ctypes.POINTER(ctypes.c_void_p)
    pp = ctypes.cast(pools, P)
    # nothing to move: accepted without touching the GPU
    a = cb.cb_swap_args(0, None, None, 2, pp, pp, 4, 4, 4096, None)
    assert lib.cb_kv_swap(ctypes.byref(a), None) == cb.CB_OK
    a = cb.cb_swap_args(3, None, None, 0, None, None, 4, 4, 4096, None)
    assert lib.cb_kv_swap(ctypes.byref(a), None) == cb.CB_OK
    # too many pools, NULL ids, bad block size, bad capacity, misaligned pool
    a = cb.cb_swap_args(1, 16, 16, cb.SWAP_MAX_POOLS + 1, pp, pp, 4, 4, 4096, None)
    assert lib.cb_kv_swap(ctypes.byref(a), None) == cb.CB_ERR_INVALID_ARG
    a = cb.cb_swap_args(1, None, 16, 2, pp, pp, 4, 4, 4096, None)
    assert lib.cb_kv_swap(ctypes.byref(a), None) == cb.CB_ERR_INVALID_ARG
    a = cb.cb_swap_args(1, 16, 16, 2, pp, pp, 4, 4, 4100, None)
    assert lib.cb_kv_swap(ctypes.byref(a), None) == cb.CB_ERR_INVALID_ARG
    assert "multiple of 16" in lib.cb_last_error().decode()
    a = cb.cb_swap_args(1, 16, 16, 2, pp, pp, 0, 4, 4096, None)
    assert lib.cb_kv_swap(ctypes.byref(a), None) == cb.CB_ERR_INVALID_ARG
    bad = (ctypes.c_void_p * 2)(256, 520)
    a = cb.cb_swap_args(1, 16, 16, 2, pp, ctypes.cast(bad, P), 4, 4, 4096, None)
    assert lib.cb_kv_swap(ctypes.byref(a), None) == cb.CB_ERR_INVALID_ARG
    assert "aligned" in lib.cb_last_error().decode()
