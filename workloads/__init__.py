"""Seeded synthetic inputs for the continuous-batching attention step.

This module is the only code shared by the CPU oracle (``oracle/``) and the
CUDA path (``paged_attention_continuous_gb300``).  It draws random numbers and
describes workloads (request lengths, states, pool sizes, budgets); it holds
none of the method's arithmetic: no slot computation, no block accounting,
no attention.

Workload shapes follow the pages' serving scenarios:

* ``chunked_prefill_1000`` -- the worked example of *Chunked Prefill*
  (Ultralytics glossary, section "How chunked prefill works"): one layer,
  8 heads of 64 dims, a 1000-token prompt drawn with ``torch.manual_seed(0)``
  as ``torch.randn(3, 1, 8, 1000, 64)``, prefilled in 256-token chunks.
* ``decode_64`` -- a decode-only step: 64 requests, contexts U[128, 4096],
  32 query / 8 KV heads, head_dim 128, a 20,000-block pool.
* ``mixed_2048`` -- a mixed chunked-prefill step under the FIFO policy
  (*Continuous batching architecture*, section "Scheduler"/"FIFO"): 96 decodes
  with contexts U[256, 8192], one prefill in flight on its second chunk
  (prompt 3000, 1024 cached), new prompts U[64, 1024] filling the budget.
* ``long_prompt_32k`` -- a 32,768-token prompt prefilled in 512-token chunks
  (*vLLM serving internals*, section "Chunked prefill protects TTFT tail")
  while 128 requests decode, 64 query / 8 KV heads.
* ``trace_2000`` -- 2,000 requests, Poisson arrivals (mean 20 per step),
  lognormal prompt/output lengths, 4 stacked layers.

A ``Scenario`` lists scheduler settings and the requests to load: requests
already in flight (``running``: prompt length, output length, tokens already
in the cache) and requests arriving in order (``waiting``).  Both the oracle
scheduler and the C scheduler are driven from the same ``Scenario``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Tuple

import numpy as np

BLOCK_SIZE = 16
# output length of requests that keep decoding through a benchmark
LONG_OUTPUT = 1024


@dataclasses.dataclass
class RunningRequest:
    req_id: int
    prompt_len: int
    output_len: int
    num_cached: int          # tokens whose K/V is already in the paged cache


@dataclasses.dataclass
class WaitingRequest:
    req_id: int
    prompt_len: int
    output_len: int
    arrival_step: int = 0    # step at which the request joins the queue
    tokens: Optional[np.ndarray] = None  # synthetic prompt token ids (prefix caching)


@dataclasses.dataclass
class Scenario:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: str                       # "f32" or "bf16"
    num_blocks: int
    max_batch_tokens: int
    max_requests_per_batch: int
    max_prefill_chunk: int           # 0 = no per-request chunk cap
    safety_margin: float
    max_blocks_per_seq: int          # raised to fit the longest request
    free_list: np.ndarray            # int32 permutation of range(num_blocks)
    running: List[RunningRequest]
    waiting: List[WaitingRequest]
    num_layers: int = 1
    value_scale: float = 1.0         # q/k/v ~ value_scale * N(0, 1)
    seed: int = 0
    block_size: int = BLOCK_SIZE
    policy: int = 0                  # 0 FIFO, 1 PrefillFirst
    offload: bool = False            # offload requests when blocks run out
    swap_blocks: int = 0             # CPU swap pool capacity in blocks
    prefix_caching: bool = False     # share blocks of equal prompt prefixes
    sliding_window: int = 0          # > 0: every layer attends the last W tokens

    def __post_init__(self):
        longest = max([r.prompt_len + r.output_len - 1 for r in self.running]
                      + [r.prompt_len + r.output_len - 1 for r in self.waiting]
                      + [1])
        need = -(-longest // self.block_size)
        self.max_blocks_per_seq = max(int(self.max_blocks_per_seq), need)

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


def permuted_free_list(num_blocks: int, seed: int) -> np.ndarray:
    """A seeded random permutation of the physical block ids."""
    rng = np.random.default_rng(seed)
    return rng.permutation(num_blocks).astype(np.int32)


def margin_as_float32(m: float) -> float:
    """The safety margin as the C ABI stores it (an IEEE float32)."""
    return float(np.float32(m))


# ---------------------------------------------------------------- scenarios
def chunked_prefill_1000(chunk: int = 256, num_blocks: int = 64,
                         permute: bool = True, seed: int = 0) -> Scenario:
    fl = permuted_free_list(num_blocks, seed + 1) if permute else \
        np.arange(num_blocks, dtype=np.int32)
    return Scenario(
        name="chunked_prefill_1000", num_q_heads=8, num_kv_heads=8,
        head_dim=64, dtype="f32", num_blocks=num_blocks,
        max_batch_tokens=chunk, max_requests_per_batch=8,
        max_prefill_chunk=0, safety_margin=0.0, max_blocks_per_seq=0,
        free_list=fl, running=[],
        waiting=[WaitingRequest(req_id=0, prompt_len=1000, output_len=1)],
        value_scale=1.0, seed=seed)


def decode_64(seed: int = 0, num_reqs: int = 64, lo: int = 128,
              hi: int = 4096, num_blocks: int = 20000) -> Scenario:
    rng = np.random.default_rng(seed)
    ctx = rng.integers(lo, hi, size=num_reqs, endpoint=True)
    running = []
    for i, c in enumerate(ctx):
        c = int(c)
        # context c = seq_len of this step, the newest token not yet cached
        running.append(RunningRequest(req_id=i, prompt_len=c - 1,
                                      output_len=LONG_OUTPUT, num_cached=c - 1))
    return Scenario(
        name="decode_64", num_q_heads=32, num_kv_heads=8, head_dim=128,
        dtype="bf16", num_blocks=num_blocks, max_batch_tokens=max(num_reqs, 1),
        max_requests_per_batch=max(num_reqs, 1), max_prefill_chunk=0,
        safety_margin=0.0, max_blocks_per_seq=0,
        free_list=permuted_free_list(num_blocks, seed + 1), running=running,
        waiting=[], value_scale=0.5, seed=seed)


def mixed_2048(seed: int = 0, num_decodes: int = 96,
               num_waiting: int = 24, num_blocks: int = 65536) -> Scenario:
    rng = np.random.default_rng(seed)
    ctx = rng.integers(256, 8192, size=num_decodes, endpoint=True)
    running = [RunningRequest(req_id=i, prompt_len=int(c) - 1,
                              output_len=LONG_OUTPUT, num_cached=int(c) - 1)
               for i, c in enumerate(ctx)]
    running.append(RunningRequest(req_id=num_decodes, prompt_len=3000,
                                  output_len=LONG_OUTPUT, num_cached=1024))
    plen = rng.integers(64, 1024, size=num_waiting, endpoint=True)
    waiting = [WaitingRequest(req_id=num_decodes + 1 + i,
                              prompt_len=int(p), output_len=LONG_OUTPUT)
               for i, p in enumerate(plen)]
    return Scenario(
        name="mixed_2048", num_q_heads=32, num_kv_heads=8, head_dim=128,
        dtype="bf16", num_blocks=num_blocks, max_batch_tokens=2048,
        max_requests_per_batch=128, max_prefill_chunk=1024,
        safety_margin=0.15, max_blocks_per_seq=0,
        free_list=permuted_free_list(num_blocks, seed + 1), running=running,
        waiting=waiting, value_scale=0.5, seed=seed)


def long_prompt_32k(seed: int = 0, num_decodes: int = 128,
                    prompt_len: int = 32768, num_blocks: int = 65536) -> Scenario:
    rng = np.random.default_rng(seed)
    ctx = rng.integers(512, 8192, size=num_decodes, endpoint=True)
    running = [RunningRequest(req_id=i, prompt_len=int(c) - 1,
                              output_len=LONG_OUTPUT, num_cached=int(c) - 1)
               for i, c in enumerate(ctx)]
    waiting = [WaitingRequest(req_id=num_decodes, prompt_len=prompt_len,
                              output_len=LONG_OUTPUT)]
    return Scenario(
        name="long_prompt_32k", num_q_heads=64, num_kv_heads=8, head_dim=128,
        dtype="bf16", num_blocks=num_blocks, max_batch_tokens=num_decodes + 512,
        max_requests_per_batch=256, max_prefill_chunk=0, safety_margin=0.15,
        max_blocks_per_seq=0,
        free_list=permuted_free_list(num_blocks, seed + 1), running=running,
        waiting=waiting, value_scale=0.5, seed=seed)


def trace_2000(seed: int = 0, num_requests: int = 2000,
               mean_arrivals: float = 20.0, num_blocks: int = 65536) -> Scenario:
    """Poisson arrivals; prompt ~ lognormal(ln 512, 1) clipped [16, 16384],
    output ~ lognormal(ln 128, 1) clipped [1, 2048] (sigma = 1 for both)."""
    rng = np.random.default_rng(seed)
    waiting: List[WaitingRequest] = []
    step = 0
    while len(waiting) < num_requests:
        n = int(rng.poisson(mean_arrivals))
        for _ in range(n):
            if len(waiting) >= num_requests:
                break
            p = int(np.clip(np.rint(rng.lognormal(math.log(512.0), 1.0)), 16, 16384))
            o = int(np.clip(np.rint(rng.lognormal(math.log(128.0), 1.0)), 1, 2048))
            waiting.append(WaitingRequest(req_id=len(waiting), prompt_len=p,
                                          output_len=o, arrival_step=step))
        step += 1
    return Scenario(
        name="trace_2000", num_q_heads=32, num_kv_heads=8, head_dim=128,
        dtype="bf16", num_blocks=num_blocks, max_batch_tokens=8192,
        max_requests_per_batch=256, max_prefill_chunk=0, safety_margin=0.15,
        max_blocks_per_seq=0,
        free_list=permuted_free_list(num_blocks, seed + 1), running=[],
        waiting=waiting, num_layers=4, value_scale=1.0, seed=seed)


def prefill_chunk_16k(seed: int = 0, chunk: int = 512, offset: int = 16384,
                      num_blocks: int = 4096) -> Scenario:
    """One 512-token prefill chunk of a 32K prompt at absolute offset 16,384
    (a mid-prompt step of the long-prompt interleave), 64 Q / 8 KV heads."""
    running = [RunningRequest(req_id=0, prompt_len=32768, output_len=LONG_OUTPUT,
                              num_cached=offset)]
    return Scenario(
        name="prefill_chunk_16k", num_q_heads=64, num_kv_heads=8, head_dim=128,
        dtype="bf16", num_blocks=num_blocks, max_batch_tokens=chunk,
        max_requests_per_batch=8, max_prefill_chunk=0, safety_margin=0.0,
        max_blocks_per_seq=0, free_list=permuted_free_list(num_blocks, seed + 1),
        running=running, waiting=[], value_scale=0.5, seed=seed)


def offload_pressure(seed: int = 0, num_requests: int = 24, num_blocks: int = 40,
                     swap_blocks: int = 8, num_layers: int = 2) -> Scenario:
    """A KV pool too small for the requests it admits, with offloading on:
    requests arrive over the first steps (prompts 24-160, outputs 16-96
    tokens), the pool holds 640 tokens, so decodes outgrow it and requests
    are moved to an 8-block CPU swap pool, or soft-reset when it is full, and
    later resumed (seeds 0-3: 160-560 block swaps and 6-9 soft resets over
    about 350 steps).  Each request alone fits the pool."""
    rng = np.random.default_rng(seed)
    waiting = []
    for i in range(num_requests):
        waiting.append(WaitingRequest(req_id=i, prompt_len=int(rng.integers(24, 160, endpoint=True)),
                                      output_len=int(rng.integers(16, 96, endpoint=True)),
                                      arrival_step=int(rng.integers(0, 12))))
    waiting.sort(key=lambda w: w.arrival_step)
    return Scenario(
        name="offload_pressure", num_q_heads=16, num_kv_heads=4, head_dim=128,
        dtype="bf16", num_blocks=num_blocks, max_batch_tokens=256,
        max_requests_per_batch=16, max_prefill_chunk=0, safety_margin=0.0,
        max_blocks_per_seq=0, free_list=permuted_free_list(num_blocks, seed + 1),
        running=[], waiting=waiting, num_layers=num_layers, value_scale=1.0, seed=seed,
        offload=True, swap_blocks=swap_blocks)


def shared_prefix(seed: int = 0, num_requests: int = 48, num_system: int = 4,
                  num_blocks: int = 4096, num_layers: int = 2) -> Scenario:
    """Requests that share long prompt prefixes (a few "system prompts"),
    for prefix caching: 4 system prompts of U[200, 1200] synthetic token ids
    (vocabulary 32,000), each request one of them plus its own U[16, 400]
    suffix, outputs U[8, 64]; arrivals over the first 16 steps; 32 Q / 8 KV
    heads, D = 128, bf16, budget 2048 tokens."""
    rng = np.random.default_rng(seed)
    systems = [rng.integers(0, 32000, size=int(rng.integers(200, 1200, endpoint=True)))
               for _ in range(num_system)]
    waiting = []
    for i in range(num_requests):
        sysp = systems[int(rng.integers(0, num_system))]
        toks = np.concatenate([sysp, rng.integers(0, 32000, size=int(rng.integers(16, 400,
                                                                                 endpoint=True)))])
        waiting.append(WaitingRequest(req_id=i, prompt_len=int(len(toks)),
                                      output_len=int(rng.integers(8, 64, endpoint=True)),
                                      arrival_step=int(rng.integers(0, 16)),
                                      tokens=toks.astype(np.int32)))
    waiting.sort(key=lambda w: w.arrival_step)
    return Scenario(
        name="shared_prefix", num_q_heads=32, num_kv_heads=8, head_dim=128,
        dtype="bf16", num_blocks=num_blocks, max_batch_tokens=2048,
        max_requests_per_batch=64, max_prefill_chunk=0, safety_margin=0.0,
        max_blocks_per_seq=0, free_list=permuted_free_list(num_blocks, seed + 1),
        running=[], waiting=waiting, num_layers=num_layers, value_scale=1.0, seed=seed,
        prefix_caching=True)


def sliding_trace(seed: int = 0, num_requests: int = 32, window: int = 384,
                  num_blocks: int = 512, num_layers: int = 2) -> Scenario:
    """A model whose layers all use a sliding window of 384 tokens: prompts
    U[64, 1500], outputs U[8, 200], arrivals over the first 10 steps, 32 Q /
    8 KV heads, D = 128, bf16, budget 1024 tokens, a 512-block pool (8,192
    tokens) that only fits the traffic because pages out of the window are
    recycled."""
    rng = np.random.default_rng(seed)
    waiting = [WaitingRequest(req_id=i, prompt_len=int(rng.integers(64, 1500, endpoint=True)),
                              output_len=int(rng.integers(8, 200, endpoint=True)),
                              arrival_step=int(rng.integers(0, 10)))
               for i in range(num_requests)]
    waiting.sort(key=lambda w: w.arrival_step)
    return Scenario(
        name="sliding_trace", num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
        num_blocks=num_blocks, max_batch_tokens=1024, max_requests_per_batch=32,
        max_prefill_chunk=0, safety_margin=0.0, max_blocks_per_seq=0,
        free_list=permuted_free_list(num_blocks, seed + 1), running=[], waiting=waiting,
        num_layers=num_layers, value_scale=1.0, seed=seed, sliding_window=window)


SCENARIOS = {
    "chunked_prefill_1000": chunked_prefill_1000,
    "decode_64": decode_64,
    "mixed_2048": mixed_2048,
    "long_prompt_32k": long_prompt_32k,
    "trace_2000": trace_2000,
    "prefill_chunk_16k": prefill_chunk_16k,
    "offload_pressure": offload_pressure,
    "shared_prefix": shared_prefix,
    "sliding_trace": sliding_trace,
}


# ------------------------------------------------------------ tensor inputs
def worked_example_qkv():
    """q, k, v of the chunked-prefill worked example: seed 0,
    ``torch.randn(3, 1, 8, 1000, 64)`` split along the first axis.
    Returns three float32 CPU tensors of shape [1, 8, 1000, 64]."""
    import torch
    torch.manual_seed(0)
    q, k, v = torch.randn(3, 1, 8, 1000, 64).unbind(0)
    return q, k, v


def _torch_dtype(dtype: str):
    import torch
    return {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]


def token_tensors(num_tokens: int, num_heads: int, head_dim: int, *,
                  seed: int, dtype: str = "bf16", scale: float = 1.0,
                  device: str = "cpu"):
    """A [num_tokens, num_heads, head_dim] tensor ~ scale * N(0, 1), drawn in
    float32 from a seeded generator on ``device`` and rounded (to nearest
    even) to ``dtype``.  The same (seed, device) always gives the same
    values."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(num_tokens, num_heads, head_dim, generator=g,
                    dtype=torch.float32, device=device)
    if scale != 1.0:
        x = x * scale
    return x.to(_torch_dtype(dtype))


def step_seed(base: int, step: int, layer: int, which: int) -> int:
    """Seed for the q/k/v (which = 0/1/2) of one step and layer; a pure
    function of its arguments, so any step can be regenerated alone."""
    return (int(base) * 1_000_003 + step * 4099 + layer * 17 + which) & 0x7FFFFFFF


def cache_fill(num_blocks: int, num_kv_heads: int, block_size: int,
               head_dim: int, *, seed: int, dtype: str = "bf16",
               scale: float = 1.0, device: str = "cpu"):
    """Random contents for a whole K (or V) pool [num_blocks, Hkv, bs, D],
    standing in for KV written by earlier steps."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(num_blocks, num_kv_heads, block_size, head_dim,
                    generator=g, dtype=torch.float32, device=device)
    if scale != 1.0:
        x = x * scale
    return x.to(_torch_dtype(dtype))
