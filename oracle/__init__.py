"""CPU oracle for the continuous-batching paged-attention step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
this package.  The product path (``paged_attention_continuous_gb300``) never
imports it and shares no code with it.

Contents (plain, slow, fp64 where floating point is involved):

* ``scheduler.FifoScheduler`` -- the FIFO continuous-batching scheduler of
  *Continuous batching architecture* (sections "Request lifecycle",
  "Chunked prefill", "Scheduler", "FIFO", "Admission") and the iteration loop
  of *vLLM serving internals* (section "What the scheduler looks like"),
  with paged blocks as in *vLLM serving internals* ("PagedAttention as a
  virtual memory system").
* ``paged_kv.append`` -- writes a step's new K/V into the paged cache
  through the slot mapping.
* ``attention.paged_attention`` -- per-request causal attention over
  absolute positions, reading K/V through block tables (*Chunked Prefill*,
  Ultralytics glossary, section "How chunked prefill works").
* ``attention.dense_causal_attention`` -- the one-shot definition the
  chunked/paged computation must reproduce.

Parity status of each function is stated in its module header.
"""
from . import scheduler, paged_kv, attention  # noqa: F401
