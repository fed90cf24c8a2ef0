"""Run a workload step by step through the CUDA path (C scheduler + StepRunner)
and through the oracle (oracle scheduler + oracle append + oracle attention)
on the same seeded inputs, and compare.

Inputs: the paged pool's initial contents (context written before the
workload starts) and every step's q/k/v come from ``workloads`` generators,
drawn on the device.  The oracle never sees anything the CUDA kernels wrote:
it snapshots, from a pristine copy of the initial pool, the blocks its own
block tables reference, appends each step's new K/V itself, and attends with
its own scheduler's metadata.  To keep full-size cases cheap the oracle can
follow a sample of requests only; block ids are remapped into a compact
sub-pool (paging is invisible, which the oracle's own pins establish).
"""
from __future__ import annotations

import numpy as np
import torch

import workloads
from oracle import attention as oatt
from oracle import paged_kv
from tests.sched_driver import (add_waiting, c_from_config, load_scenario, normalize,
                                oracle_from_config, scenario_to_config)

TOL = {"f32": (1e-4, 0.0), "bf16": (2e-2, 1e-2)}


def tolerance_ok(gpu: np.ndarray, ref: np.ndarray, dtype: str):
    atol, rtol = TOL[dtype]
    err = np.abs(gpu - ref)
    bound = atol + rtol * np.abs(ref)
    return bool((err <= bound).all()), float(err.max(initial=0.0)), float((err - bound).max(initial=-1))


RUNNERS = ("eager", "graph", "pipelined", "native", "native_run")


class ParityRun:
    """``arrivals``: add each waiting request before the step numbered by its
    arrival_step (a trace), instead of all of them up front.

    ``runner`` picks the CUDA step path compared with the oracle: "eager"
    (StepRunner: upload + append + attention on the current stream),
    "graph" (GraphStepRunner: the step padded to its bucket and replayed
    from a CUDA graph) or "pipelined" (PipelinedStepRunner: inputs and
    output in pinned host memory, copied on their own streams), "native"
    (the C step executor, cb_executor_submit, on the C scheduler's step) or
    "native_run" (cb_executor_run_step: the executor itself schedules,
    submits and commits each step of the C scheduler)."""

    def __init__(self, sc, sample=None, device="cuda", fill_seed=1234, max_tokens=None,
                 arrivals=False, runner="eager"):
        from paged_attention_continuous_gb300.step import (GraphStepRunner,
                                                           PipelinedStepRunner, StepRunner)
        assert runner in RUNNERS, runner
        self.kind = runner
        self.sc = sc
        self.dtype = sc.dtype
        cfg = scenario_to_config(sc)
        self.o = oracle_from_config(cfg)
        self.c = c_from_config(cfg)
        self.arrivals = arrivals
        self.next_arrival = 0
        if arrivals:
            for sched in (self.o, self.c):
                for r in sc.running:
                    sched.add_running_request(r.req_id, r.prompt_len, r.output_len, r.num_cached)
        else:
            load_scenario(self.o, sc)
            load_scenario(self.c, sc)
        Runner = {"eager": StepRunner, "graph": GraphStepRunner, "pipelined": PipelinedStepRunner,
                  "native": StepRunner, "native_run": StepRunner}[runner]
        self.runner = Runner(num_blocks=sc.num_blocks, num_q_heads=sc.num_q_heads,
                                 num_kv_heads=sc.num_kv_heads, head_dim=sc.head_dim,
                                 dtype=sc.dtype, max_reqs=sc.max_requests_per_batch,
                                 max_tokens=max_tokens or sc.max_batch_tokens,
                                 max_blocks_per_seq=sc.max_blocks_per_seq,
                                 num_layers=sc.num_layers, device=device,
                                 swap_blocks=sc.swap_blocks, sliding_window=sc.sliding_window)
        self.device = device
        self.torch = torch
        self.ex = None
        if runner.startswith("native"):
            import paged_attention_continuous_gb300 as cb
            self.ex = cb.Executor(self.runner.k_cache, self.runner.v_cache,
                                  num_q_heads=sc.num_q_heads, max_reqs=sc.max_requests_per_batch,
                                  max_tokens=max_tokens or sc.max_batch_tokens,
                                  max_blocks_per_seq=self.c_width(),
                                  scale=self.runner.scale, sliding_window=sc.sliding_window)
        self.pristine = []
        for layer in range(sc.num_layers):
            kp = workloads.cache_fill(sc.num_blocks, sc.num_kv_heads, sc.block_size, sc.head_dim,
                                      seed=fill_seed + 2 * layer, dtype=sc.dtype,
                                      scale=sc.value_scale, device=device)
            vp = workloads.cache_fill(sc.num_blocks, sc.num_kv_heads, sc.block_size, sc.head_dim,
                                      seed=fill_seed + 2 * layer + 1, dtype=sc.dtype,
                                      scale=sc.value_scale, device=device)
            self.runner.k_cache[layer].copy_(kp)
            self.runner.v_cache[layer].copy_(vp)
            self.pristine.append((kp, vp))
        self.sample = None if sample is None else set(int(x) for x in sample)
        # oracle sub-pool: physical block -> compact index, per layer arrays
        self.idx = {}
        shape = (0, sc.num_kv_heads, sc.block_size, sc.head_dim)
        self.sub_k = [np.zeros(shape) for _ in range(sc.num_layers)]
        self.sub_v = [np.zeros(shape) for _ in range(sc.num_layers)]
        # oracle swap pool: slot -> (k rows, v rows) per layer, or None when
        # the block it came from was never followed
        self.oswap = {}
        self.swap_pairs = 0
        self.step_idx = 0

    def c_width(self):
        """Block-table width of the C scheduler's steps."""
        return int(self.runner.W)

    def _followed(self, rid):
        return self.sample is None or int(rid) in self.sample

    def _snapshot(self, blocks):
        new = [int(b) for b in blocks if int(b) >= 0 and int(b) not in self.idx]
        if not new:
            return
        base = len(self.idx)
        for i, b in enumerate(new):
            self.idx[b] = base + i
        sel = torch.tensor(new, dtype=torch.long, device=self.device)
        for layer, (kp, vp) in enumerate(self.pristine):
            k = kp.index_select(0, sel).double().cpu().numpy()
            v = vp.index_select(0, sel).double().cpu().numpy()
            self.sub_k[layer] = np.concatenate([self.sub_k[layer], k])
            self.sub_v[layer] = np.concatenate([self.sub_v[layer], v])

    def _mirror_swaps(self, st):
        """The oracle's side of a step's swaps, on its own sub-pool: swap-ins
        (slot -> block) first, then swap-outs (block -> slot)."""
        for slot, blk in st["swap_in"]:
            got = self.oswap.pop(int(slot), None)
            if got is None:
                continue
            self._snapshot([blk])
            i = self.idx[int(blk)]
            for layer, (k, v) in enumerate(got):
                self.sub_k[layer][i] = k
                self.sub_v[layer][i] = v
        for blk, slot in st["swap_out"]:
            i = self.idx.get(int(blk))
            self.oswap[int(slot)] = None if i is None else [
                (self.sub_k[layer][i].copy(), self.sub_v[layer][i].copy())
                for layer in range(self.sc.num_layers)]
        self.swap_pairs += len(st["swap_in"]) + len(st["swap_out"])

    def _gpu_step(self, sg, qkv):
        """Run one scheduled step through the chosen CUDA path; qkv[layer] =
        (q, k, v) on the device.  Returns the outputs per layer (device or
        pinned host tensors with the step's T rows)."""
        r = self.runner
        T = int(sg["num_tokens"])
        if self.kind == "eager":
            ds = r.upload(sg)
            return [r.run(ds, q, k, v, layer=layer) for layer, (q, k, v) in enumerate(qkv)]
        if self.kind == "graph":
            key, _ = r.prepare(sg)
            for layer, (q, k, v) in enumerate(qkv):
                r.q_buf[layer][:T].copy_(q)
                r.k_buf[layer][:T].copy_(k)
                r.v_buf[layer][:T].copy_(v)
            r.run(key)
            return [r.out_buf[layer][:T] for layer in range(len(qkv))]
        # the host paths: the step's inputs and output live in pinned host memory
        hq = [q.cpu().pin_memory() for q, _, _ in qkv]
        hk = [k.cpu().pin_memory() for _, k, _ in qkv]
        hv = [v.cpu().pin_memory() for _, _, v in qkv]
        ho = [self.torch.empty(q.shape, dtype=q.dtype, pin_memory=True) for q, _, _ in qkv]
        if self.kind == "native":
            self.ex.submit(sg, hq, hk, hv, ho)
            self.ex.synchronize()
            return ho
        if self.kind == "native_run":
            n, _ = self.ex.run_step(self.c, hq, hk, hv, ho)
            assert n == T, (n, T)
            self.ex.synchronize()
            return ho
        r.submit(sg, hq, hk, hv, ho).synchronize()
        return ho

    def _gpu_no_batch(self, sg):
        """A step that found no batch may still carry swaps: queue them where
        the chosen runner queues its kernels."""
        if self.kind == "pipelined":
            with self.torch.cuda.stream(self.runner.compute_stream):
                self.runner.apply_swaps(sg)
            return
        if self.kind == "native_run":
            assert self.c.schedule_step()["status"] == sg["status"]
            return
        self.runner.apply_swaps(sg)

    def step(self, check=True):
        """One step on both sides.  Returns (status, gpu_out[layer] as float64
        numpy for followed rows, oracle_out[layer], followed token indices).
        With check=False the oracle appends the followed rows' K/V but skips
        attention (and nothing is compared): (status, None, None, toks)."""
        sc = self.sc
        if self.arrivals:
            while (self.next_arrival < len(sc.waiting) and
                   sc.waiting[self.next_arrival].arrival_step <= self.step_idx):
                w = sc.waiting[self.next_arrival]
                add_waiting(self.o, w)
                add_waiting(self.c, w)
                self.next_arrival += 1
        so = self.o.schedule_step()
        if self.kind == "native_run":
            sg = so     # the executor schedules the C scheduler's step itself
        else:
            sg = self.c.schedule_step()
            assert normalize(so) == normalize(sg), "schedulers disagree"
        self.last = so
        self._mirror_swaps(so)
        if so["status"] != 0:
            self._gpu_no_batch(sg)
            self.step_idx += 1
            return so["status"], None, None, None
        T = so["num_tokens"]
        rows = [i for i, rid in enumerate(so["req_ids"]) if self._followed(rid)]
        toks = np.concatenate([np.arange(so["cu_seqlens_q"][i], so["cu_seqlens_q"][i + 1])
                               for i in rows]) if rows else np.zeros(0, dtype=np.int64)
        for i in rows:
            self._snapshot(so["block_tables"][i])
        gpu_outs, ref_outs = [], []
        bs = sc.block_size
        qkv, oin = [], []
        sel = torch.as_tensor(toks, dtype=torch.long, device=self.device)
        for layer in range(sc.num_layers):
            seeds = [workloads.step_seed(sc.seed, self.step_idx, layer, w) for w in range(3)]
            q = workloads.token_tensors(T, sc.num_q_heads, sc.head_dim, seed=seeds[0], dtype=sc.dtype,
                                        scale=sc.value_scale, device=self.device)
            k = workloads.token_tensors(T, sc.num_kv_heads, sc.head_dim, seed=seeds[1], dtype=sc.dtype,
                                        scale=sc.value_scale, device=self.device)
            v = workloads.token_tensors(T, sc.num_kv_heads, sc.head_dim, seed=seeds[2], dtype=sc.dtype,
                                        scale=sc.value_scale, device=self.device)
            qkv.append((q, k, v))
            # oracle inputs (copies of the generator's output, before any kernel runs)
            oin.append((q.index_select(0, sel).double().cpu().numpy(),
                        k.index_select(0, sel).double().cpu().numpy(),
                        v.index_select(0, sel).double().cpu().numpy()))
        outs = self._gpu_step(sg, qkv)
        for layer in range(sc.num_layers):
            qo, ko, vo = oin[layer]
            if check:
                o = outs[layer]
                gpu_outs.append(o.index_select(0, sel.to(o.device)).double().cpu().numpy())
            # oracle: append followed rows' tokens into the sub-pool, then attend
            slots = []
            for t in toks:
                s = int(so["slot_mapping"][t])
                slots.append(self.idx[s // bs] * bs + s % bs)
            paged_kv.append(self.sub_k[layer], self.sub_v[layer], ko, vo,
                            np.asarray(slots, dtype=np.int64), bs)
            if not check:
                continue
            cu = [0]
            for i in rows:
                cu.append(cu[-1] + int(so["cu_seqlens_q"][i + 1] - so["cu_seqlens_q"][i]))
            bt = np.full((len(rows), so["block_tables"].shape[1]), -1, dtype=np.int64)
            for j, i in enumerate(rows):
                for c, b in enumerate(so["block_tables"][i]):
                    if b >= 0:
                        bt[j, c] = self.idx[int(b)]
            ref = oatt.paged_attention(qo, self.sub_k[layer], self.sub_v[layer], np.asarray(cu),
                                       so["seq_lens"][rows], bt, bs, sc.softmax_scale,
                                       window=sc.sliding_window)
            ref_outs.append(ref)
        if self.kind == "native_run":
            self.o.step_done()      # the executor committed the C scheduler's step
        else:
            assert self.o.step_done() == self.c.step_done()
        if self.kind == "pipelined":
            self.runner.synchronize()
        errs = self.ex.read_errors() if self.ex is not None else self.runner.workspace.read_errors()
        assert errs == 0, f"device error bits {errs:#x}"
        if self.runner.swap is not None:
            errs = self.runner.swap.read_errors()
            assert errs == 0, f"swap error bits {errs:#x}"
        self.step_idx += 1
        if not check:
            return 0, None, None, toks
        return 0, gpu_outs, ref_outs, toks
