"""Oracle FIFO scheduler (TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__``).

Follows:

* *Continuous batching architecture* (HF Transformers docs), "Request
  lifecycle": PENDING -> PREFILLING -> DECODING -> FINISHED, one output token
  per decode step.
* same page, "Chunked prefill": a prompt larger than the remaining token
  budget (``max_batch_tokens``) is processed as far as the budget allows and
  resumed next step from where it stopped.
* same page, "Scheduler": token budget, cache budget (free KV pages) and the
  request cap ``max_requests_per_batch``.
* same page, "FIFO": active decodes first, then active prefills, then new
  waiting requests in arrival order.
* same page, "Admission": a request joins only if every allocator has room;
  otherwise nothing is allocated.  ``safety_margin`` (FIFO default 0.15)
  holds new prefills back when free capacity would fall below the margin.
* same page, "Offloading": active requests that fail to get the blocks they
  need are reported as stalled, with their block demand.
* *vLLM serving internals*, "PagedAttention as a virtual memory system":
  fixed 16-token blocks, a per-sequence block table from logical to physical
  block, one more block when a sequence outgrows its last one, blocks back to
  the pool when the sequence finishes; "What the scheduler looks like":
  release finished, admit waiting while blocks allow, one batch per
  iteration.
* *Chunked Prefill* (Ultralytics glossary), "How chunked prefill works": one
  token per running decode first, then chunks of waiting prompts fill the
  remaining budget.
* *Continuous batching architecture*, "PrefillFirst": chunked prefills are
  completed before decoding resumes (policy PREFILL_FIRST).
* *Continuous batching architecture*, "Offloading" and "Soft reset": when
  requests stall, the fewest of them are offloaded, newest first, never the
  last active request -- to a CPU swap pool when it has room (resumed later
  without recomputation), else by a soft reset (generated tokens appended
  to the prompt, blocks freed, back to the queue).  Two triggers: a batch
  was scheduled but requests stalled (offload enough stalled requests for
  the rest); no batch fits at all (offload and retry within the step).
* *Continuous batching architecture*, "Prefix caching" and "Eviction": a
  content key per complete block; a later request whose prompt starts with
  the same blocks reuses them and skips their prefill; shared blocks are
  reference-counted and return to the pool when the last user finishes;
  freed blocks keep their content and key ("initialized") so later requests
  can still match them, and when uninitialized blocks run out the newest
  initialized ones are demoted (key dropped) and reused.
* *Continuous batching architecture*, Memory management (sliding
  attention): sliding-window layers keep only a fixed window of recent
  tokens by recycling a small set of pages, and do not share blocks.
* vLLM performance-series post (page 5), "Request-parallel prefill": several
  requests may prefill in one batch, but only a limited number of LONG
  prompts at a time, so short prompts are not held behind a long one.

Readings where the pages leave a step open:

1. Batch order = decodes (admission order), active prefills (admission
   order), newly admitted prompts (arrival order).
2. Admission of waiting requests is strict head-of-line: the first waiting
   request that does not fit (budget, request cap, blocks or margin) stops
   admission for this step.
3. A prefill chunk takes min(remaining prompt, remaining budget,
   max_prefill_chunk) tokens (max_prefill_chunk = 0 means no cap).
4. Blocks are allocated only for the tokens scheduled this step, all or
   nothing per request.  The free list is a FIFO queue: allocation pops from
   its head, freed blocks are pushed to its tail (finished requests in batch
   order, each block table in logical order).
5. The safety margin applies to admitting new requests only:
   admit iff free_after >= ceil(margin * num_blocks), margin taken as an
   IEEE float32 and the product computed in double precision.
6. Decodes or prefills past the token budget or the request cap simply wait;
   an active request whose blocks cannot be allocated is "stalled" and
   reported with its demand.  A step that schedules nothing while requests
   are stalled or waiting returns status NO_BLOCKS.
7. The step that completes a prompt yields output token 1; each decode step
   yields one more; a request with output_len n finishes after n-1 decode
   steps.  A decode step's query token sits at position num_cached and its
   K/V is appended in the same step.
8. slot = block_table[pos // block_size] * block_size + pos % block_size.
9. PREFILL_FIRST takes the same three groups in the order running prefills,
   new prompts, decodes (the decodes get what budget and request cap are
   left; blocks are taken in that order); the emitted rows stay decodes
   first (the attention call's layout), then running prefills, then new
   prompts.
10. ``max_prefill_reqs`` (0 = none) caps the prefill rows (running + new)
   of a step.  A prompt is long when prompt_len > ``long_prefill_tokens``
   (0 = no long cap); a long waiting request is admitted only while fewer
   than ``max_long_prefills`` long requests are in their prefill phase, and
   one held by that cap is skipped (keeps its place) instead of blocking
   the requests behind it.
11. Offloading (``offload=True``): swapped requests are resumed at the start
   of a step, oldest offload first, head-of-line, when free blocks minus
   their blocks stay >= the safety reserve; they rejoin the running list at
   its end and are not chosen as victims in that step.  "Newest" = latest
   in the running (admission) list.  A victim goes to the swap pool iff its
   free slots hold all its blocks (slots from a FIFO queue, freed to its
   tail); otherwise it is soft-reset: prompt_len += num_generated,
   output_len -= num_generated, nothing cached, put at the FRONT of the
   waiting queue.  Trigger 2 retries the whole schedule after each victim.
   The step reports the copies to make before its kernels: swap-ins
   (slot -> new block) first, then swap-outs (block -> slot).
12. Prefix caching (``prefix_caching=True``; only requests given prompt
   token ids take part): a block's key is the whole token prefix up to its
   end (so a block matches only after every block before it matched), for
   blocks fully inside the known prompt tokens.  At admission the longest
   leading run of cached keys is reused, capped so at least one prompt token
   is computed (the step that completes the prompt yields the first output
   token); the reused tokens count as cached and take no budget.  Reused
   blocks with no other user leave the free pool, so admission needs
   free - reused_free - new >= reserve.  A block is keyed at the step_done
   that completes it, unless its key is already held by another block.  A
   freed block whose count drops to 0 goes to the initialized pool (freed
   order) if keyed, else to the tail of the free queue.  Allocation pops the
   free queue; when it is empty it demotes the NEWEST initialized block.
   Free capacity = free queue + initialized pool.  Offloaded or reset
   requests release their blocks the same way; blocks swapped back in are
   new private blocks.

13. Sliding window (``sliding_window`` = W > 0; the whole pool serves
   sliding layers -- a model mixing full and sliding layers would need a
   second pool): a query at position p reads keys p-W+1 .. p, so once a
   request has num_cached tokens, its pages whose last position is below
   num_cached - W + 1 are never read again.  At step_done, after the state
   updates, such pages of every request of the batch that did not finish
   are freed (batch order, then logical order) to the free queue's tail and
   their table entries become -1; then finished requests release their
   remaining pages.  Block demand still counts table entries (dropped ones
   included), so a request holds at most ceil((W - 1) / bs) + 1 pages
   plus its next chunk.  Only live pages are swapped out (and back in, to new
   blocks at the same table positions).  Prefix caching is refused with a
   window (sliding layers do not share blocks).

14. Fault injection (not on the pages; a test hook for memory pressure):
   hold_blocks(n) takes up to n blocks out of the allocatable pool exactly
   as allocation would (free queue head first, then the newest
   initialized blocks, demoted), between steps; release_blocks(ids) puts
   them back at the free queue's tail in the given order.

Parity: pinned by hand-derived traces (tests/golden/scheduler_*.json) and by
invariants (budget, cap, FIFO order, block conservation, all-or-nothing
admission); the full batch composition beyond the pages' rules rests on the
readings above ("parity unpinned" beyond those pins).
"""
from __future__ import annotations

import collections
import math
from typing import Dict, List, Optional, Sequence

import numpy as np

WAITING, PREFILLING, DECODING, FINISHED = "waiting", "prefilling", "decoding", "finished"
SWAPPED = "swapped"

STATUS_OK = 0
STATUS_NO_BLOCKS = 2
POLICY_FIFO, POLICY_PREFILL_FIRST = 0, 1


class Request:
    def __init__(self, req_id: int, prompt_len: int, output_len: int):
        self.req_id = int(req_id)
        self.prompt_len = int(prompt_len)
        self.output_len = int(output_len)
        self.num_cached = 0       # tokens whose K/V is in the cache
        self.num_generated = 0    # output tokens produced so far
        self.blocks: List[int] = []
        self.state = WAITING
        self.swap_slots: List[int] = []
        self.swapped_table: List[bool] = []   # while swapped: live entries
        self.resume_state = None
        self.tokens = None        # known prompt token ids (prefix caching)
        self.num_registered = 0   # leading blocks already considered for keys


class FifoScheduler:
    def __init__(self, *, block_size: int, num_blocks: int,
                 max_batch_tokens: int, max_requests_per_batch: int,
                 max_blocks_per_seq: int, max_prefill_chunk: int = 0,
                 safety_margin: float = 0.15,
                 free_list: Optional[Sequence[int]] = None,
                 policy: int = POLICY_FIFO, max_prefill_reqs: int = 0,
                 long_prefill_tokens: int = 0, max_long_prefills: int = 1,
                 offload: bool = False, swap_blocks: int = 0,
                 prefix_caching: bool = False, sliding_window: int = 0):
        self.block_size = int(block_size)
        self.num_blocks = int(num_blocks)
        self.max_batch_tokens = int(max_batch_tokens)
        self.max_requests_per_batch = int(max_requests_per_batch)
        self.max_blocks_per_seq = int(max_blocks_per_seq)
        self.max_prefill_chunk = int(max_prefill_chunk)
        self.policy = int(policy)
        self.max_prefill_reqs = int(max_prefill_reqs)
        self.long_prefill_tokens = int(long_prefill_tokens)
        self.max_long_prefills = int(max_long_prefills)
        self.offload = bool(offload)
        self.swap_free = collections.deque(range(int(swap_blocks)))
        self.swapped: List[Request] = []
        margin32 = float(np.float32(safety_margin))
        self.reserved_blocks = int(math.ceil(margin32 * float(self.num_blocks)))
        if free_list is None:
            free_list = range(self.num_blocks)
        self.free = collections.deque(int(b) for b in free_list)
        # prefix caching: reference counts of blocks in use, keyed blocks
        # (key = token prefix up to the block's end) and the initialized pool
        self.prefix_caching = bool(prefix_caching)
        self.sliding_window = int(sliding_window)
        if self.sliding_window < 0:
            raise ValueError("sliding_window must be >= 0")
        if self.sliding_window and self.prefix_caching:
            raise ValueError("sliding-window layers do not share blocks")
        self.refs: Dict[int, int] = {}
        self.cache_index: Dict[tuple, int] = {}
        self.block_key: Dict[int, tuple] = {}
        self.free_init: List[int] = []
        self.prefix_hit_tokens = 0
        self.held: List[int] = []   # blocks taken out by hold_blocks
        self.waiting: collections.deque = collections.deque()
        self.running: List[Request] = []
        self.requests: Dict[int, Request] = {}
        self._pending = None      # list of (request, num_tokens) of the open step

    # ------------------------------------------------------------ requests
    def _blocks_for(self, num_tokens: int) -> int:
        return -(-num_tokens // self.block_size)

    def add_request(self, req_id: int, prompt_len: int, output_len: int,
                    tokens: Optional[Sequence[int]] = None) -> None:
        """``tokens``: ids of the first len(tokens) <= prompt_len prompt
        tokens (for prefix caching), or None."""
        if req_id in self.requests or prompt_len < 1 or output_len < 1:
            raise ValueError("bad request")
        if self._blocks_for(prompt_len + output_len - 1) > self.max_blocks_per_seq:
            raise ValueError("request longer than max_blocks_per_seq blocks")
        if tokens is not None and len(tokens) > prompt_len:
            raise ValueError("more tokens than prompt_len")
        r = Request(req_id, prompt_len, output_len)
        if tokens is not None:
            r.tokens = tuple(int(t) for t in tokens)
        self.requests[r.req_id] = r
        self.waiting.append(r)

    # ------------------------------------------------------- block pool
    def _num_free(self) -> int:
        return len(self.free) + len(self.free_init)

    def _alloc(self) -> int:
        if self.free:
            b = self.free.popleft()
        else:
            b = self.free_init.pop()          # demote the newest initialized block
            del self.cache_index[self.block_key.pop(b)]
        self.refs[b] = 1
        return b

    def _release(self, r) -> None:
        for b in r.blocks:
            if b < 0:
                continue                      # dropped out of the window
            self.refs[b] -= 1
            if self.refs[b] == 0:
                del self.refs[b]
                if b in self.block_key:
                    self.free_init.append(b)
                else:
                    self.free.append(b)
        r.blocks = []
        r.num_registered = 0

    def _match(self, r) -> List[int]:
        """Blocks of the longest leading run of r's prompt already cached."""
        if not self.prefix_caching or r.tokens is None:
            return []
        limit = min(len(r.tokens), r.prompt_len - 1)
        bs = self.block_size
        out: List[int] = []
        while (len(out) + 1) * bs <= limit:
            b = self.cache_index.get(r.tokens[:(len(out) + 1) * bs])
            if b is None:
                break
            out.append(b)
        return out

    # ------------------------------------------------- fault injection
    def hold_blocks(self, n: int) -> List[int]:
        """Take up to n blocks out of the allocatable pool, as allocation
        would (free queue head, then the newest initialized blocks), to
        simulate memory taken by something else; they stay out until
        release_blocks."""
        if self._pending is not None:
            raise RuntimeError("a step is open")
        out = []
        while len(out) < n and self._num_free() > 0:
            out.append(self._alloc())
        self.held.extend(out)
        return out

    def release_blocks(self, ids) -> None:
        """Return held blocks to the free queue's tail, in the given order."""
        if self._pending is not None:
            raise RuntimeError("a step is open")
        ids = [int(b) for b in ids]
        if len(set(ids)) != len(ids) or any(b not in self.held for b in ids):
            raise ValueError("not a held block")
        for b in ids:
            self.held.remove(b)
            del self.refs[b]
            self.free.append(b)

    def free_list(self) -> List[int]:
        """Allocatable blocks: the free queue, then the initialized pool."""
        return list(self.free) + list(self.free_init)

    def add_running_request(self, req_id: int, prompt_len: int,
                            output_len: int, num_cached: int) -> None:
        """Resume a request whose first ``num_cached`` tokens already have K/V
        in the cache (the swap-in path of "Offloading"): it joins the running
        set after the requests already there, with ceil(num_cached/bs) blocks
        taken from the free list."""
        if req_id in self.requests or prompt_len < 1 or output_len < 1:
            raise ValueError("bad request")
        if num_cached < 0 or num_cached > prompt_len + output_len - 2:
            raise ValueError("bad num_cached")
        if self._blocks_for(prompt_len + output_len - 1) > self.max_blocks_per_seq:
            raise ValueError("request longer than max_blocks_per_seq blocks")
        need = self._blocks_for(num_cached)
        if need > self._num_free():
            raise MemoryError("not enough free blocks")
        r = Request(req_id, prompt_len, output_len)
        r.num_cached = num_cached
        if num_cached >= prompt_len:
            r.state = DECODING
            r.num_generated = num_cached - prompt_len + 1
        else:
            r.state = PREFILLING
        for _ in range(need):
            r.blocks.append(self._alloc())
        self.requests[r.req_id] = r
        self.running.append(r)

    def slots(self, req_id: int, start: int, count: int) -> np.ndarray:
        r = self.requests[req_id]
        out = np.empty(count, dtype=np.int32)
        for i in range(count):
            pos = start + i
            out[i] = r.blocks[pos // self.block_size] * self.block_size + pos % self.block_size
        return out

    # ---------------------------------------------------------------- step
    def _is_long(self, r) -> bool:
        return self.long_prefill_tokens > 0 and r.prompt_len > self.long_prefill_tokens

    def _schedule(self):
        """One scheduling pass (no offloading); returns (batch, num_decodes,
        stalled).  An empty batch has allocated nothing."""
        budget = self.max_batch_tokens
        cap = self.max_requests_per_batch
        mpr = self.max_prefill_reqs
        dec, pre, new = [], [], []   # (request, num_tokens) per group
        stalled = []                 # (req_id, blocks demanded)
        rows = lambda: len(dec) + len(pre) + len(new)
        prefill_cap_hit = lambda: mpr > 0 and len(pre) + len(new) >= mpr

        def decodes():
            # active decodes, one token each, in admission order
            nonlocal budget
            for r in self.running:
                if r.state != DECODING:
                    continue
                if budget == 0 or rows() == cap:
                    break
                need = self._blocks_for(r.num_cached + 1) - len(r.blocks)
                if need > self._num_free():
                    stalled.append((r.req_id, need))
                    continue
                for _ in range(need):
                    r.blocks.append(self._alloc())
                dec.append((r, 1))
                budget -= 1

        def running_prefills():
            # active prefills, next chunk each, in admission order
            nonlocal budget
            for r in self.running:
                if r.state != PREFILLING:
                    continue
                if budget == 0 or rows() == cap or prefill_cap_hit():
                    break
                n = min(r.prompt_len - r.num_cached, budget)
                if self.max_prefill_chunk > 0:
                    n = min(n, self.max_prefill_chunk)
                need = self._blocks_for(r.num_cached + n) - len(r.blocks)
                if need > self._num_free():
                    stalled.append((r.req_id, need))
                    continue
                for _ in range(need):
                    r.blocks.append(self._alloc())
                pre.append((r, n))
                budget -= n

        def admissions():
            # waiting requests in arrival order, head-of-line except for long
            # prompts held back by the long-prefill cap
            nonlocal budget
            i = 0
            while i < len(self.waiting) and budget > 0 and rows() < cap and not prefill_cap_hit():
                r = self.waiting[i]
                if self._is_long(r):
                    active = sum(1 for x in self.running if x.state == PREFILLING and self._is_long(x))
                    if active >= self.max_long_prefills:
                        i += 1
                        continue
                shared = self._match(r)
                m = len(shared) * self.block_size
                n = min(r.prompt_len - m, budget)
                if self.max_prefill_chunk > 0:
                    n = min(n, self.max_prefill_chunk)
                need = self._blocks_for(m + n) - len(shared)
                from_pool = sum(1 for b in shared if b not in self.refs)
                if self._num_free() - from_pool - need < self.reserved_blocks:
                    break
                del self.waiting[i]
                for b in shared:
                    if b in self.refs:
                        self.refs[b] += 1
                    else:
                        self.free_init.remove(b)
                        self.refs[b] = 1
                r.blocks = list(shared)
                r.num_cached = m
                r.num_registered = len(shared)
                self.prefix_hit_tokens += m
                for _ in range(need):
                    r.blocks.append(self._alloc())
                r.state = PREFILLING
                self.running.append(r)
                new.append((r, n))
                budget -= n

        if self.policy == POLICY_PREFILL_FIRST:
            running_prefills()
            admissions()
            decodes()
        else:
            decodes()
            running_prefills()
            admissions()
        batch = dec + pre + new
        return batch, len(dec), stalled

    def _offload(self, r, swap_out) -> None:
        """Take an active request off the GPU: to the swap pool if it has room
        for all its blocks, else a soft reset."""
        self.running.remove(r)
        live = [b for b in r.blocks if b >= 0]
        if self.swap_free and len(self.swap_free) >= len(live):
            r.swap_slots = [self.swap_free.popleft() for _ in live]
            swap_out.extend(zip(live, r.swap_slots))
            r.swapped_table = [b >= 0 for b in r.blocks]
            r.resume_state = r.state
            r.state = SWAPPED
            self.swapped.append(r)
        else:
            r.prompt_len += r.num_generated
            r.output_len -= r.num_generated
            r.num_cached = 0
            r.num_generated = 0
            r.state = WAITING
            self.waiting.appendleft(r)
        self._release(r)

    def schedule_step(self) -> dict:
        if self._pending is not None:
            raise RuntimeError("schedule_step called twice without step_done")
        swap_in, swap_out = [], []     # (slot, block), (block, slot)
        resumed = set()
        if self.offload:
            # resume swapped requests, oldest offload first, while blocks allow
            while self.swapped:
                r = self.swapped[0]
                need = len(r.swap_slots)
                if self._num_free() - need < self.reserved_blocks:
                    break
                del self.swapped[0]
                slots = iter(r.swap_slots)
                for was_live in r.swapped_table:
                    if not was_live:
                        r.blocks.append(-1)
                        continue
                    slot = next(slots)
                    b = self._alloc()
                    r.blocks.append(b)
                    swap_in.append((slot, b))
                for slot in r.swap_slots:
                    self.swap_free.append(slot)
                r.swap_slots = []
                r.state = r.resume_state
                self.running.append(r)
                resumed.add(r.req_id)
        while True:
            batch, nd, stalled = self._schedule()
            if batch or not self.offload or not (stalled or self.waiting):
                break
            # nothing fits: offload the newest active request and retry
            cands = [r for r in self.running if r.req_id not in resumed]
            if len(self.running) <= 1 or not cands:
                break
            self._offload(cands[-1], swap_out)
        if self.offload and batch and stalled:
            # a batch fits but requests stalled: offload stalled requests,
            # newest first, until the rest of the demand can be met
            demand = {rid: need for rid, need in stalled}
            order = [r for r in reversed(self.running)
                     if r.req_id in demand and r.req_id not in resumed]
            for r in order:
                if self._num_free() >= sum(demand.values()) or len(self.running) <= 1:
                    break
                del demand[r.req_id]
                self._offload(r, swap_out)

        status = STATUS_OK
        if not batch and (stalled or self.waiting):
            status = STATUS_NO_BLOCKS
        step = self._emit(batch, nd, stalled, status)
        step["swap_in"] = np.asarray(swap_in, dtype=np.int32).reshape(-1, 2)
        step["swap_out"] = np.asarray(swap_out, dtype=np.int32).reshape(-1, 2)
        # an OK step (possibly empty) is committed by step_done; a NO_BLOCKS
        # step allocated nothing and leaves nothing to commit
        self._pending = batch if status == STATUS_OK else None
        return step

    def _emit(self, batch, num_decodes, stalled, status) -> dict:
        R = len(batch)
        cu = np.zeros(R + 1, dtype=np.int32)
        seq_lens = np.zeros(R, dtype=np.int32)
        tables = np.full((R, self.max_blocks_per_seq), -1, dtype=np.int32)
        req_ids = np.zeros(R, dtype=np.int64)
        slots = []
        for i, (r, n) in enumerate(batch):
            req_ids[i] = r.req_id
            cu[i + 1] = cu[i] + n
            seq_lens[i] = r.num_cached + n
            tables[i, :len(r.blocks)] = r.blocks
            for pos in range(r.num_cached, r.num_cached + n):
                slots.append(r.blocks[pos // self.block_size] * self.block_size
                             + pos % self.block_size)
        return {
            "status": status,
            "num_reqs": R,
            "num_tokens": int(cu[-1]),
            "num_decodes": num_decodes,
            "req_ids": req_ids,
            "cu_seqlens_q": cu,
            "seq_lens": seq_lens,
            "block_tables": tables,
            "slot_mapping": np.asarray(slots, dtype=np.int32),
            "stalled_ids": np.asarray([s[0] for s in stalled], dtype=np.int64),
            "stalled_demand": np.asarray([s[1] for s in stalled], dtype=np.int32),
        }

    def step_done(self) -> List[int]:
        """Commit the open step; returns the ids of requests that finished."""
        if self._pending is None:
            raise RuntimeError("no open step")
        finished = []
        for r, n in self._pending:
            r.num_cached += n
            if r.state == PREFILLING:
                if r.num_cached == r.prompt_len:
                    r.num_generated = 1
                    r.state = DECODING
            else:
                r.num_generated += 1
            if r.state == DECODING and r.num_generated >= r.output_len:
                r.state = FINISHED
                finished.append(r)
        if self.prefix_caching:
            # key every block this step completed inside the known tokens
            bs = self.block_size
            for r, _ in self._pending:
                if r.tokens is None:
                    continue
                full = min(r.num_cached, len(r.tokens)) // bs
                while r.num_registered < full:
                    i = r.num_registered
                    key = r.tokens[:(i + 1) * bs]
                    if key not in self.cache_index:
                        self.cache_index[key] = r.blocks[i]
                        self.block_key[r.blocks[i]] = key
                    r.num_registered += 1
        if self.sliding_window > 0:
            # pages wholly before every future query's window go back
            bs = self.block_size
            for r, _ in self._pending:
                if r.state == FINISHED:
                    continue
                lo = max(0, r.num_cached - self.sliding_window + 1) // bs
                for j in range(min(lo, len(r.blocks))):
                    b = r.blocks[j]
                    if b >= 0:
                        self.refs[b] -= 1
                        if self.refs[b] == 0:
                            del self.refs[b]
                            self.free.append(b)
                        r.blocks[j] = -1
        for r in finished:
            self.running.remove(r)
            self._release(r)
        self._pending = None
        return [r.req_id for r in finished]

    # -------------------------------------------------------------- counts
    def counts(self):
        return self._num_free(), len(self.waiting), len(self.running)

    def swapped_ids(self) -> List[int]:
        return [r.req_id for r in self.swapped]
