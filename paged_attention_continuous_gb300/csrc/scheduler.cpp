// FIFO continuous-batching scheduler with a paged block pool (host side).
//
// Behaviour follows "Continuous batching architecture" (HF Transformers docs):
//   * Request lifecycle: PENDING -> PREFILLING -> DECODING -> FINISHED; one
//     output token per decode step.
//   * Chunked prefill: a prompt beyond the remaining token budget is cut; the
//     rest resumes next step where it stopped.
//   * Scheduler: token budget (max_batch_tokens), cache budget (free blocks),
//     request cap (max_requests_per_batch).
//   * FIFO: running decodes first, then running prefills, then waiting
//     requests in arrival order.
//   * Admission: all-or-nothing allocation; safety_margin keeps new prefills
//     out while free capacity would drop below it.
//   * Offloading: active requests that cannot get their blocks are reported
//     as stalled together with their block demand.
// and the block pool of "vLLM serving internals" (PagedAttention as a virtual
// memory system): fixed-size blocks, one block table per sequence, a new
// block when a sequence outgrows its last one, blocks back to the pool when
// it finishes.
//
// Where the pages leave a step open the choices are: batch rows in the order
// decodes / running prefills / new prompts; strict head-of-line admission;
// chunk = min(remaining prompt, remaining budget, max_prefill_chunk);
// allocation only for the scheduled tokens; the free list is a FIFO queue
// (pop from the head, finished requests push their blocks to the tail in
// batch order and logical block order); the margin test is
// free_after >= ceil((double)margin * num_blocks) for new requests only; the
// step that completes a prompt yields the first output token.
//
// Policies: FIFO (above) or PrefillFirst ("Continuous batching architecture",
// PrefillFirst: chunked prefills are completed before decoding resumes):
// running prefills, then new prompts, then decodes with the budget and
// request cap that are left; rows are still emitted decodes first.  Optional
// caps: prefill rows per step, and (vLLM performance post, request-parallel
// prefill) the number of long prompts in their prefill phase at once -- a
// long waiting request held by that cap is skipped instead of blocking the
// shorter requests behind it.
//
// Offloading ("Continuous batching architecture", Offloading and Soft
// reset), when enabled: if a batch was scheduled but requests stalled, the
// fewest stalled requests, newest first, are taken off the GPU until the
// rest of the demand fits; if no batch fits at all, the newest active
// request is taken off and the step is scheduled again, until one fits or
// nothing is left to take.  The last active request is never taken.  A
// victim goes to the CPU swap pool when its free slots hold all its blocks
// (resumed later, oldest offload first, at the start of a step when blocks
// allow, without recomputation), else it is soft-reset: its generated
// tokens join its prompt, its blocks are freed and it goes to the front of
// the waiting queue.  A request resumed in a step is not a victim in it.
//
// Prefix caching ("Continuous batching architecture", Prefix caching,
// Eviction), when enabled, for requests queued with their prompt token ids:
// a block that lies inside the known tokens is keyed, when the step that
// completes it is committed, by a fingerprint of the whole token prefix up
// to its end -- so blocks match only as a leading run -- unless another
// block already holds that key.  A new request reuses the longest leading
// run of keyed blocks (one prompt token is always left to compute, since
// the step that completes a prompt yields its first output token), and the
// reused tokens count as cached.  Blocks are reference-counted.  A freed
// keyed block keeps its contents and key in an "initialized" pool, still
// matchable; allocation takes the free queue first and, when it is empty,
// demotes the newest initialized block (dropping its key).
//
// Sliding-window layers ("Continuous batching architecture", Memory
// management: they keep a fixed window of recent tokens by recycling a small
// set of pages), when the pool serves such layers: a query at position p
// reads keys p-W+1..p, so after each committed step the pages of a running
// request that lie wholly before num_cached - W + 1 go back to the free
// queue and their table entries become -1.
//
// The fingerprint is two 64-bit lanes over the prefix's token ids: FNV-1a
// (Fowler, Noll, Vo) over their little-endian bytes, and a chain of the
// splitmix64 output function (Steele, Lea, Flood) over the ids; a match
// also compares the block's own tokens.  Two different prefixes that end
// in the same block of tokens would have to agree on all 128 bits to be
// confused.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <deque>
#include <list>
#include <memory>
#include <new>
#include <unordered_map>
#include <vector>

#include "cb_error.h"

namespace cb {

std::string& last_error_slot() {
  static thread_local std::string s;
  return s;
}

struct Fp {
  uint64_t a = 0, b = 0;
  bool operator==(const Fp& o) const { return a == o.a && b == o.b; }
};

struct FpHash {
  size_t operator()(const Fp& f) const { return (size_t)(f.a ^ (f.b * 0x9E3779B97F4A7C15ull)); }
};

constexpr uint64_t kFnvOffset = 14695981039346656037ull;
constexpr uint64_t kFnvPrime = 1099511628211ull;

uint64_t splitmix_out(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Fingerprints of the prefixes ending at each full block of `tokens`.
std::vector<Fp> prefix_fingerprints(const std::vector<int32_t>& tokens, int32_t bs) {
  std::vector<Fp> out;
  Fp h{kFnvOffset, 0};
  for (size_t i = 0; i < tokens.size(); ++i) {
    const uint32_t t = (uint32_t)tokens[i];
    for (int k = 0; k < 4; ++k) {
      h.a ^= (t >> (8 * k)) & 0xffu;
      h.a *= kFnvPrime;
    }
    h.b = splitmix_out(h.b + 0x9E3779B97F4A7C15ull + t);
    if ((i + 1) % (size_t)bs == 0) out.push_back(h);
  }
  return out;
}

enum class State { kWaiting, kPrefilling, kDecoding, kFinished, kSwapped };

struct Request {
  int64_t id = 0;
  int32_t prompt_len = 0;
  int32_t output_len = 0;
  int32_t num_cached = 0;     // tokens whose K/V is in the cache
  int32_t num_generated = 0;  // output tokens produced so far
  State state = State::kWaiting;
  std::vector<int32_t> blocks;
  std::vector<int32_t> swap_slots;    // while swapped: slot of each live block
  std::vector<char> swapped_live;     // while swapped: table entry was live
  State resume_state = State::kWaiting;
  // prefix caching: known prompt token ids, the fingerprint of each full
  // block of them (prefix up to the block's end), leading blocks already
  // considered for keys
  std::vector<int32_t> tokens;
  bool has_tokens = false;
  std::vector<Fp> fps;
  size_t num_registered = 0;
};

struct Scheduled {
  Request* req;
  int32_t num_tokens;
};

}  // namespace cb

struct cb_sched {
  cb_config cfg{};
  int64_t reserved_blocks = 0;
  std::deque<int32_t> free_list;
  std::deque<cb::Request*> waiting;
  std::vector<cb::Request*> running;  // admission order
  std::unordered_map<int64_t, std::unique_ptr<cb::Request>> requests;
  bool step_open = false;
  std::vector<cb::Scheduled> batch;
  // step outputs (host arrays owned here)
  std::vector<int64_t> req_ids;
  std::vector<int32_t> cu_seqlens_q, seq_lens, block_tables, slot_mapping;
  std::vector<int64_t> stalled_ids;
  std::vector<int32_t> stalled_demand;
  std::vector<int64_t> finished_ids;
  // offloading
  std::deque<int32_t> swap_free;
  std::vector<cb::Request*> swapped;  // offload order
  std::vector<int32_t> swap_in_slots, swap_in_blocks, swap_out_blocks, swap_out_slots;
  // block pool state for prefix caching (reference counts are kept always)
  std::vector<int32_t> refs;                       // users of each block
  std::list<int32_t> free_init;                    // initialized pool, freed order
  std::vector<std::list<int32_t>::iterator> init_pos;
  std::vector<char> in_init, keyed;
  std::vector<cb::Fp> block_fp;                    // key of a keyed block
  std::vector<int32_t> block_tokens;               // its own tokens [num_blocks][bs]
  std::unordered_map<cb::Fp, int32_t, cb::FpHash> index;
  int64_t prefix_hits = 0;
  std::vector<char> held;                          // taken by cb_sched_hold_blocks
};

namespace {

int64_t blocks_for(const cb_sched* s, int64_t tokens) {
  const int64_t bs = s->cfg.block_size;
  return (tokens + bs - 1) / bs;
}

int64_t num_free(const cb_sched* s) {
  return (int64_t)s->free_list.size() + (int64_t)s->free_init.size();
}

// One block for a new user: the free queue's head, else the newest
// initialized block, demoted (its key dropped).
int32_t alloc_block(cb_sched* s) {
  int32_t b;
  if (!s->free_list.empty()) {
    b = s->free_list.front();
    s->free_list.pop_front();
  } else {
    b = s->free_init.back();
    s->free_init.pop_back();
    s->in_init[b] = 0;
    s->index.erase(s->block_fp[b]);
    s->keyed[b] = 0;
  }
  s->refs[b] = 1;
  return b;
}

void take_blocks(cb_sched* s, cb::Request* r, int64_t n) {
  for (int64_t i = 0; i < n; ++i) r->blocks.push_back(alloc_block(s));
}

// Drop r's use of its blocks (logical order): a block with no user left goes
// to the initialized pool if keyed, else to the tail of the free queue.
void release_blocks(cb_sched* s, cb::Request* r) {
  for (int32_t b : r->blocks) {
    if (b < 0) continue;  // recycled out of the window
    if (--s->refs[b] > 0) continue;
    if (s->keyed[b]) {
      s->free_init.push_back(b);
      s->init_pos[b] = std::prev(s->free_init.end());
      s->in_init[b] = 1;
    } else {
      s->free_list.push_back(b);
    }
  }
  r->blocks.clear();
  r->num_registered = 0;
}

// Blocks of the longest leading run of r's prompt that are keyed.
void match_prefix(const cb_sched* s, const cb::Request* r, std::vector<int32_t>* out) {
  out->clear();
  if (!s->cfg.prefix_caching || !r->has_tokens) return;
  const int64_t bs = s->cfg.block_size;
  const int64_t limit = std::min<int64_t>((int64_t)r->tokens.size(), (int64_t)r->prompt_len - 1);
  for (size_t i = 0; (int64_t)(i + 1) * bs <= limit; ++i) {
    auto it = s->index.find(r->fps[i]);
    if (it == s->index.end()) break;
    const int32_t b = it->second;
    if (!std::equal(r->tokens.begin() + (std::ptrdiff_t)(i * bs),
                    r->tokens.begin() + (std::ptrdiff_t)((i + 1) * bs),
                    s->block_tokens.begin() + (std::ptrdiff_t)b * bs))
      break;
    out->push_back(b);
  }
}

cb_status check_new_request(cb_sched* s, int64_t id, int32_t prompt_len,
                            int32_t output_len) {
  if (s->requests.count(id)) return cb::fail(CB_ERR_INVALID_ARG, "duplicate request id %lld", (long long)id);
  if (prompt_len < 1 || output_len < 1)
    return cb::fail(CB_ERR_INVALID_ARG, "prompt_len and output_len must be >= 1");
  const int64_t longest = (int64_t)prompt_len + output_len - 1;
  if (blocks_for(s, longest) > s->cfg.max_blocks_per_seq)
    return cb::fail(CB_ERR_INVALID_ARG,
                    "request %lld needs %lld blocks > max_blocks_per_seq %d", (long long)id,
                    (long long)blocks_for(s, longest), s->cfg.max_blocks_per_seq);
  return CB_OK;
}

void emit_step(cb_sched* s, int32_t num_decodes, cb_step* out) {
  const int32_t R = (int32_t)s->batch.size();
  const int32_t W = s->cfg.max_blocks_per_seq;
  const int32_t bs = s->cfg.block_size;
  s->req_ids.assign(R, 0);
  s->cu_seqlens_q.assign(R + 1, 0);
  s->seq_lens.assign(R, 0);
  s->block_tables.assign((size_t)R * W, -1);
  s->slot_mapping.clear();
  int32_t max_q = 0, max_seq = 0;
  for (int32_t i = 0; i < R; ++i) {
    const cb::Request* r = s->batch[i].req;
    const int32_t n = s->batch[i].num_tokens;
    s->req_ids[i] = r->id;
    s->cu_seqlens_q[i + 1] = s->cu_seqlens_q[i] + n;
    s->seq_lens[i] = r->num_cached + n;
    max_q = std::max(max_q, n);
    max_seq = std::max(max_seq, s->seq_lens[i]);
    std::copy(r->blocks.begin(), r->blocks.end(), s->block_tables.begin() + (size_t)i * W);
    // slot of position pos = blocks[pos / bs] * bs + pos % bs, walked block
    // by block (one division per row, not per token)
    int32_t pos = r->num_cached;
    const int32_t end = r->num_cached + n;
    while (pos < end) {
      const int32_t bi = pos / bs;
      const int32_t off = pos - bi * bs;
      const int32_t run = std::min(bs - off, end - pos);
      const int32_t base = r->blocks[bi] * bs + off;
      for (int32_t k = 0; k < run; ++k) s->slot_mapping.push_back(base + k);
      pos += run;
    }
  }
  out->num_reqs = R;
  out->num_tokens = s->cu_seqlens_q[R];
  out->num_decodes = num_decodes;
  out->max_q_len = max_q;
  out->max_seq_len = max_seq;
  out->max_blocks_per_seq = W;
  out->req_ids = s->req_ids.data();
  out->cu_seqlens_q = s->cu_seqlens_q.data();
  out->seq_lens = s->seq_lens.data();
  out->block_tables = s->block_tables.data();
  out->slot_mapping = s->slot_mapping.data();
  out->num_stalled = (int32_t)s->stalled_ids.size();
  out->stalled_ids = s->stalled_ids.data();
  out->stalled_demand = s->stalled_demand.data();
  out->num_swap_in = (int32_t)s->swap_in_slots.size();
  out->swap_in_slots = s->swap_in_slots.data();
  out->swap_in_blocks = s->swap_in_blocks.data();
  out->num_swap_out = (int32_t)s->swap_out_blocks.size();
  out->swap_out_blocks = s->swap_out_blocks.data();
  out->swap_out_slots = s->swap_out_slots.data();
}

// Take an active request off the GPU: to the swap pool if its free slots
// hold all its blocks, else a soft reset.
void offload_request(cb_sched* s, cb::Request* r) {
  s->running.erase(std::find(s->running.begin(), s->running.end(), r));
  size_t live = 0;
  for (int32_t b : r->blocks) live += b >= 0;
  if (!s->swap_free.empty() && s->swap_free.size() >= live) {
    r->swap_slots.clear();
    r->swapped_live.clear();
    for (int32_t b : r->blocks) r->swapped_live.push_back(b >= 0);
    for (int32_t b : r->blocks) {
      if (b < 0) continue;
      const int32_t slot = s->swap_free.front();
      s->swap_free.pop_front();
      r->swap_slots.push_back(slot);
      s->swap_out_blocks.push_back(b);
      s->swap_out_slots.push_back(slot);
    }
    r->resume_state = r->state;
    r->state = cb::State::kSwapped;
    s->swapped.push_back(r);
  } else {
    r->prompt_len += r->num_generated;
    r->output_len -= r->num_generated;
    r->num_cached = 0;
    r->num_generated = 0;
    r->state = cb::State::kWaiting;
    s->waiting.push_front(r);
  }
  release_blocks(s, r);
}

}  // namespace

namespace {
// One scheduling pass without offloading: fills s->batch (rows decodes
// first) and the stalled lists.  An empty batch has allocated nothing.
void schedule_pass(cb_sched* s, int32_t* num_decodes) {
  int64_t budget = s->cfg.max_batch_tokens;
  const size_t cap = (size_t)s->cfg.max_requests_per_batch;
  const int64_t chunk_cap = s->cfg.max_prefill_chunk;
  const size_t mpr = (size_t)s->cfg.max_prefill_reqs;
  s->batch.clear();
  s->stalled_ids.clear();
  s->stalled_demand.clear();
  std::vector<cb::Scheduled> dec, pre, fresh;
  auto rows = [&] { return dec.size() + pre.size() + fresh.size(); };
  auto prefill_cap_hit = [&] { return mpr > 0 && pre.size() + fresh.size() >= mpr; };
  auto is_long = [&](const cb::Request* r) {
    return s->cfg.long_prefill_tokens > 0 && r->prompt_len > s->cfg.long_prefill_tokens;
  };
  auto stall = [&](const cb::Request* r, int64_t need) {
    s->stalled_ids.push_back(r->id);
    s->stalled_demand.push_back((int32_t)need);
  };

  // running decodes, one token each, admission order
  auto decodes = [&] {
    for (cb::Request* r : s->running) {
      if (r->state != cb::State::kDecoding) continue;
      if (budget == 0 || rows() == cap) break;
      const int64_t need = blocks_for(s, (int64_t)r->num_cached + 1) - (int64_t)r->blocks.size();
      if (need > num_free(s)) {
        stall(r, need);
        continue;
      }
      take_blocks(s, r, need);
      dec.push_back({r, 1});
      budget -= 1;
    }
  };
  // running prefills, next chunk each, admission order
  auto running_prefills = [&] {
    for (cb::Request* r : s->running) {
      if (r->state != cb::State::kPrefilling) continue;
      if (budget == 0 || rows() == cap || prefill_cap_hit()) break;
      int64_t n = std::min<int64_t>(r->prompt_len - r->num_cached, budget);
      if (chunk_cap > 0) n = std::min(n, chunk_cap);
      const int64_t need = blocks_for(s, r->num_cached + n) - (int64_t)r->blocks.size();
      if (need > num_free(s)) {
        stall(r, need);
        continue;
      }
      take_blocks(s, r, need);
      pre.push_back({r, (int32_t)n});
      budget -= n;
    }
  };
  // waiting requests, arrival order, head-of-line except long prompts held
  // back by the long-prefill cap
  std::vector<int32_t> shared;
  auto admissions = [&] {
    size_t i = 0;
    while (i < s->waiting.size() && budget > 0 && rows() < cap && !prefill_cap_hit()) {
      cb::Request* r = s->waiting[i];
      if (is_long(r)) {
        int32_t active = 0;
        for (const cb::Request* x : s->running)
          if (x->state == cb::State::kPrefilling && is_long(x)) ++active;
        if (active >= s->cfg.max_long_prefills) {
          ++i;
          continue;
        }
      }
      match_prefix(s, r, &shared);
      const int64_t m = (int64_t)shared.size() * s->cfg.block_size;
      int64_t n = std::min<int64_t>(r->prompt_len - m, budget);
      if (chunk_cap > 0) n = std::min(n, chunk_cap);
      const int64_t need = blocks_for(s, m + n) - (int64_t)shared.size();
      int64_t from_pool = 0;
      for (int32_t b : shared) from_pool += s->refs[b] == 0;
      if (num_free(s) - from_pool - need < s->reserved_blocks) break;
      s->waiting.erase(s->waiting.begin() + (std::ptrdiff_t)i);
      for (int32_t b : shared) {
        if (s->refs[b] > 0) {
          ++s->refs[b];
        } else {
          s->free_init.erase(s->init_pos[b]);
          s->in_init[b] = 0;
          s->refs[b] = 1;
        }
      }
      r->blocks = shared;
      r->num_cached = (int32_t)m;
      r->num_registered = shared.size();
      s->prefix_hits += m;
      take_blocks(s, r, need);
      r->state = cb::State::kPrefilling;
      s->running.push_back(r);
      fresh.push_back({r, (int32_t)n});
      budget -= n;
    }
  };

  if (s->cfg.policy == CB_POLICY_PREFILL_FIRST) {
    running_prefills();
    admissions();
    decodes();
  } else {
    decodes();
    running_prefills();
    admissions();
  }
  *num_decodes = (int32_t)dec.size();
  s->batch = dec;
  s->batch.insert(s->batch.end(), pre.begin(), pre.end());
  s->batch.insert(s->batch.end(), fresh.begin(), fresh.end());

}

}  // namespace

extern "C" {

const char* cb_last_error(void) { return cb::last_error_slot().c_str(); }

int32_t cb_version(void) { return (1 << 16) | 0; }

cb_status cb_sched_create(const cb_config* cfg, cb_sched** out) {
  if (!out) return cb::fail(CB_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!cfg) return cb::fail(CB_ERR_INVALID_ARG, "cfg is NULL");
  if (cfg->block_size <= 0 || cfg->num_blocks <= 0 || cfg->max_batch_tokens <= 0 ||
      cfg->max_requests_per_batch <= 0 || cfg->max_blocks_per_seq <= 0 ||
      cfg->max_prefill_chunk < 0 || cfg->max_prefill_reqs < 0 || cfg->long_prefill_tokens < 0 ||
      cfg->max_long_prefills < 0 || cfg->swap_blocks < 0 || cfg->sliding_window < 0)
    return cb::fail(CB_ERR_INVALID_ARG, "config sizes must be positive");
  if (cfg->sliding_window > 0 && cfg->prefix_caching)
    return cb::fail(CB_ERR_INVALID_ARG, "sliding-window layers do not share blocks (prefix_caching)");
  if (cfg->policy != CB_POLICY_FIFO && cfg->policy != CB_POLICY_PREFILL_FIRST)
    return cb::fail(CB_ERR_INVALID_ARG, "unknown policy %d", cfg->policy);
  if (!(cfg->safety_margin >= 0.0f) || cfg->safety_margin > 1.0f)
    return cb::fail(CB_ERR_INVALID_ARG, "safety_margin must be in [0, 1]");
  std::unique_ptr<cb_sched> s(new (std::nothrow) cb_sched());
  if (!s) return cb::fail(CB_ERR_INVALID_ARG, "out of host memory");
  s->cfg = *cfg;
  s->cfg.initial_free_list = nullptr;
  s->reserved_blocks = (int64_t)std::ceil((double)cfg->safety_margin * (double)cfg->num_blocks);
  for (int32_t i = 0; i < cfg->swap_blocks; ++i) s->swap_free.push_back(i);
  // touch the per-step output arrays once (up to 16 MB) so that the first
  // scheduled step does not pay their page faults
  {
    const size_t rows = (size_t)cfg->max_requests_per_batch;
    const size_t table = rows * (size_t)cfg->max_blocks_per_seq;
    if (table * sizeof(int32_t) <= ((size_t)16 << 20)) {
      s->block_tables.assign(table, -1);
      s->block_tables.clear();
    }
    s->slot_mapping.assign((size_t)cfg->max_batch_tokens, 0);
    s->slot_mapping.clear();
    s->req_ids.assign(rows, 0);
    s->cu_seqlens_q.assign(rows + 1, 0);
    s->seq_lens.assign(rows, 0);
  }
  s->refs.assign(cfg->num_blocks, 0);
  s->held.assign(cfg->num_blocks, 0);
  s->init_pos.resize(cfg->num_blocks);
  s->in_init.assign(cfg->num_blocks, 0);
  s->keyed.assign(cfg->num_blocks, 0);
  if (cfg->prefix_caching) {
    s->block_fp.resize(cfg->num_blocks);
    s->block_tokens.assign((size_t)cfg->num_blocks * cfg->block_size, 0);
  }
  if (cfg->initial_free_list) {
    std::vector<char> seen(cfg->num_blocks, 0);
    for (int32_t i = 0; i < cfg->num_blocks; ++i) {
      const int32_t b = cfg->initial_free_list[i];
      if (b < 0 || b >= cfg->num_blocks || seen[b])
        return cb::fail(CB_ERR_INVALID_ARG, "initial_free_list is not a permutation");
      seen[b] = 1;
      s->free_list.push_back(b);
    }
  } else {
    for (int32_t i = 0; i < cfg->num_blocks; ++i) s->free_list.push_back(i);
  }
  *out = s.release();
  return CB_OK;
}

void cb_sched_destroy(cb_sched* s) { delete s; }

cb_status cb_add_request(cb_sched* s, int64_t req_id, int32_t prompt_len, int32_t output_len) {
  if (!s) return cb::fail(CB_ERR_INVALID_ARG, "scheduler is NULL");
  cb_status st = check_new_request(s, req_id, prompt_len, output_len);
  if (st != CB_OK) return st;
  auto r = std::make_unique<cb::Request>();
  r->id = req_id;
  r->prompt_len = prompt_len;
  r->output_len = output_len;
  s->waiting.push_back(r.get());
  s->requests.emplace(req_id, std::move(r));
  return CB_OK;
}

cb_status cb_add_request_tokens(cb_sched* s, int64_t req_id, int32_t prompt_len,
                                int32_t output_len, const int32_t* tokens, int32_t num_tokens) {
  if (!s) return cb::fail(CB_ERR_INVALID_ARG, "scheduler is NULL");
  if (num_tokens < 0 || num_tokens > prompt_len || (num_tokens > 0 && !tokens))
    return cb::fail(CB_ERR_INVALID_ARG, "num_tokens must be in [0, prompt_len] with tokens given");
  cb_status st = cb_add_request(s, req_id, prompt_len, output_len);
  if (st != CB_OK) return st;
  cb::Request* r = s->requests[req_id].get();
  r->has_tokens = true;
  if (s->cfg.prefix_caching) {
    r->tokens.assign(tokens, tokens + num_tokens);
    r->fps = cb::prefix_fingerprints(r->tokens, s->cfg.block_size);
  }
  return CB_OK;
}

cb_status cb_add_running_request(cb_sched* s, int64_t req_id, int32_t prompt_len,
                                 int32_t output_len, int32_t num_cached) {
  if (!s) return cb::fail(CB_ERR_INVALID_ARG, "scheduler is NULL");
  cb_status st = check_new_request(s, req_id, prompt_len, output_len);
  if (st != CB_OK) return st;
  if (num_cached < 0 || (int64_t)num_cached > (int64_t)prompt_len + output_len - 2)
    return cb::fail(CB_ERR_INVALID_ARG, "num_cached must be in [0, prompt_len + output_len - 2]");
  if (s->step_open) return cb::fail(CB_ERR_STATE, "a step is open; call cb_step_done first");
  const int64_t need = blocks_for(s, num_cached);
  if (need > num_free(s))
    return cb::fail(CB_ERR_NO_BLOCKS, "not enough free blocks to resume request %lld", (long long)req_id);
  auto r = std::make_unique<cb::Request>();
  r->id = req_id;
  r->prompt_len = prompt_len;
  r->output_len = output_len;
  r->num_cached = num_cached;
  if (num_cached >= prompt_len) {
    r->state = cb::State::kDecoding;
    r->num_generated = num_cached - prompt_len + 1;
  } else {
    r->state = cb::State::kPrefilling;
  }
  take_blocks(s, r.get(), need);
  s->running.push_back(r.get());
  s->requests.emplace(req_id, std::move(r));
  return CB_OK;
}

cb_status cb_schedule_step(cb_sched* s, cb_step* out) {
  if (!s || !out) return cb::fail(CB_ERR_INVALID_ARG, "NULL argument");
  if (s->step_open) return cb::fail(CB_ERR_STATE, "previous step not committed with cb_step_done");
  s->swap_in_slots.clear();
  s->swap_in_blocks.clear();
  s->swap_out_blocks.clear();
  s->swap_out_slots.clear();
  std::vector<cb::Request*> resumed;
  const bool offload = s->cfg.offload != 0;
  if (offload) {
    // resume swapped requests, oldest offload first, while blocks allow
    while (!s->swapped.empty()) {
      cb::Request* r = s->swapped.front();
      const int64_t need = (int64_t)r->swap_slots.size();
      if (num_free(s) - need < s->reserved_blocks) break;
      s->swapped.erase(s->swapped.begin());
      size_t k = 0;
      for (char was_live : r->swapped_live) {
        if (!was_live) {
          r->blocks.push_back(-1);
          continue;
        }
        const int32_t slot = r->swap_slots[k++];
        const int32_t b = alloc_block(s);
        r->blocks.push_back(b);
        s->swap_in_slots.push_back(slot);
        s->swap_in_blocks.push_back(b);
      }
      for (int32_t slot : r->swap_slots) s->swap_free.push_back(slot);
      r->swap_slots.clear();
      r->state = r->resume_state;
      s->running.push_back(r);
      resumed.push_back(r);
    }
  }
  auto was_resumed = [&](const cb::Request* r) {
    return std::find(resumed.begin(), resumed.end(), r) != resumed.end();
  };
  int32_t num_decodes = 0;
  while (true) {
    schedule_pass(s, &num_decodes);
    if (!s->batch.empty() || !offload || (s->stalled_ids.empty() && s->waiting.empty())) break;
    // nothing fits: take the newest active request off and schedule again
    cb::Request* victim = nullptr;
    for (auto it = s->running.rbegin(); it != s->running.rend(); ++it)
      if (!was_resumed(*it)) {
        victim = *it;
        break;
      }
    if (s->running.size() <= 1 || !victim) break;
    offload_request(s, victim);
  }
  if (offload && !s->batch.empty() && !s->stalled_ids.empty()) {
    // a batch fits but requests stalled: take stalled requests off, newest
    // first, until the rest of the demand can be met
    std::vector<std::pair<int64_t, int64_t>> demand;  // (id, blocks)
    for (size_t i = 0; i < s->stalled_ids.size(); ++i)
      demand.push_back({s->stalled_ids[i], s->stalled_demand[i]});
    std::vector<cb::Request*> order;
    for (auto it = s->running.rbegin(); it != s->running.rend(); ++it) {
      const int64_t id = (*it)->id;
      if (was_resumed(*it)) continue;
      for (const auto& d : demand)
        if (d.first == id) {
          order.push_back(*it);
          break;
        }
    }
    for (cb::Request* r : order) {
      int64_t total = 0;
      for (const auto& d : demand) total += d.second;
      if (num_free(s) >= total || s->running.size() <= 1) break;
      for (size_t i = 0; i < demand.size(); ++i)
        if (demand[i].first == r->id) {
          demand.erase(demand.begin() + (std::ptrdiff_t)i);
          break;
        }
      offload_request(s, r);
    }
  }

  emit_step(s, num_decodes, out);
  if (s->batch.empty() && (!s->stalled_ids.empty() || !s->waiting.empty())) {
    s->step_open = false;
    return cb::fail(CB_ERR_NO_BLOCKS, "no batch could be scheduled (%d stalled, %zu waiting)",
                    out->num_stalled, s->waiting.size());
  }
  s->step_open = true;
  return CB_OK;
}

cb_status cb_step_done(cb_sched* s, int32_t* num_finished, const int64_t** finished_ids) {
  if (!s) return cb::fail(CB_ERR_INVALID_ARG, "scheduler is NULL");
  if (!s->step_open) return cb::fail(CB_ERR_STATE, "no open step");
  s->finished_ids.clear();
  std::vector<cb::Request*> done;
  for (const cb::Scheduled& e : s->batch) {
    cb::Request* r = e.req;
    r->num_cached += e.num_tokens;
    if (r->state == cb::State::kPrefilling) {
      if (r->num_cached == r->prompt_len) {
        r->num_generated = 1;
        r->state = cb::State::kDecoding;
      }
    } else {
      r->num_generated += 1;
    }
    if (r->state == cb::State::kDecoding && r->num_generated >= r->output_len) {
      r->state = cb::State::kFinished;
      done.push_back(r);
    }
  }
  if (s->cfg.prefix_caching) {
    // key every block this step completed inside the known tokens
    const size_t bs = (size_t)s->cfg.block_size;
    for (const cb::Scheduled& e : s->batch) {
      cb::Request* r = e.req;
      if (!r->has_tokens) continue;
      const size_t full = std::min<size_t>((size_t)r->num_cached, r->tokens.size()) / bs;
      for (; r->num_registered < full; ++r->num_registered) {
        const size_t i = r->num_registered;
        const int32_t b = r->blocks[i];
        if (!s->index.emplace(r->fps[i], b).second) continue;
        s->keyed[b] = 1;
        s->block_fp[b] = r->fps[i];
        std::copy(r->tokens.begin() + (std::ptrdiff_t)(i * bs),
                  r->tokens.begin() + (std::ptrdiff_t)((i + 1) * bs),
                  s->block_tokens.begin() + (std::ptrdiff_t)b * (std::ptrdiff_t)bs);
      }
    }
  }
  if (s->cfg.sliding_window > 0) {
    // pages wholly before every future query's window go back
    const int64_t bs = s->cfg.block_size;
    for (const cb::Scheduled& e : s->batch) {
      cb::Request* r = e.req;
      if (r->state == cb::State::kFinished) continue;
      const int64_t lo =
          std::min<int64_t>(std::max<int64_t>(0, (int64_t)r->num_cached - s->cfg.sliding_window + 1) / bs,
                            (int64_t)r->blocks.size());
      for (int64_t j = 0; j < lo; ++j) {
        const int32_t b = r->blocks[j];
        if (b < 0) continue;
        if (--s->refs[b] == 0) s->free_list.push_back(b);
        r->blocks[j] = -1;
      }
    }
  }
  for (cb::Request* r : done) {
    s->running.erase(std::find(s->running.begin(), s->running.end(), r));
    release_blocks(s, r);
    s->finished_ids.push_back(r->id);
    s->requests.erase(r->id);
  }
  s->batch.clear();
  s->step_open = false;
  if (num_finished) *num_finished = (int32_t)s->finished_ids.size();
  if (finished_ids) *finished_ids = s->finished_ids.data();
  return CB_OK;
}

cb_status cb_request_slots(const cb_sched* s, int64_t req_id, int32_t start, int32_t count,
                           int32_t* slots_out) {
  if (!s || (count > 0 && !slots_out)) return cb::fail(CB_ERR_INVALID_ARG, "NULL argument");
  auto it = s->requests.find(req_id);
  if (it == s->requests.end()) return cb::fail(CB_ERR_INVALID_ARG, "unknown request %lld", (long long)req_id);
  const cb::Request* r = it->second.get();
  const int64_t bs = s->cfg.block_size;
  if (start < 0 || count < 0 || (int64_t)start + count > (int64_t)r->blocks.size() * bs)
    return cb::fail(CB_ERR_INVALID_ARG, "positions outside the request's blocks");
  for (int32_t i = 0; i < count; ++i) {
    const int64_t pos = (int64_t)start + i;
    slots_out[i] = (int32_t)(r->blocks[pos / bs] * bs + pos % bs);
  }
  return CB_OK;
}

cb_status cb_sched_counts(const cb_sched* s, int32_t* free_blocks, int32_t* num_waiting,
                          int32_t* num_running) {
  if (!s) return cb::fail(CB_ERR_INVALID_ARG, "scheduler is NULL");
  if (free_blocks) *free_blocks = (int32_t)num_free(s);
  if (num_waiting) *num_waiting = (int32_t)s->waiting.size();
  if (num_running) *num_running = (int32_t)s->running.size();
  return CB_OK;
}

cb_status cb_sched_swapped(const cb_sched* s, int64_t* out, int32_t capacity, int32_t* count,
                           int32_t* free_slots) {
  if (!s) return cb::fail(CB_ERR_INVALID_ARG, "scheduler is NULL");
  const int32_t n = (int32_t)s->swapped.size();
  if (count) *count = n;
  if (free_slots) *free_slots = (int32_t)s->swap_free.size();
  if (out)
    for (int32_t i = 0; i < std::min(n, capacity); ++i) out[i] = s->swapped[i]->id;
  return CB_OK;
}

cb_status cb_sched_free_list(const cb_sched* s, int32_t* out, int32_t capacity, int32_t* count) {
  if (!s) return cb::fail(CB_ERR_INVALID_ARG, "scheduler is NULL");
  const int32_t n = (int32_t)num_free(s);
  if (count) *count = n;
  if (out) {
    int32_t i = 0;
    for (int32_t b : s->free_list) {
      if (i >= capacity) break;
      out[i++] = b;
    }
    for (int32_t b : s->free_init) {
      if (i >= capacity) break;
      out[i++] = b;
    }
  }
  return CB_OK;
}

cb_status cb_sched_hold_blocks(cb_sched* s, int32_t n, int32_t* out_ids, int32_t* count) {
  if (!s || n < 0 || (n > 0 && !out_ids)) return cb::fail(CB_ERR_INVALID_ARG, "bad argument");
  if (s->step_open) return cb::fail(CB_ERR_STATE, "a step is open; call cb_step_done first");
  int32_t k = 0;
  while (k < n && num_free(s) > 0) {
    const int32_t b = alloc_block(s);
    s->held[b] = 1;
    out_ids[k++] = b;
  }
  if (count) *count = k;
  return CB_OK;
}

cb_status cb_sched_release_blocks(cb_sched* s, const int32_t* ids, int32_t n) {
  if (!s || n < 0 || (n > 0 && !ids)) return cb::fail(CB_ERR_INVALID_ARG, "bad argument");
  if (s->step_open) return cb::fail(CB_ERR_STATE, "a step is open; call cb_step_done first");
  std::vector<char> seen(s->held.size(), 0);
  for (int32_t i = 0; i < n; ++i) {
    const int32_t b = ids[i];
    if (b < 0 || b >= (int32_t)s->held.size() || !s->held[b] || seen[b])
      return cb::fail(CB_ERR_INVALID_ARG, "block %d is not held (or listed twice)", b);
    seen[b] = 1;
  }
  for (int32_t i = 0; i < n; ++i) {
    const int32_t b = ids[i];
    s->held[b] = 0;
    s->refs[b] = 0;
    s->free_list.push_back(b);
  }
  return CB_OK;
}

cb_status cb_sched_prefix_stats(const cb_sched* s, int64_t* hit_tokens, int32_t* keyed_blocks,
                                int32_t* pool_blocks) {
  if (!s) return cb::fail(CB_ERR_INVALID_ARG, "scheduler is NULL");
  if (hit_tokens) *hit_tokens = s->prefix_hits;
  if (keyed_blocks) *keyed_blocks = (int32_t)s->index.size();
  if (pool_blocks) *pool_blocks = (int32_t)s->free_init.size();
  return CB_OK;
}

}  // extern "C"
