// cb_executor: one serving step behind one C call, double-buffered.
//
// "Continuous batching architecture", Async batching: while the device
// computes step N, the host schedules step N+1 and that step's inputs cross
// the CPU-GPU link, and step N-1's output comes back.  An executor owns two
// sets of device input/output buffers (q, k_new, v_new, out per layer, and
// the packed metadata), a pinned staging buffer per set, and three streams:
// copy-in, compute and copy-out.  A step (cb_executor_submit) packs the
// scheduler's host metadata into the set's pinned staging buffer, then
// queues
//   copy-in stream:  wait until the set's previous compute finished; the
//                    metadata and every layer's q/k/v rows, host -> device;
//   compute stream:  wait for that copy and for the set's previous copy-out;
//                    per layer cb_kv_append + cb_paged_attention;
//   copy-out stream: wait for the compute; every layer's output rows,
//                    device -> host;
// and returns without waiting, so the host can schedule the next step.  The
// sets are used in turn, so one step's copies overlap its neighbours'
// compute.  cb_executor_run_step also calls the scheduler: it schedules the
// next step, submits it and commits it (cb_step_done; the scheduler's state
// is host-only and the device work of the step does not depend on it).
#include <cuda_runtime.h>

#include <cstring>
#include <vector>

#include "../../include/cb.h"
#include "cb_error.h"

using cb::fail;

struct cb_executor {
  cb_executor_config cfg{};
  std::vector<void*> k_caches, v_caches;
  size_t elem = 2;
  int64_t meta_words = 0;
  cudaStream_t in_s = nullptr, comp_s = nullptr, out_s = nullptr;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  uint32_t* append_err = nullptr;  // device word for cb_kv_append
  struct Set {
    int32_t* meta_dev = nullptr;
    int32_t* meta_host = nullptr;  // pinned
    std::vector<void*> q, k, v, o;
    cudaEvent_t copied_in = nullptr, computed = nullptr, copied_out = nullptr;
    bool used = false;
  } sets[2];
  int turn = 0;
  // per-step compute timing (CUDA events on the compute stream)
  std::vector<cudaEvent_t> free_events;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> pending;
  double compute_ms = 0.0;
  int64_t steps = 0, tokens = 0;
};

namespace {

void release(cb_executor* ex) {
  if (!ex) return;
  if (ex->comp_s) cudaStreamSynchronize(ex->comp_s);
  if (ex->in_s) cudaStreamSynchronize(ex->in_s);
  if (ex->out_s) cudaStreamSynchronize(ex->out_s);
  for (auto& s : ex->sets) {
    if (s.meta_dev) cudaFree(s.meta_dev);
    if (s.meta_host) cudaFreeHost(s.meta_host);
    for (auto* vec : {&s.q, &s.k, &s.v, &s.o})
      for (void* p : *vec)
        if (p) cudaFree(p);
    for (cudaEvent_t e : {s.copied_in, s.computed, s.copied_out})
      if (e) cudaEventDestroy(e);
  }
  for (auto& pr : ex->pending) {
    cudaEventDestroy(pr.first);
    cudaEventDestroy(pr.second);
  }
  for (cudaEvent_t e : ex->free_events) cudaEventDestroy(e);
  if (ex->ws) cudaFree(ex->ws);
  if (ex->append_err) cudaFree(ex->append_err);
  for (cudaStream_t s : {ex->in_s, ex->comp_s, ex->out_s})
    if (s) cudaStreamDestroy(s);
  delete ex;
}

cudaEvent_t timing_event(cb_executor* ex) {
  if (!ex->free_events.empty()) {
    cudaEvent_t e = ex->free_events.back();
    ex->free_events.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Sum the compute time of finished steps (all of them when `all`).
void collect_timing(cb_executor* ex, bool all) {
  size_t keep = 0;
  for (size_t i = 0; i < ex->pending.size(); ++i) {
    auto pr = ex->pending[i];
    float ms = 0.f;
    const cudaError_t e = all ? cudaEventSynchronize(pr.second) : cudaEventQuery(pr.second);
    if (e == cudaSuccess && cudaEventElapsedTime(&ms, pr.first, pr.second) == cudaSuccess) {
      ex->compute_ms += ms;
      ex->free_events.push_back(pr.first);
      ex->free_events.push_back(pr.second);
    } else {
      ex->pending[keep++] = pr;
    }
  }
  ex->pending.resize(keep);
}

}  // namespace

extern "C" cb_status cb_executor_create(const cb_executor_config* cfg, cb_executor** out) {
  if (!out) return fail(CB_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!cfg) return fail(CB_ERR_INVALID_ARG, "config is NULL");
  const cb_executor_config& c = *cfg;
  if (c.num_layers < 1 || !c.k_caches || !c.v_caches)
    return fail(CB_ERR_INVALID_ARG, "need at least one layer and its caches");
  if (c.max_reqs < 1 || c.max_tokens < 1 || c.max_blocks_per_seq < 1 || c.num_blocks < 1)
    return fail(CB_ERR_INVALID_ARG, "bad sizes");
  if (c.num_q_heads <= 0 || c.num_kv_heads <= 0 || c.num_q_heads % c.num_kv_heads != 0 ||
      c.head_dim <= 0 || c.block_size <= 0)
    return fail(CB_ERR_INVALID_ARG, "bad head sizes");
  if (c.dtype != CB_DTYPE_BF16 && c.dtype != CB_DTYPE_F32) return fail(CB_ERR_INVALID_ARG, "unknown dtype");
  for (int l = 0; l < c.num_layers; ++l)
    if (!c.k_caches[l] || !c.v_caches[l]) return fail(CB_ERR_INVALID_ARG, "NULL cache of layer %d", l);
  cb_executor* ex = new cb_executor();
  ex->cfg = c;
  ex->k_caches.assign(c.k_caches, c.k_caches + c.num_layers);
  ex->v_caches.assign(c.v_caches, c.v_caches + c.num_layers);
  ex->cfg.k_caches = ex->k_caches.data();
  ex->cfg.v_caches = ex->v_caches.data();
  ex->elem = c.dtype == CB_DTYPE_BF16 ? 2 : 4;
  ex->meta_words = (int64_t)(c.max_reqs + 1) + c.max_reqs + (int64_t)c.max_reqs * c.max_blocks_per_seq +
                   c.max_tokens;
  cudaError_t e = cudaSuccess;
  auto ok = [&](cudaError_t r) {
    if (r != cudaSuccess && e == cudaSuccess) e = r;
    return r == cudaSuccess;
  };
  ok(cudaStreamCreateWithFlags(&ex->in_s, cudaStreamNonBlocking));
  ok(cudaStreamCreateWithFlags(&ex->comp_s, cudaStreamNonBlocking));
  ok(cudaStreamCreateWithFlags(&ex->out_s, cudaStreamNonBlocking));
  ex->ws_bytes = cb_attention_workspace_size(c.max_reqs, c.num_q_heads, c.num_kv_heads, c.head_dim);
  if (ex->ws_bytes == 0) {
    release(ex);
    return fail(CB_ERR_INVALID_ARG, "workspace size");
  }
  ok(cudaMalloc(&ex->ws, ex->ws_bytes));
  ok(cudaMalloc(reinterpret_cast<void**>(&ex->append_err), 4));
  const size_t q_bytes = (size_t)c.max_tokens * c.num_q_heads * c.head_dim * ex->elem;
  const size_t kv_bytes = (size_t)c.max_tokens * c.num_kv_heads * c.head_dim * ex->elem;
  for (auto& s : ex->sets) {
    ok(cudaMalloc(reinterpret_cast<void**>(&s.meta_dev), ex->meta_words * 4));
    ok(cudaHostAlloc(reinterpret_cast<void**>(&s.meta_host), ex->meta_words * 4, cudaHostAllocDefault));
    for (int l = 0; l < c.num_layers; ++l) {
      void *q = nullptr, *k = nullptr, *v = nullptr, *o = nullptr;
      ok(cudaMalloc(&q, q_bytes));
      ok(cudaMalloc(&k, kv_bytes));
      ok(cudaMalloc(&v, kv_bytes));
      ok(cudaMalloc(&o, q_bytes));
      s.q.push_back(q);
      s.k.push_back(k);
      s.v.push_back(v);
      s.o.push_back(o);
    }
    ok(cudaEventCreateWithFlags(&s.copied_in, cudaEventDisableTiming));
    ok(cudaEventCreateWithFlags(&s.computed, cudaEventDisableTiming));
    ok(cudaEventCreateWithFlags(&s.copied_out, cudaEventDisableTiming));
  }
  if (e == cudaSuccess) {
    ok(cudaMemsetAsync(ex->append_err, 0, 4, ex->comp_s));
    cb_status st = cb_attention_workspace_init(ex->ws, ex->ws_bytes, (cb_stream_t)ex->comp_s);
    if (st != CB_OK) {
      release(ex);
      return st;
    }
    ok(cudaStreamSynchronize(ex->comp_s));
  }
  if (e != cudaSuccess) {
    release(ex);
    return fail(CB_ERR_CUDA, "executor set-up: %s", cudaGetErrorString(e));
  }
  *out = ex;
  return CB_OK;
}

extern "C" void cb_executor_destroy(cb_executor* ex) { release(ex); }

extern "C" cb_status cb_executor_submit(cb_executor* ex, const cb_step* step,
                                        const void* const* q_host, const void* const* k_host,
                                        const void* const* v_host, void* const* out_host) {
  if (!ex || !step) return fail(CB_ERR_INVALID_ARG, "NULL executor or step");
  const cb_executor_config& c = ex->cfg;
  const int R = step->num_reqs, T = step->num_tokens, W = c.max_blocks_per_seq;
  if (R == 0 || T == 0) return CB_OK;
  if (R < 0 || T < 0 || R > c.max_reqs || T > c.max_tokens)
    return fail(CB_ERR_INVALID_ARG, "step of %d rows / %d tokens exceeds the executor (%d / %d)", R, T,
                c.max_reqs, c.max_tokens);
  if (step->max_blocks_per_seq != W)
    return fail(CB_ERR_INVALID_ARG, "block table width %d differs from the executor's %d",
                step->max_blocks_per_seq, W);
  if (step->num_swap_in > 0 || step->num_swap_out > 0)
    return fail(CB_ERR_UNSUPPORTED, "the executor does not move offloaded blocks (step carries swaps)");
  if (!q_host || !k_host || !v_host || !out_host) return fail(CB_ERR_INVALID_ARG, "NULL host buffers");
  for (int l = 0; l < c.num_layers; ++l)
    if (!q_host[l] || !k_host[l] || !v_host[l] || !out_host[l])
      return fail(CB_ERR_INVALID_ARG, "NULL host buffer of layer %d", l);
  cb_executor::Set& s = ex->sets[ex->turn];
  ex->turn ^= 1;
  cudaError_t e = cudaSuccess;
  // the set's staging buffer is free once its previous copy-in has run
  if (s.used) e = cudaEventSynchronize(s.copied_in);
  if (e != cudaSuccess) return fail(CB_ERR_CUDA, "waiting for a staging buffer: %s", cudaGetErrorString(e));
  int32_t* h = s.meta_host;
  const int64_t o1 = R + 1, o2 = o1 + R, o3 = o2 + (int64_t)R * W;
  std::memcpy(h, step->cu_seqlens_q, sizeof(int32_t) * (R + 1));
  std::memcpy(h + o1, step->seq_lens, sizeof(int32_t) * R);
  std::memcpy(h + o2, step->block_tables, sizeof(int32_t) * (size_t)R * W);
  std::memcpy(h + o3, step->slot_mapping, sizeof(int32_t) * T);
  const int64_t words = o3 + T;
  const size_t qb = (size_t)T * c.num_q_heads * c.head_dim * ex->elem;
  const size_t kvb = (size_t)T * c.num_kv_heads * c.head_dim * ex->elem;
  auto chk = [&](cudaError_t r) {
    if (r != cudaSuccess && e == cudaSuccess) e = r;
  };
  // copy-in: after the set's previous compute (its device inputs are free)
  if (s.used) chk(cudaStreamWaitEvent(ex->in_s, s.computed, 0));
  chk(cudaMemcpyAsync(s.meta_dev, h, words * 4, cudaMemcpyHostToDevice, ex->in_s));
  for (int l = 0; l < c.num_layers; ++l) {
    chk(cudaMemcpyAsync(s.q[l], q_host[l], qb, cudaMemcpyHostToDevice, ex->in_s));
    chk(cudaMemcpyAsync(s.k[l], k_host[l], kvb, cudaMemcpyHostToDevice, ex->in_s));
    chk(cudaMemcpyAsync(s.v[l], v_host[l], kvb, cudaMemcpyHostToDevice, ex->in_s));
  }
  chk(cudaEventRecord(s.copied_in, ex->in_s));
  // compute: after the copy-in and after the set's previous copy-out
  chk(cudaStreamWaitEvent(ex->comp_s, s.copied_in, 0));
  if (s.used) chk(cudaStreamWaitEvent(ex->comp_s, s.copied_out, 0));
  if (e != cudaSuccess) return fail(CB_ERR_CUDA, "queueing step copies: %s", cudaGetErrorString(e));
  cudaEvent_t t0 = timing_event(ex), t1 = timing_event(ex);
  if (t0) cudaEventRecord(t0, ex->comp_s);
  int max_q = 1, max_seq = 1;
  for (int r = 0; r < R; ++r) {
    const int ql = step->cu_seqlens_q[r + 1] - step->cu_seqlens_q[r];
    if (ql > max_q) max_q = ql;
    if (step->seq_lens[r] > max_seq) max_seq = step->seq_lens[r];
  }
  cb_attention_args a{};
  a.cu_seqlens_q = s.meta_dev;
  a.seq_lens = s.meta_dev + o1;
  a.block_tables = s.meta_dev + o2;
  a.num_reqs = R;
  a.num_decodes = step->num_decodes;
  a.num_tokens = T;
  a.max_q_len = max_q;
  a.max_seq_len = max_seq;
  a.num_blocks = c.num_blocks;
  a.max_blocks_per_seq = W;
  a.block_size = c.block_size;
  a.num_q_heads = c.num_q_heads;
  a.num_kv_heads = c.num_kv_heads;
  a.head_dim = c.head_dim;
  a.scale = c.scale;
  a.dtype = c.dtype;
  a.workspace = ex->ws;
  a.workspace_bytes = ex->ws_bytes;
  a.sliding_window = c.sliding_window;
  a.after_append = 1;  // each layer's attention follows its append on comp_s
  for (int l = 0; l < c.num_layers; ++l) {
    cb_status st = cb_kv_append(s.k[l], s.v[l], s.meta_dev + o3, T, ex->k_caches[l], ex->v_caches[l],
                                c.num_blocks, c.num_kv_heads, c.head_dim, c.block_size, c.dtype,
                                ex->append_err, (cb_stream_t)ex->comp_s);
    if (st != CB_OK) return st;
    a.q = s.q[l];
    a.out = s.o[l];
    a.k_cache = ex->k_caches[l];
    a.v_cache = ex->v_caches[l];
    st = cb_paged_attention(&a, (cb_stream_t)ex->comp_s);
    if (st != CB_OK) return st;
  }
  if (t1) cudaEventRecord(t1, ex->comp_s);
  if (t0 && t1) ex->pending.emplace_back(t0, t1);
  chk(cudaEventRecord(s.computed, ex->comp_s));
  // copy-out: after the compute
  chk(cudaStreamWaitEvent(ex->out_s, s.computed, 0));
  for (int l = 0; l < c.num_layers; ++l)
    chk(cudaMemcpyAsync(out_host[l], s.o[l], qb, cudaMemcpyDeviceToHost, ex->out_s));
  chk(cudaEventRecord(s.copied_out, ex->out_s));
  if (e != cudaSuccess) return fail(CB_ERR_CUDA, "queueing the step: %s", cudaGetErrorString(e));
  s.used = true;
  ex->steps += 1;
  ex->tokens += T;
  if (ex->pending.size() > 64) collect_timing(ex, false);
  return CB_OK;
}

extern "C" cb_status cb_executor_run_step(cb_executor* ex, cb_sched* sched,
                                          const void* const* q_host, const void* const* k_host,
                                          const void* const* v_host, void* const* out_host,
                                          int32_t* num_tokens, int32_t* num_reqs) {
  if (num_tokens) *num_tokens = 0;
  if (num_reqs) *num_reqs = 0;
  if (!ex || !sched) return fail(CB_ERR_INVALID_ARG, "NULL executor or scheduler");
  cb_step step{};
  cb_status st = cb_schedule_step(sched, &step);
  if (st != CB_OK) return st;
  if (step.num_reqs > 0) {
    st = cb_executor_submit(ex, &step, q_host, k_host, v_host, out_host);
    if (st != CB_OK) return st;
  }
  if (num_tokens) *num_tokens = step.num_tokens;
  if (num_reqs) *num_reqs = step.num_reqs;
  return cb_step_done(sched, nullptr, nullptr);
}

extern "C" cb_status cb_executor_synchronize(cb_executor* ex) {
  if (!ex) return fail(CB_ERR_INVALID_ARG, "NULL executor");
  cudaError_t e = cudaStreamSynchronize(ex->in_s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(ex->comp_s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(ex->out_s);
  if (e != cudaSuccess) return fail(CB_ERR_CUDA, "executor synchronize: %s", cudaGetErrorString(e));
  collect_timing(ex, true);
  return CB_OK;
}

extern "C" cb_status cb_executor_stats(cb_executor* ex, int64_t* steps, int64_t* tokens,
                                       double* compute_ms) {
  if (!ex) return fail(CB_ERR_INVALID_ARG, "NULL executor");
  collect_timing(ex, false);
  if (steps) *steps = ex->steps;
  if (tokens) *tokens = ex->tokens;
  if (compute_ms) *compute_ms = ex->compute_ms;
  return CB_OK;
}

extern "C" cb_status cb_executor_reset_stats(cb_executor* ex) {
  if (!ex) return fail(CB_ERR_INVALID_ARG, "NULL executor");
  collect_timing(ex, true);
  ex->steps = 0;
  ex->tokens = 0;
  ex->compute_ms = 0.0;
  return CB_OK;
}

extern "C" cb_status cb_executor_read_errors(cb_executor* ex, uint32_t* bits) {
  if (!ex) return fail(CB_ERR_INVALID_ARG, "NULL executor");
  cb_status st = cb_executor_synchronize(ex);
  if (st != CB_OK) return st;
  uint32_t attn = 0, app = 0;
  st = cb_attention_read_errors(ex->ws, ex->ws_bytes, (cb_stream_t)ex->comp_s, &attn);
  if (st != CB_OK && st != CB_ERR_DEVICE_CHECK) return st;
  cudaError_t e = cudaMemcpy(&app, ex->append_err, 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && app != 0) e = cudaMemset(ex->append_err, 0, 4);
  if (e != cudaSuccess) return fail(CB_ERR_CUDA, "reading executor errors: %s", cudaGetErrorString(e));
  if (bits) *bits = attn | app;
  if (attn | app) return fail(CB_ERR_DEVICE_CHECK, "device error bits 0x%x", attn | app);
  return CB_OK;
}
