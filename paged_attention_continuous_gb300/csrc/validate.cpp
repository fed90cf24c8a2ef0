// Host-side validation of a step's metadata.
//
// The kernels range-check what they read and report problems as device
// error bits; this check runs on the host, before any launch, and names
// the row and the problem.  It is the debugging mode of the GPU calls
// (CB_VALIDATE=1 copies their metadata back and checks it) and a plain C
// call for callers that hold the host arrays.  The rules are the ones the
// attention definition needs ("Chunked Prefill", How chunked prefill works;
// "vLLM serving internals", PagedAttention as a virtual memory system):
// query rows are consecutive runs of tokens, decode rows have one token, a
// row's keys are the seq_len positions its block table covers (from the
// window's first page with a sliding window), and every slot a token is
// written to lies in the pool.
#include "validate.h"

#include <algorithm>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "cb_error.h"

extern "C" cb_status cb_validate_step(const int32_t* cu_seqlens_q, const int32_t* seq_lens,
                                      const int32_t* block_tables, const int32_t* slot_mapping,
                                      int32_t num_reqs, int32_t num_decodes, int32_t num_tokens,
                                      int32_t max_blocks_per_seq, int32_t num_blocks,
                                      int32_t block_size, int32_t sliding_window) {
  using cb::fail;
  if (num_reqs < 0 || num_decodes < 0 || num_decodes > num_reqs || num_tokens < 0)
    return fail(CB_ERR_INVALID_ARG, "validate: bad row or token counts");
  if (max_blocks_per_seq <= 0 || num_blocks <= 0 || block_size <= 0 || sliding_window < 0)
    return fail(CB_ERR_INVALID_ARG, "validate: bad pool or table sizes");
  if (num_reqs > 0 && (!cu_seqlens_q || !seq_lens || !block_tables))
    return fail(CB_ERR_INVALID_ARG, "validate: NULL metadata array");
  if (num_reqs > 0 && cu_seqlens_q[0] < 0)
    return fail(CB_ERR_INVALID_ARG, "validate: cu_seqlens_q[0] = %d < 0", cu_seqlens_q[0]);
  for (int32_t i = 0; i < num_reqs; ++i) {
    const int32_t q0 = cu_seqlens_q[i], q1 = cu_seqlens_q[i + 1];
    const int32_t q_len = q1 - q0, L = seq_lens[i];
    if (q_len < 0)
      return fail(CB_ERR_INVALID_ARG, "validate: row %d: cu_seqlens_q decreases (%d -> %d)", i, q0, q1);
    if (q1 > num_tokens)
      return fail(CB_ERR_INVALID_ARG, "validate: row %d: queries end at %d > num_tokens %d", i, q1,
                  num_tokens);
    if (i < num_decodes && !(q_len == 1 || (q_len == 0 && L == 0)))
      return fail(CB_ERR_INVALID_ARG, "validate: decode row %d has %d query tokens", i, q_len);
    if (q_len == 0 && L == 0) continue;  // padding row
    if (q_len == 0) return fail(CB_ERR_INVALID_ARG, "validate: row %d: no queries but seq_len %d", i, L);
    if (L < q_len)
      return fail(CB_ERR_INVALID_ARG, "validate: row %d: seq_len %d < query length %d", i, L, q_len);
    const int64_t pages = ((int64_t)L + block_size - 1) / block_size;
    if (pages > max_blocks_per_seq)
      return fail(CB_ERR_INVALID_ARG, "validate: row %d: seq_len %d needs %lld blocks > %d", i, L,
                  (long long)pages, max_blocks_per_seq);
    // keys the row's first query can read: all, or its window
    const int64_t first_key =
        sliding_window > 0 ? std::max<int64_t>(0, (int64_t)L - q_len - sliding_window + 1) : 0;
    const int32_t* row = block_tables + (int64_t)i * max_blocks_per_seq;
    for (int64_t pg = first_key / block_size; pg < pages; ++pg)
      if (row[pg] < 0 || row[pg] >= num_blocks)
        return fail(CB_ERR_INVALID_ARG, "validate: row %d: block_tables[%lld] = %d outside [0, %d)", i,
                    (long long)pg, row[pg], num_blocks);
  }
  if (slot_mapping) {
    const int64_t slots = (int64_t)num_blocks * block_size;
    for (int32_t t = 0; t < num_tokens; ++t)
      if (slot_mapping[t] < -1 || slot_mapping[t] >= slots)
        return fail(CB_ERR_INVALID_ARG, "validate: slot_mapping[%d] = %d outside [-1, %lld)", t,
                    slot_mapping[t], (long long)slots);
  }
  return CB_OK;
}

namespace cb {

bool validate_enabled() {
  static bool on = false;
  static std::once_flag once;
  std::call_once(once, [] {
    const char* v = std::getenv("CB_VALIDATE");
    on = v && std::atoi(v) != 0;
  });
  return on;
}

namespace {

bool capturing(cudaStream_t stream) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &st) != cudaSuccess) return false;
  return st != cudaStreamCaptureStatusNone;
}

cb_status copy_back(std::vector<int32_t>* dst, const int32_t* src, size_t n, cudaStream_t stream) {
  dst->assign(n, 0);
  if (n == 0) return CB_OK;
  cudaError_t e = cudaMemcpyAsync(dst->data(), src, n * sizeof(int32_t), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return fail(CB_ERR_CUDA, "validate: copying metadata: %s", cudaGetErrorString(e));
  return CB_OK;
}

}  // namespace

cb_status validate_attention_call(const cb_attention_args& a, cudaStream_t stream) {
  if (capturing(stream)) return CB_OK;
  std::vector<int32_t> cu, sl, bt;
  cb_status st = copy_back(&cu, a.cu_seqlens_q, (size_t)a.num_reqs + 1, stream);
  if (st == CB_OK) st = copy_back(&sl, a.seq_lens, (size_t)a.num_reqs, stream);
  if (st == CB_OK)
    st = copy_back(&bt, a.block_tables, (size_t)a.num_reqs * (size_t)a.max_blocks_per_seq, stream);
  if (st != CB_OK) return st;
  return cb_validate_step(cu.data(), sl.data(), bt.data(), nullptr, a.num_reqs, a.num_decodes,
                          a.num_tokens, a.max_blocks_per_seq, a.num_blocks, a.block_size,
                          a.sliding_window);
}

cb_status validate_append_call(const int32_t* slot_mapping, int32_t num_tokens, int32_t num_blocks,
                               int32_t block_size, cudaStream_t stream) {
  if (capturing(stream)) return CB_OK;
  std::vector<int32_t> sm;
  cb_status st = copy_back(&sm, slot_mapping, (size_t)num_tokens, stream);
  if (st != CB_OK) return st;
  const int64_t slots = (int64_t)num_blocks * block_size;
  for (int32_t t = 0; t < num_tokens; ++t)
    if (sm[t] < -1 || sm[t] >= slots)
      return fail(CB_ERR_INVALID_ARG, "validate: slot_mapping[%d] = %d outside [-1, %lld)", t, sm[t],
                  (long long)slots);
  return CB_OK;
}

}  // namespace cb
