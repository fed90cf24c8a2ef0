// cb_paged_attention: argument checks, workspace layout and kernel dispatch.
//
// Rows [0, num_decodes) of a step are decodes (one query token each) and run
// the split-KV decode kernel; the remaining rows (prefill chunks) run the
// prefill-chunk kernel.  Shapes outside the specialised kernels run the
// row-generic CUDA-core kernel.
#include <cuda_runtime.h>

#include "cb_error.h"
#include "decode_launch.h"
#include "device_utils.cuh"
#include "launch_common.h"
#include "prefill_dispatch.h"
#include "simt_attention.cuh"
#include "validate.h"

namespace cb {

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct WsLayout {
  size_t header = 0, counters = 0, prefill = 0, part_ml = 0, part_acc = 0, total = 0;
  int64_t slots = 0;  // decode partial slots
};

// Workspace regions.  The header, the decode split tickets and the prefill
// region hold state that must read zero at the start of every call (each
// call leaves them zero), so they sit at FIXED offsets that do not depend on
// the call's sizes.  The split partials are scratch rewritten by every call,
// sized by the call's decode rows.
//   header words: [0] device error bits, [1] decode item counter
//   counters: done[kPlanMax * kMaxKvHeads] (one ticket counter per
//             (decode row, KV head) of a launch)
constexpr int64_t kMaxKvHeads = 64;
constexpr int kPlanMax = decode::kPlanMax;
constexpr size_t kCounterWords = (size_t)kPlanMax * kMaxKvHeads;

WsLayout ws_layout(int64_t num_reqs, int64_t Hq, int64_t Hkv, int64_t D) {
  WsLayout w;
  const int64_t rows = num_reqs < kPlanMax ? num_reqs : kPlanMax;
  w.header = 0;
  w.counters = kAlign;
  w.prefill = w.counters + align_up(kCounterWords * 4);
  w.part_ml = w.prefill + align_up(prefill_workspace_bytes(Hq, Hkv, D));
  const size_t slots = (size_t)decode::partial_slots(rows, Hkv);
  w.part_acc = w.part_ml + align_up(slots * Hq * 2 * 4);
  w.total = w.part_acc + align_up(slots * Hq * D * 4);
  w.slots = (int64_t)slots;
  return w;
}

decode::Scratch decode_scratch(const cb_attention_args& a, const WsLayout& L) {
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  decode::Scratch s{};
  s.work_counter = reinterpret_cast<uint32_t*>(ws + L.header) + 1;
  s.done = reinterpret_cast<uint32_t*>(ws + L.counters);
  s.part_ml = reinterpret_cast<float*>(ws + L.part_ml);
  s.part_acc = reinterpret_cast<float*>(ws + L.part_acc);
  s.slots = L.slots;
  return s;
}

template <typename T, int D>
cb_status launch_simt_rows(const cb_attention_args& a, const WsLayout& L, int row_begin,
                           int row_end, int tok_begin, int tok_end, cudaStream_t stream) {
  if (row_end <= row_begin || tok_end <= tok_begin) return CB_OK;
  simt::Params p{};
  p.q = a.q;
  p.out = a.out;
  p.k_cache = a.k_cache;
  p.v_cache = a.v_cache;
  p.cu_seqlens_q = a.cu_seqlens_q;
  p.seq_lens = a.seq_lens;
  p.block_tables = a.block_tables;
  p.row_begin = row_begin;
  p.row_end = row_end;
  p.tok_begin = tok_begin;
  p.tok_end = tok_end;
  p.num_blocks = a.num_blocks;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.block_size = a.block_size;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.window = a.sliding_window;
  p.error_word = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(a.workspace) + L.header);
  const int64_t warps = (int64_t)(tok_end - tok_begin) * a.num_q_heads;
  const int64_t blocks = (warps + 7) / 8;
  simt::rows_kernel<T, D><<<(unsigned)blocks, 256, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(CB_ERR_CUDA, "simt kernel launch: %s", cudaGetErrorString(e));
  return CB_OK;
}

template <typename T>
cb_status dispatch_simt(const cb_attention_args& a, const WsLayout& L, int row_begin, int row_end,
                        int tok_begin, int tok_end, cudaStream_t s) {
  if (a.head_dim == 64) return launch_simt_rows<T, 64>(a, L, row_begin, row_end, tok_begin, tok_end, s);
  if (a.head_dim == 128) return launch_simt_rows<T, 128>(a, L, row_begin, row_end, tok_begin, tok_end, s);
  return fail(CB_ERR_UNSUPPORTED, "head_dim %d not supported", a.head_dim);
}

}  // namespace

}  // namespace cb

using cb::fail;

extern "C" size_t cb_attention_workspace_size(int32_t num_reqs, int32_t num_q_heads,
                                              int32_t num_kv_heads, int32_t head_dim) {
  if (num_reqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0) return 0;
  return cb::ws_layout(num_reqs > 0 ? num_reqs : 1, num_q_heads, num_kv_heads, head_dim).total;
}

extern "C" cb_status cb_attention_workspace_init(void* workspace, size_t workspace_bytes,
                                                 cb_stream_t stream) {
  if (!workspace || workspace_bytes == 0) return fail(CB_ERR_INVALID_ARG, "workspace is NULL");
  cudaError_t e = cudaMemsetAsync(workspace, 0, workspace_bytes, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(CB_ERR_CUDA, "workspace memset: %s", cudaGetErrorString(e));
  return CB_OK;
}

extern "C" cb_status cb_attention_read_errors(void* workspace, size_t workspace_bytes,
                                              cb_stream_t stream, uint32_t* bits) {
  if (!workspace || workspace_bytes < 4) return fail(CB_ERR_INVALID_ARG, "workspace is NULL");
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, workspace, 4, cudaMemcpyDeviceToHost, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e == cudaSuccess && v != 0) e = cudaMemsetAsync(workspace, 0, 4, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return fail(CB_ERR_CUDA, "reading device errors: %s", cudaGetErrorString(e));
  if (bits) *bits = v;
  if (v != 0) return fail(CB_ERR_DEVICE_CHECK, "device error bits 0x%x", v);
  return CB_OK;
}

extern "C" cb_status cb_paged_attention(const cb_attention_args* args, cb_stream_t stream_) {
  if (!args) return fail(CB_ERR_INVALID_ARG, "args is NULL");
  const cb_attention_args& a = *args;
  cudaStream_t stream = (cudaStream_t)stream_;
  if (a.num_reqs < 0 || a.num_decodes < 0 || a.num_decodes > a.num_reqs || a.num_tokens < 0)
    return fail(CB_ERR_INVALID_ARG, "bad row/token counts");
  if (a.num_reqs == 0 || a.num_tokens == 0) return CB_OK;
  if (!a.q || !a.out || !a.k_cache || !a.v_cache || !a.cu_seqlens_q || !a.seq_lens ||
      !a.block_tables || !a.workspace)
    return fail(CB_ERR_INVALID_ARG, "NULL pointer argument");
  if (a.num_tokens < a.num_reqs) return fail(CB_ERR_INVALID_ARG, "num_tokens < num_reqs");
  if (a.num_q_heads <= 0 || a.num_kv_heads <= 0 || a.num_q_heads % a.num_kv_heads != 0)
    return fail(CB_ERR_INVALID_ARG, "num_q_heads must be a positive multiple of num_kv_heads");
  if (a.num_kv_heads > cb::kMaxKvHeads)
    return fail(CB_ERR_UNSUPPORTED, "num_kv_heads > %d", (int)cb::kMaxKvHeads);
  if (a.block_size != 16) return fail(CB_ERR_UNSUPPORTED, "block_size must be 16");
  if (a.head_dim != 64 && a.head_dim != 128) return fail(CB_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (a.dtype != CB_DTYPE_F32 && a.dtype != CB_DTYPE_BF16) return fail(CB_ERR_INVALID_ARG, "unknown dtype");
  if (a.num_blocks <= 0 || a.max_blocks_per_seq <= 0) return fail(CB_ERR_INVALID_ARG, "bad pool sizes");
  if (a.sliding_window < 0) return fail(CB_ERR_INVALID_ARG, "sliding_window must be >= 0");
  if (a.max_q_len < 1 || a.max_seq_len < a.max_q_len ||
      (a.max_seq_len + a.block_size - 1) / a.block_size > a.max_blocks_per_seq)
    return fail(CB_ERR_INVALID_ARG, "max_q_len / max_seq_len inconsistent with the block table");
  const uintptr_t al = (uintptr_t)a.q | (uintptr_t)a.out | (uintptr_t)a.k_cache | (uintptr_t)a.v_cache;
  if (al & 15u) return fail(CB_ERR_INVALID_ARG, "q/out/cache pointers must be 16-byte aligned");
  if ((uintptr_t)a.workspace & (cb::kAlign - 1))
    return fail(CB_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  const cb::WsLayout L = cb::ws_layout(a.num_reqs, a.num_q_heads, a.num_kv_heads, a.head_dim);
  if (a.workspace_bytes < L.total)
    return fail(CB_ERR_INVALID_ARG, "workspace too small: %zu < %zu", a.workspace_bytes, L.total);

  if (cb::validate_enabled()) {
    cb_status vs = cb::validate_attention_call(a, stream);
    if (vs != CB_OK) return vs;
  }
  const int nd = a.num_decodes;
  const int G = a.num_q_heads / a.num_kv_heads;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  uint32_t* ew = reinterpret_cast<uint32_t*>(ws + L.header);
  const bool tc_prefill = nd < a.num_reqs && a.dtype == CB_DTYPE_BF16 && a.head_dim == 128 &&
                          cb::prefill_supported(G);
  auto run_decode = [&](cb::decode::After after) -> cb_status {
    const cb::decode::Scratch ds = cb::decode_scratch(a, L);
    cb_status s = a.dtype == CB_DTYPE_BF16 ? cb::decode::dispatch_bf16(a, ds, ew, stream, after)
                                           : cb::decode::dispatch_f32(a, ds, ew, stream, after);
    if (s == CB_ERR_UNSUPPORTED) {
      s = a.dtype == CB_DTYPE_BF16 ? cb::dispatch_simt<__nv_bfloat16>(a, L, 0, nd, 0, nd, stream)
                                   : cb::dispatch_simt<float>(a, L, 0, nd, 0, nd, stream);
    }
    return s;
  };
  // Order of the two kernels (they share no data).  Normally the decode rows
  // go first and the prefill grid starts on the SMs the decode kernel frees
  // as it ends.  When the prefill grid leaves SMs idle for its whole length
  // (at least 16 fewer CTAs than SMs) and its CTAs are long (the longest row
  // holds 16k keys or more), the prefill rows go first and the decode
  // kernel runs beside them on the idle SMs (programmatic dependent launch).
  if (nd > 0 && tc_prefill && a.max_seq_len >= 16384 &&
      cb::prefill_ctas(a) + 16 <= cb::sm_count_current_device()) {
    cb_status st = cb::launch_prefill_bf16(a, ew, ws + L.prefill, stream, false);
    if (st == CB_OK) return run_decode(cb::decode::After::kPrefill);
    if (st != CB_ERR_UNSUPPORTED) return st;
  }
  cb_status st = CB_OK;
  if (nd > 0) {
    st = run_decode(a.after_append ? cb::decode::After::kAppend : cb::decode::After::kStream);
    if (st != CB_OK) return st;
  }
  if (nd < a.num_reqs) {
    // decode rows hold exactly one token each, so prefill tokens start at nd
    if (tc_prefill) {
      // the decode kernel just queued (if any) reads and writes nothing the
      // prefill rows use: let the prefill grid start on the SMs it frees
      st = cb::launch_prefill_bf16(a, ew, ws + L.prefill, stream, nd > 0);
      if (st != CB_ERR_UNSUPPORTED) return st;
    }
    st = a.dtype == CB_DTYPE_BF16
             ? cb::dispatch_simt<__nv_bfloat16>(a, L, nd, a.num_reqs, nd, a.num_tokens, stream)
             : cb::dispatch_simt<float>(a, L, nd, a.num_reqs, nd, a.num_tokens, stream);
  }
  return st;
}
