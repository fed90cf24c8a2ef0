// Host launcher template of the split-KV decode kernel (included by the
// per-dtype translation units decode_bf16.cu and decode_f32.cu).
#pragma once

#include <atomic>
#include <type_traits>

#include "cb_error.h"
#include "decode_attention.cuh"
#include "decode_launch.h"
#include "launch_common.h"
#include "tensor_map.h"

namespace cb {
namespace decode {

constexpr size_t kSmemLimit = 227 * 1024;

// The most warps per CTA (at most 8) whose stages fit the shared memory.
template <typename T, int D, int G, int kStages>
constexpr int warps_for() {
  int w = 8;
  while (w > 1 && sizeof(WarpSmem<T, D, G, kStages>) * w + kPlanSmemBytes + 1024 > kSmemLimit) --w;
  return w;
}

template <typename T, int D, int G, bool kWindow>
cb_status launch(const cb_attention_args& a, const Scratch& s, uint32_t* error_word,
                 cudaStream_t stream, After after) {
  constexpr int kStages = 2;
  constexpr int kWarps = warps_for<T, D, G, kStages>();
  constexpr size_t smem = smem_bytes<T, D, G, kWarps, kStages>();
  static_assert(smem <= kSmemLimit, "decode stages do not fit shared memory");
  auto kern = decode_kernel<T, D, G, kWarps, kStages, kWindow>;
  static std::atomic<uint8_t> attr_set[kMaxDevices];
  cb_status st = ensure_smem_attr(reinterpret_cast<const void*>(kern), smem, attr_set);
  if (st != CB_OK) return st;
  Params p{};
  if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    const int64_t rows = (int64_t)a.num_blocks * a.num_kv_heads * kPageTokens;
    if (rows >= ((int64_t)1 << 31))
      return fail(CB_ERR_UNSUPPORTED, "cache of %lld rows is too large for a tensor map", (long long)rows);
    st = cached_cache_map(&p.tmap_k, a.k_cache, rows, D);
    if (st != CB_OK) return st;
    st = cached_cache_map(&p.tmap_v, a.v_cache, rows, D);
    if (st != CB_OK) return st;
  }
  p.q = a.q;
  p.out = a.out;
  p.k_cache = a.k_cache;
  p.v_cache = a.v_cache;
  p.cu_seqlens_q = a.cu_seqlens_q;
  p.seq_lens = a.seq_lens;
  p.block_tables = a.block_tables;
  p.num_tokens = a.num_tokens;
  p.num_blocks = a.num_blocks;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.window = a.sliding_window;
  p.error_word = error_word;
  p.work_counter = s.work_counter;
  p.done = s.done;
  p.max_slots = (int32_t)(s.slots < (1 << 30) ? s.slots : (1 << 30));
  p.part_ml = s.part_ml;
  p.part_acc = s.part_acc;
  p.wait_ns = wait_limit_ns();
  p.withhold_item = withheld_decode_item();
  const int grid = sm_count_current_device();
  for (int r0 = 0; r0 < a.num_decodes; r0 += kPlanMax) {
    p.row_begin = r0;
    p.num_rows = a.num_decodes - r0 < kPlanMax ? a.num_decodes - r0 : kPlanMax;
    // the first launch may overlap the kernel queued just before it (After);
    // later launches share this call's workspace with the one before and
    // follow it fully
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute lattr[1];
    lattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    const After mode = r0 == 0 ? after : After::kStream;
    p.pdl_mode = (int32_t)mode;
    lattr[0].val.programmaticStreamSerializationAllowed = mode != After::kStream ? 1 : 0;
    cfg.attrs = lattr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(CB_ERR_CUDA, "decode kernel launch: %s", cudaGetErrorString(e));
  }
  return CB_OK;
}

}  // namespace decode
}  // namespace cb
