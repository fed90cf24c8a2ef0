// cb_kv_append: scatter a step's new K/V rows into the paged cache.
//
// "vLLM serving internals", PagedAttention as a virtual memory system: the KV
// cache is a pool of fixed-size blocks; a token at logical position pos of a
// sequence lives in physical block block_table[pos / block_size] at offset
// pos % block_size.  The scheduler has already turned that into one slot per
// new token (slot = block * block_size + offset); this kernel is the copy.
//
// Layout: new rows [T][Hkv][D]; cache [num_blocks][Hkv][block_size][D].  Each
// thread moves one 16-byte vector of K and the matching one of V: loads are
// fully coalesced over (t, h, vector), and each (t, h) row lands as
// D*elem contiguous bytes in the cache.  The row loads are issued before the
// slot lookup they do not depend on.
#include <cuda_runtime.h>

#include "cb_error.h"
#include "validate.h"
#include "device_utils.cuh"

namespace cb {

__global__ void __launch_bounds__(256) kv_append_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
    const int32_t* __restrict__ slot_mapping, int32_t num_tokens, uint4* __restrict__ k_cache,
    uint4* __restrict__ v_cache, int64_t num_slots, int32_t num_kv_heads, int32_t vec_shift,
    int32_t block_shift, int32_t block_mask, uint32_t* error_word) {
  // the attention launch that follows (when it asks for it) may start now;
  // it reads the cache only after this grid has completed
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // 32-bit indices (the host checks that they fit): thread i moves vector c
  // of row (t, h) = i >> vec_shift
  const int32_t total = (num_tokens * num_kv_heads) << vec_shift;
  const int32_t vec_mask = (1 << vec_shift) - 1;
  for (int32_t i = (int32_t)(blockIdx.x * blockDim.x + threadIdx.x); i < total;
       i += (int32_t)(gridDim.x * blockDim.x)) {
    const int32_t row = i >> vec_shift;
    const int32_t c = i & vec_mask;
    const int32_t t = row / num_kv_heads;
    const int32_t h = row - t * num_kv_heads;
    const uint4 kv = __ldg(k_new + i);
    const uint4 vv = __ldg(v_new + i);
    const int32_t slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;
    if ((int64_t)slot >= num_slots) {
      set_error(error_word, CB_DEVERR_SLOT_RANGE);
      continue;
    }
    const int64_t block = slot >> block_shift;
    const int32_t off = slot & block_mask;
    const int64_t dst = ((((block * num_kv_heads + h) << block_shift) + off) << vec_shift) + c;
    k_cache[dst] = kv;
    v_cache[dst] = vv;
  }
}

}  // namespace cb

extern "C" cb_status cb_kv_append(const void* k_new, const void* v_new,
                                  const int32_t* slot_mapping, int32_t num_tokens, void* k_cache,
                                  void* v_cache, int32_t num_blocks, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t block_size, cb_dtype dtype,
                                  uint32_t* error_word, cb_stream_t stream) {
  if (num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0)
    return cb::fail(CB_ERR_INVALID_ARG, "cb_kv_append: sizes must be positive");
  if (num_tokens == 0) return CB_OK;
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache)
    return cb::fail(CB_ERR_INVALID_ARG, "cb_kv_append: NULL pointer");
  if (dtype != CB_DTYPE_F32 && dtype != CB_DTYPE_BF16)
    return cb::fail(CB_ERR_INVALID_ARG, "cb_kv_append: unknown dtype");
  if ((block_size & (block_size - 1)) != 0)
    return cb::fail(CB_ERR_UNSUPPORTED, "cb_kv_append: block_size must be a power of two");
  const int elem = dtype == CB_DTYPE_F32 ? 4 : 2;
  const int row_bytes = head_dim * elem;
  if (row_bytes % 16 != 0)
    return cb::fail(CB_ERR_UNSUPPORTED, "cb_kv_append: head_dim*elem must be a multiple of 16");
  const int vecs = row_bytes / 16;
  if ((vecs & (vecs - 1)) != 0)
    return cb::fail(CB_ERR_UNSUPPORTED, "cb_kv_append: head_dim*elem/16 must be a power of two");
  if ((int64_t)num_tokens * num_kv_heads * vecs >= ((int64_t)1 << 31))
    return cb::fail(CB_ERR_UNSUPPORTED, "cb_kv_append: more than 2^31 16-byte vectors in one call");
  const uintptr_t align = (uintptr_t)k_new | (uintptr_t)v_new | (uintptr_t)k_cache | (uintptr_t)v_cache;
  if (align & 15u) return cb::fail(CB_ERR_INVALID_ARG, "cb_kv_append: pointers must be 16-byte aligned");
  if (cb::validate_enabled()) {
    cb_status vs = cb::validate_append_call(slot_mapping, num_tokens, num_blocks, block_size,
                                            (cudaStream_t)stream);
    if (vs != CB_OK) return vs;
  }
  int shift = 0;
  while ((1 << shift) < block_size) ++shift;
  int vshift = 0;
  while ((1 << vshift) < vecs) ++vshift;
  const int64_t total = (int64_t)num_tokens * num_kv_heads * vecs;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 152 * 64) blocks = 152 * 64;
  cb::kv_append_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(
      (const uint4*)k_new, (const uint4*)v_new, slot_mapping, num_tokens, (uint4*)k_cache,
      (uint4*)v_cache, (int64_t)num_blocks * block_size, num_kv_heads, vshift, shift,
      block_size - 1, error_word);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cb::fail(CB_ERR_CUDA, "cb_kv_append launch: %s", cudaGetErrorString(e));
  return CB_OK;
}
