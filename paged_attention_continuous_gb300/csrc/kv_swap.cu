// cb_kv_swap: move whole KV blocks between two sets of pools.
//
// "Continuous batching architecture", Offloading: an offloaded request's KV
// blocks are copied to a preallocated pinned CPU pool, every request that
// fits in one transfer, and copied back to (new) GPU blocks when space is
// available again, so the request resumes without recomputation.  Here one
// launch moves the listed blocks of every pool given (every layer's K and
// V), reading and writing either device memory or pinned host memory
// directly (the host side through unified addressing over the CPU-GPU
// link), so no staging copy is needed.  Each thread moves 16-byte vectors;
// consecutive threads cover consecutive bytes of one block.
#include <cuda_runtime.h>

#include "cb_error.h"
#include "device_utils.cuh"

namespace cb {
namespace {

struct SwapParams {
  const uint4* src[CB_SWAP_MAX_POOLS];
  uint4* dst[CB_SWAP_MAX_POOLS];
  const int32_t* src_ids;
  const int32_t* dst_ids;
  int64_t src_capacity, dst_capacity;
  int32_t num_pairs, num_pools;
  int64_t vecs_per_block;
  uint32_t* error_word;
};

__global__ void __launch_bounds__(256) kv_swap_kernel(const __grid_constant__ SwapParams p) {
  const int64_t per_pair = (int64_t)p.num_pools * p.vecs_per_block;
  const int64_t total = (int64_t)p.num_pairs * per_pair;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t pair = (int32_t)(i / per_pair);
    const int64_t rem = i - (int64_t)pair * per_pair;
    const int32_t pool = (int32_t)(rem / p.vecs_per_block);
    const int64_t v = rem - (int64_t)pool * p.vecs_per_block;
    const int32_t s = __ldg(p.src_ids + pair);
    const int32_t d = __ldg(p.dst_ids + pair);
    if (s < 0 || s >= p.src_capacity || d < 0 || d >= p.dst_capacity) {
      if (v == 0 && pool == 0) set_error(p.error_word, CB_DEVERR_BLOCK_RANGE);
      continue;
    }
    p.dst[pool][(int64_t)d * p.vecs_per_block + v] = p.src[pool][(int64_t)s * p.vecs_per_block + v];
  }
}

// The address the kernel uses for a pool: device memory of the current
// device as is, pinned host memory through its mapped device address.
// Anything else (pageable host memory, another device's memory) is refused
// before a launch could touch it.
cb_status device_view(const void* ptr, int dev, void** out) {
  cudaPointerAttributes at{};
  cudaError_t e = cudaPointerGetAttributes(&at, ptr);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(CB_ERR_CUDA, "cb_kv_swap: cudaPointerGetAttributes: %s", cudaGetErrorString(e));
  }
  if ((at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) && at.device == dev) {
    *out = const_cast<void*>(ptr);
    return CB_OK;
  }
  if (at.type == cudaMemoryTypeHost && at.devicePointer) {
    *out = at.devicePointer;
    return CB_OK;
  }
  return fail(CB_ERR_INVALID_ARG,
              "cb_kv_swap: a pool is neither memory of the current device nor pinned host memory");
}

}  // namespace
}  // namespace cb

extern "C" cb_status cb_kv_swap(const cb_swap_args* a, cb_stream_t stream) {
  using cb::fail;
  if (!a) return fail(CB_ERR_INVALID_ARG, "cb_kv_swap: args is NULL");
  if (a->num_pairs < 0 || a->num_pools < 0 || a->num_pools > CB_SWAP_MAX_POOLS)
    return fail(CB_ERR_INVALID_ARG, "cb_kv_swap: num_pools must be in [0, %d]", CB_SWAP_MAX_POOLS);
  if (a->num_pairs == 0 || a->num_pools == 0) return CB_OK;
  if (!a->src_ids || !a->dst_ids || !a->src_pools || !a->dst_pools)
    return fail(CB_ERR_INVALID_ARG, "cb_kv_swap: NULL pointer");
  if (a->block_bytes <= 0 || a->block_bytes % 16 != 0)
    return fail(CB_ERR_INVALID_ARG, "cb_kv_swap: block_bytes must be a positive multiple of 16");
  if (a->src_capacity <= 0 || a->dst_capacity <= 0)
    return fail(CB_ERR_INVALID_ARG, "cb_kv_swap: pool capacities must be positive");
  for (int32_t i = 0; i < a->num_pools; ++i) {
    if (!a->src_pools[i] || !a->dst_pools[i] || ((uintptr_t)a->src_pools[i] & 15u) ||
        ((uintptr_t)a->dst_pools[i] & 15u))
      return fail(CB_ERR_INVALID_ARG, "cb_kv_swap: pool %d is NULL or not 16-byte aligned", i);
  }
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(CB_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  cb::SwapParams p{};
  for (int32_t i = 0; i < a->num_pools; ++i) {
    void* dp = nullptr;
    cb_status st = cb::device_view(a->src_pools[i], dev, &dp);
    if (st != CB_OK) return st;
    p.src[i] = static_cast<const uint4*>(dp);
    st = cb::device_view(a->dst_pools[i], dev, &dp);
    if (st != CB_OK) return st;
    p.dst[i] = static_cast<uint4*>(dp);
  }
  p.src_ids = a->src_ids;
  p.dst_ids = a->dst_ids;
  p.src_capacity = a->src_capacity;
  p.dst_capacity = a->dst_capacity;
  p.num_pairs = a->num_pairs;
  p.num_pools = a->num_pools;
  p.vecs_per_block = a->block_bytes / 16;
  p.error_word = a->error_word;
  const int64_t total = (int64_t)a->num_pairs * a->num_pools * p.vecs_per_block;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 152 * 32) blocks = 152 * 32;
  cb::kv_swap_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(CB_ERR_CUDA, "cb_kv_swap launch: %s", cudaGetErrorString(e));
  return CB_OK;
}
