// TMA tensor maps of the paged K/V caches (host side).
#include "tensor_map.h"

#include <cuda_runtime.h>

#include <mutex>

#include "cb_error.h"

namespace cb {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

cb_status make_cache_map(CUtensorMap* m, const void* base, int64_t rows, int head_dim) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(CB_ERR_CUDA, "cuTensorMapEncodeTiled entry point not available");
  cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)head_dim * 2};
  cuuint32_t box[2] = {64, 16};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(CB_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return CB_OK;
}

}  // namespace

cb_status cached_cache_map(CUtensorMap* m, const void* base, int64_t rows, int head_dim) {
  if (head_dim != 64 && head_dim != 128) return fail(CB_ERR_UNSUPPORTED, "tensor map head_dim %d", head_dim);
  struct Entry {
    const void* base;
    int64_t rows;
    int head_dim;
    CUtensorMap map;
  };
  constexpr int kEntries = 64;
  static Entry entries[kEntries];
  static int used = 0, next = 0;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (entries[i].base == base && entries[i].rows == rows && entries[i].head_dim == head_dim) {
      *m = entries[i].map;
      return CB_OK;
    }
  cb_status st = make_cache_map(m, base, rows, head_dim);
  if (st != CB_OK) return st;
  entries[next] = Entry{base, rows, head_dim, *m};
  next = (next + 1) % kEntries;
  if (used < kEntries) ++used;
  return CB_OK;
}

}  // namespace cb
