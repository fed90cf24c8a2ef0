// TMA tensor maps of the paged K/V caches, shared by the decode and prefill
// kernels.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "../../include/cb.h"

namespace cb {

// The 2-D view [rows][head_dim] bf16 of a cache laid out as
// [num_blocks][Hkv][16][head_dim] (rows = num_blocks * Hkv * 16), box 16
// rows x 64 dims with the 128-byte swizzle; rows past the end read as zeros.
// head_dim is 64 or 128.  Maps depend only on (base, rows, head_dim), so the
// last few are kept and reused.
cb_status cached_cache_map(CUtensorMap* m, const void* base, int64_t rows, int head_dim);

}  // namespace cb
