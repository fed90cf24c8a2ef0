// Entry points of the prefill-chunk kernel (tcgen05 tensor cores), used by
// the attention dispatcher.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/cb.h"

namespace cb {

// Whether the tensor-core prefill kernel handles this GQA group size.
bool prefill_supported(int group);

// Bytes of the prefill kernel's region of the attention workspace (state
// that must read zero between calls; independent of the call's sizes).
size_t prefill_workspace_bytes(int64_t Hq, int64_t Hkv, int64_t D);

// CTAs the prefill-chunk kernel launches for the prefill rows of `a` (an
// upper bound on the (row, pair of query tiles) units times the KV heads;
// 0 without prefill rows).
int64_t prefill_ctas(const cb_attention_args& a);

// Launch the prefill-chunk kernel over rows [num_decodes, num_reqs) (bf16,
// head_dim 128).  Returns CB_ERR_UNSUPPORTED if it cannot take this call.
// overlap_previous: the kernel queued just before on `stream` is the decode
// kernel of the same call; the prefill grid may start on the SMs it leaves
// (programmatic stream serialization), as the two share no data.
cb_status launch_prefill_bf16(const cb_attention_args& a, uint32_t* error_word, uint8_t* scratch,
                              cudaStream_t stream, bool overlap_previous);

}  // namespace cb
