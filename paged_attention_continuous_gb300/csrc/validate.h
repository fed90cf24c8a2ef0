// Host-side validation of a step's metadata (the debugging mode that
// CB_VALIDATE=1 in the environment turns on for the GPU calls).
#pragma once

#include <cuda_runtime.h>

#include "../../include/cb.h"

namespace cb {

// True when CB_VALIDATE is set to a non-zero value (read once).
bool validate_enabled();

// Copy the attention call's metadata to the host (synchronising `stream`)
// and check it with cb_validate_step.  Skipped (CB_OK) while `stream` is
// being captured into a CUDA graph, where a synchronous copy is not allowed.
cb_status validate_attention_call(const cb_attention_args& a, cudaStream_t stream);

// The same for cb_kv_append's slot mapping.
cb_status validate_append_call(const int32_t* slot_mapping, int32_t num_tokens,
                               int32_t num_blocks, int32_t block_size, cudaStream_t stream);

}  // namespace cb
