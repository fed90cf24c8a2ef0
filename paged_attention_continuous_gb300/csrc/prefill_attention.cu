// Prefill-chunk attention on tcgen05 tensor cores (not yet enabled).
#include "cb_error.h"
#include "prefill_dispatch.h"

namespace cb {

bool prefill_supported(int) { return false; }

size_t prefill_workspace_bytes(int64_t, int64_t, int64_t) { return 0; }

cb_status launch_prefill_bf16(const cb_attention_args&, uint32_t*, uint8_t*, cudaStream_t) {
  return CB_ERR_UNSUPPORTED;
}

}  // namespace cb
