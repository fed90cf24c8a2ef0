// Split-KV decode kernel instantiations for bf16 caches (matrix-instruction
// path): head_dim 64 and 128, 1 to 16 query heads per KV head, with and
// without a sliding window.
#include "decode_launch.cuh"

namespace cb {
namespace decode {

cb_status dispatch_bf16(const cb_attention_args& a, const Scratch& s, uint32_t* error_word,
                        cudaStream_t stream, After after) {
  using T = __nv_bfloat16;
  const int G = a.num_q_heads / a.num_kv_heads;
#define CB_DEC(DD, GG)                                                              \
  if (a.head_dim == DD && G == GG)                                                  \
    return a.sliding_window > 0 ? launch<T, DD, GG, true>(a, s, error_word, stream, after) \
                                : launch<T, DD, GG, false>(a, s, error_word, stream, after);
  CB_DEC(128, 1) CB_DEC(128, 2) CB_DEC(128, 4) CB_DEC(128, 8) CB_DEC(128, 16)
  CB_DEC(64, 1) CB_DEC(64, 2) CB_DEC(64, 4) CB_DEC(64, 8) CB_DEC(64, 16)
#undef CB_DEC
  return CB_ERR_UNSUPPORTED;
}

}  // namespace decode
}  // namespace cb
