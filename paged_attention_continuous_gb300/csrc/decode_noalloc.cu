// cb_paged_decode_noalloc: the split-KV decode kernel with its scratch in a
// fixed device array that this library owns, for callers that cannot
// allocate device memory.
//
// Who needs it: code that runs inside a host framework which owns the whole
// device-memory budget and does not allow side allocations while it
// executes (an inference-server plugin called from the framework's enqueue
// path, for example), and latency-critical loops where a cudaMalloc, with
// its implicit device synchronisation, is not acceptable.  Such callers can
// hand over their inputs and outputs but not a workspace.
//
// The scratch -- split partials (m, l, acc), per-(row, KV head) split
// counters, the work counters -- lives in one file-scope __device__ array of
// kNoAllocScratchBytes.  Every GPU that loads the library holds that array
// until the process exits.  Host code must not use the array's name as a
// device address (on the host it is only a stand-in); the device address is
// fetched once per device with cudaGetSymbolAddress, with that device
// current, on the first call made on that device.
#include <cuda_runtime.h>

#include <mutex>

#include "cb_error.h"
#include "decode_launch.h"
#include "launch_common.h"

namespace cb {
namespace {

constexpr size_t kNoAllocScratchBytes = CB_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) uint8_t g_decode_scratch[kNoAllocScratchBytes];

struct NoAllocLayout {
  size_t counters = 0, part_ml = 0, part_acc = 0, total = 0, zeroed = 0;
  int64_t slots = 0;  // partial slots (0: the call does not fit)
};

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// As many partial slots as the decode plan would like, or as fit in the
// array; at least 2 per row are needed (the plan then uses larger splits).
// Hq, Hkv and D are validated (positive) before this is called.
NoAllocLayout noalloc_layout(int64_t rows, int64_t Hq, int64_t Hkv, int64_t D) {
  NoAllocLayout l;
  // [0, 256): word 1 item counter; then the split tickets done[rows * Hkv]
  l.counters = 256;
  l.part_ml = l.counters + up256((size_t)rows * Hkv * 4);
  const size_t per_slot = (size_t)Hq * (D + 2) * 4;
  const size_t room = kNoAllocScratchBytes - l.part_ml - 512;  // two roundings to 256
  int64_t slots = decode::partial_slots(rows, Hkv);
  if ((size_t)slots > room / per_slot) slots = (int64_t)(room / per_slot);
  l.slots = slots >= 2 * rows ? slots : 0;
  l.part_acc = l.part_ml + up256((size_t)slots * Hq * 2 * 4);
  l.total = l.part_acc + up256((size_t)slots * Hq * D * 4);
  l.zeroed = l.part_ml;  // counters must read zero when a launch starts
  return l;
}

std::mutex g_mu;
uint8_t* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once
// per device, with that device current).
cb_status scratch_for_current_device(uint8_t** out) {
  int dev = -1;
  cb_status st = current_device(&dev);
  if (st != CB_OK) return st;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || !p)
      return fail(CB_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    g_scratch_ptr[dev] = static_cast<uint8_t*>(p);
  }
  *out = g_scratch_ptr[dev];
  return CB_OK;
}

}  // namespace
}  // namespace cb

extern "C" cb_status cb_paged_decode_noalloc(const cb_attention_args* args, uint32_t* error_word,
                                             cb_stream_t stream_) {
  using cb::fail;
  if (!args) return fail(CB_ERR_INVALID_ARG, "args is NULL");
  const cb_attention_args& a = *args;
  cudaStream_t stream = (cudaStream_t)stream_;
  if (a.num_reqs < 0 || a.num_decodes != a.num_reqs || a.num_tokens != a.num_reqs)
    return fail(CB_ERR_INVALID_ARG,
                "no-alloc decode: every row must be a decode (num_decodes == num_reqs == num_tokens)");
  if (a.num_reqs == 0) return CB_OK;
  if (!a.q || !a.out || !a.k_cache || !a.v_cache || !a.cu_seqlens_q || !a.seq_lens || !a.block_tables)
    return fail(CB_ERR_INVALID_ARG, "NULL pointer argument");
  if (a.num_q_heads <= 0 || a.num_kv_heads <= 0 || a.num_q_heads % a.num_kv_heads != 0)
    return fail(CB_ERR_INVALID_ARG, "num_q_heads must be a positive multiple of num_kv_heads");
  if (a.num_kv_heads > 64) return fail(CB_ERR_UNSUPPORTED, "num_kv_heads > 64");
  if (a.head_dim != 64 && a.head_dim != 128)
    return fail(CB_ERR_UNSUPPORTED, "no-alloc decode: head_dim must be 64 or 128");
  const int G = a.num_q_heads / a.num_kv_heads;
  const int max_g = a.dtype == CB_DTYPE_BF16 ? 16 : 8;
  if (G > max_g || (G & (G - 1)) != 0)
    return fail(CB_ERR_UNSUPPORTED, "no-alloc decode: %d query heads per KV head", G);
  if (a.block_size != 16) return fail(CB_ERR_UNSUPPORTED, "block_size must be 16");
  if (a.dtype != CB_DTYPE_F32 && a.dtype != CB_DTYPE_BF16) return fail(CB_ERR_INVALID_ARG, "unknown dtype");
  if (a.num_blocks <= 0 || a.max_blocks_per_seq <= 0) return fail(CB_ERR_INVALID_ARG, "bad pool sizes");
  if (a.sliding_window < 0) return fail(CB_ERR_INVALID_ARG, "sliding_window must be >= 0");
  const uintptr_t al = (uintptr_t)a.q | (uintptr_t)a.out | (uintptr_t)a.k_cache | (uintptr_t)a.v_cache;
  if (al & 15u) return fail(CB_ERR_INVALID_ARG, "q/out/cache pointers must be 16-byte aligned");
  if (a.num_reqs > cb::decode::kPlanMax)
    return fail(CB_ERR_INVALID_ARG, "no-alloc decode: at most %d rows per call", cb::decode::kPlanMax);
  const cb::NoAllocLayout L =
      cb::noalloc_layout(a.num_reqs, a.num_q_heads, a.num_kv_heads, a.head_dim);
  if (L.slots == 0 || L.total > cb::kNoAllocScratchBytes)
    return fail(CB_ERR_INVALID_ARG,
                "no-alloc decode: %d rows x %d query heads x head_dim %d need at least %zu "
                "scratch bytes, more than the fixed %zu",
                a.num_reqs, a.num_q_heads, a.head_dim,
                (size_t)2 * a.num_reqs * a.num_q_heads * (a.head_dim + 2) * 4 + L.part_ml,
                cb::kNoAllocScratchBytes);
  uint8_t* scratch = nullptr;
  cb_status st = cb::scratch_for_current_device(&scratch);
  if (st != CB_OK) return st;
  // the array keeps the previous call's contents: the counters must read
  // zero when the kernel starts
  cudaError_t e = cudaMemsetAsync(scratch, 0, L.zeroed, stream);
  if (e != cudaSuccess) return fail(CB_ERR_CUDA, "clearing scratch: %s", cudaGetErrorString(e));
  cb::decode::Scratch ds{};
  ds.work_counter = reinterpret_cast<uint32_t*>(scratch) + 1;
  ds.done = reinterpret_cast<uint32_t*>(scratch + L.counters);
  ds.part_ml = reinterpret_cast<float*>(scratch + L.part_ml);
  ds.part_acc = reinterpret_cast<float*>(scratch + L.part_acc);
  ds.slots = L.slots;
  const cb::decode::After after = a.after_append ? cb::decode::After::kAppend : cb::decode::After::kStream;
  st = a.dtype == CB_DTYPE_BF16 ? cb::decode::dispatch_bf16(a, ds, error_word, stream, after)
                                : cb::decode::dispatch_f32(a, ds, error_word, stream, after);
  if (st == CB_ERR_UNSUPPORTED)
    return fail(CB_ERR_UNSUPPORTED, "no-alloc decode: head_dim %d with %d query heads per KV head",
                a.head_dim, G);
  return st;
}
