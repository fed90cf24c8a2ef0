// Host helpers shared by the kernel launchers.
#include "launch_common.h"

#include "cb_error.h"

namespace cb {
namespace {
constexpr uint64_t kDefaultWaitNs = 1000ull * 1000ull * 1000ull;  // 1 s
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};
std::atomic<int32_t> g_withhold_decode{-1};
std::atomic<int32_t> g_withhold_prefill{-1};
std::atomic<int32_t> g_sm_count[kMaxDevices];
}  // namespace

cb_status current_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return fail(CB_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (*dev < 0 || *dev >= kMaxDevices) return fail(CB_ERR_UNSUPPORTED, "device index %d", *dev);
  return CB_OK;
}

int sm_count_current_device() {
  int dev = 0;
  if (current_device(&dev) != CB_OK) return 152;
  int n = g_sm_count[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 152;
  g_sm_count[dev].store(n, std::memory_order_relaxed);
  return n;
}

cb_status ensure_smem_attr(const void* kernel, size_t smem, std::atomic<uint8_t>* flags) {
  int dev = 0;
  cb_status st = current_device(&dev);
  if (st != CB_OK) return st;
  if (flags[dev].load(std::memory_order_acquire)) return CB_OK;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess)
    return fail(CB_ERR_CUDA, "kernel shared-memory attribute: %s", cudaGetErrorString(e));
  flags[dev].store(1, std::memory_order_release);
  return CB_OK;
}

uint64_t wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
int32_t withheld_decode_item() { return g_withhold_decode.load(std::memory_order_relaxed); }
int32_t withheld_prefill_tile() { return g_withhold_prefill.load(std::memory_order_relaxed); }

}  // namespace cb

extern "C" cb_status cb_debug_inject_wait_timeout(uint64_t wait_ns, int32_t decode_item,
                                                  int32_t prefill_tile) {
  cb::g_wait_ns.store(wait_ns ? wait_ns : cb::kDefaultWaitNs, std::memory_order_relaxed);
  cb::g_withhold_decode.store(decode_item < 0 ? -1 : decode_item, std::memory_order_relaxed);
  cb::g_withhold_prefill.store(prefill_tile < 0 ? -1 : prefill_tile, std::memory_order_relaxed);
  return CB_OK;
}
