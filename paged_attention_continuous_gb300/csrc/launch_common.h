// Host helpers shared by the kernel launchers: per-device launch state and
// the test hooks of the bounded device waits.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "../../include/cb.h"

namespace cb {

constexpr int kMaxDevices = 64;

// Current device index, checked against kMaxDevices.
cb_status current_device(int* dev);

// SM count of the current device (cached per device).
int sm_count_current_device();

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) for `kernel` on the
// current device, once per device: function attributes are per device.
// `flags` is the caller's per-kernel array of kMaxDevices flags.
cb_status ensure_smem_attr(const void* kernel, size_t smem, std::atomic<uint8_t>* flags);

// Test hooks (cb_debug_inject_wait_timeout): the limit of every bounded
// device wait of later launches, and the decode work item / prefill KV
// tile whose copies are withheld (-1: none).
uint64_t wait_limit_ns();
int32_t withheld_decode_item();
int32_t withheld_prefill_tile();

}  // namespace cb
