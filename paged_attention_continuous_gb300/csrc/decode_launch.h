// Launch of the split-KV decode kernel, shared by cb_paged_attention and
// cb_paged_decode_noalloc (the kernel instantiations live in one
// translation unit per cache dtype).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/cb.h"

namespace cb {
namespace decode {

constexpr int kItemsA = 1;          // phase-A items per warp (target)
constexpr int kItemsABeside = 8;    // phase-A items per warp beside a prefill grid
constexpr int kItemsB = 1;          // phase-B items per warp (target)
constexpr int kPlanMax = 1024;      // decode rows planned per launch
// Partial slots a call should provide for `rows` decode rows: kSlotsPerRow
// per row (the splits that rounding adds per row stay below this while the
// phase-A split is at most ~20x the phase-B split, as the kernel's sizing
// gives) plus the slots that kMaxWorkers warps' target item counts need.
// With fewer slots the kernel doubles the split sizes until the plan fits
// (2 slots per row always do).
constexpr int kSlotsPerRow = 32;
constexpr int kMaxWorkers = 2048;
constexpr int64_t partial_slots(int64_t rows, int64_t Hkv) {
  return rows * kSlotsPerRow + ((int64_t)kMaxWorkers * (kItemsABeside + kItemsB) + Hkv - 1) / Hkv;
}

// Scratch of one call; the caller owns it.
struct Scratch {
  uint32_t* work_counter;  // one word; zero between launches
  uint32_t* done;          // split tickets, >= min(rows, 1024) * Hkv words; zero between launches
  float* part_ml;          // [slots][Hkv][G][2]
  float* part_acc;         // [slots][Hkv][G][D]
  int64_t slots;           // partial slots per launch (>= 2 * min(rows, 1024))
};

// What the kernel queued just before the (first) decode launch on the
// stream is, and so how the decode grid may overlap it (programmatic
// dependent launch).
enum class After : int32_t {
  kStream = 0,   // anything: plain stream order
  kAppend = 1,   // the step's K/V append: the grid plans while it finishes
                 // and waits for it before reading the cache
  kPrefill = 2,  // the prefill rows of the same call, launched in plain
                 // order after everything they and the decode rows need; the
                 // grid runs beside them on the SMs they leave idle and only
                 // its completion waits for theirs
};

// Runs the decode rows [0, a.num_decodes) of `a` (query length 1 each),
// in launches of at most 1024 rows.  Returns CB_ERR_UNSUPPORTED (without
// setting an error message) when no instantiation covers the head_dim and
// group size, so the caller can fall back.
cb_status dispatch_bf16(const cb_attention_args& a, const Scratch& s, uint32_t* error_word,
                        cudaStream_t stream, After after);
cb_status dispatch_f32(const cb_attention_args& a, const Scratch& s, uint32_t* error_word,
                       cudaStream_t stream, After after);

}  // namespace decode
}  // namespace cb
