// Row-generic paged attention on the CUDA cores (fp32 arithmetic).
//
// Handles any query length and any head dim that is a multiple of 32: one
// warp per (query token, query head), lanes split the head dim, keys are
// walked page by page through the block table with an online softmax.
// It is the fp32 path (every row of an fp32 step) and the path for shapes
// the specialised kernels do not cover.  Same definition as every other
// path: "Chunked Prefill" (Ultralytics glossary), How chunked prefill works
// -- query i of a row at absolute position p = seq_len - q_len + i attends
// keys 0..p of its request; with a sliding window W > 0 only keys
// p-W+1..p ("Continuous batching architecture", Memory management).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "device_utils.cuh"

namespace cb {
namespace simt {

struct Params {
  const void* q;
  void* out;
  const void* k_cache;
  const void* v_cache;
  const int32_t* cu_seqlens_q;
  const int32_t* seq_lens;
  const int32_t* block_tables;
  int32_t row_begin, row_end;   // rows handled
  int32_t tok_begin, tok_end;   // = cu_seqlens_q[row_begin], cu_seqlens_q[row_end]
  int32_t num_blocks, max_blocks_per_seq, block_size;
  int32_t num_q_heads, num_kv_heads;
  float scale_log2;
  int32_t window;               // sliding window (0: full attention)
  uint32_t* error_word;
};

template <typename T>
__device__ __forceinline__ float load_elem(const T* p);
template <>
__device__ __forceinline__ float load_elem<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float load_elem<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

template <typename T>
__device__ __forceinline__ void store_elem(T* p, float v);
template <>
__device__ __forceinline__ void store_elem<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void store_elem<__nv_bfloat16>(__nv_bfloat16* p, float v) {
  *p = __float2bfloat16_rn(v);
}

template <typename T, int D>
__global__ void __launch_bounds__(256) rows_kernel(const Params p) {
  constexpr int kDPL = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int Hq = p.num_q_heads;
  const int64_t ntok = p.tok_end - p.tok_begin;
  if (wid >= ntok * Hq) return;
  const int t = p.tok_begin + (int)(wid / Hq);
  const int h = (int)(wid % Hq);
  // row of token t
  int lo = p.row_begin, hi = p.row_end - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.cu_seqlens_q[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int r = lo;
  const int q0 = p.cu_seqlens_q[r];
  const int q_len = p.cu_seqlens_q[r + 1] - q0;
  const int L = p.seq_lens[r];
  const int bs = p.block_size;
  T* orow = static_cast<T*>(p.out) + ((int64_t)t * Hq + h) * D;
  if (q_len < 1 || L < q_len || (L + bs - 1) / bs > p.max_blocks_per_seq) {
    if (lane == 0) set_error(p.error_word, CB_DEVERR_SEQ_RANGE);
    for (int e = lane; e < D; e += 32) store_elem<T>(orow + e, 0.f);
    return;
  }
  const int pos = L - q_len + (t - q0);
  const int g = h / (Hq / p.num_kv_heads);
  const T* qrow = static_cast<const T*>(p.q) + ((int64_t)t * Hq + h) * D;
  float qf[kDPL], acc[kDPL];
#pragma unroll
  for (int e = 0; e < kDPL; ++e) {
    qf[e] = load_elem<T>(qrow + lane * kDPL + e) * p.scale_log2;
    acc[e] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const T* kc = static_cast<const T*>(p.k_cache);
  const T* vc = static_cast<const T*>(p.v_cache);
  const int npages = pos / bs + 1;
  const int k_lo = p.window > 0 && pos + 1 > p.window ? pos + 1 - p.window : 0;
  for (int pg = k_lo / bs; pg < npages; ++pg) {
    const int blk = p.block_tables[(int64_t)r * p.max_blocks_per_seq + pg];
    if (blk < 0 || blk >= p.num_blocks) {
      if (lane == 0) set_error(p.error_word, CB_DEVERR_BLOCK_RANGE);
      continue;
    }
    const int64_t page_off = ((int64_t)blk * p.num_kv_heads + g) * bs * D;
    const int nk = min(bs, pos + 1 - pg * bs);
    for (int i = max(0, k_lo - pg * bs); i < nk; ++i) {
      const T* krow = kc + page_off + (int64_t)i * D + lane * kDPL;
      const T* vrow = vc + page_off + (int64_t)i * D + lane * kDPL;
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < kDPL; ++e) dot = fmaf(qf[e], load_elem<T>(krow + e), dot);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
      const float m_new = fmaxf(m, dot);
      const float a = exp2f(m - m_new);
      const float pr = exp2f(dot - m_new);
      l = l * a + pr;
#pragma unroll
      for (int e = 0; e < kDPL; ++e) acc[e] = fmaf(pr, load_elem<T>(vrow + e), acc[e] * a);
      m = m_new;
    }
  }
  const float inv = 1.f / l;
#pragma unroll
  for (int e = 0; e < kDPL; ++e) store_elem<T>(orow + lane * kDPL + e, acc[e] * inv);
}

}  // namespace simt
}  // namespace cb
