// Split-KV paged decode attention (one query token per request).
//
// What it computes: "Chunked Prefill" (Ultralytics glossary), How chunked
// prefill works -- each query attends, causally over absolute positions, to
// every cached key of its request; for a decode token at position
// seq_len - 1 that is keys 0..seq_len-1.  K/V are read through the request's
// block table ("vLLM serving internals", PagedAttention as a virtual memory
// system).  Decode reads the whole cache of every running request each step
// and does few operations per byte ("Chunked Prefill", Prefill, decode and
// generation stalls), so this kernel is built to stream HBM:
//
//   * Work item = (decode row r, split s, KV head g): a run of consecutive
//     16-token pages of one request and one KV head.  The items come in two
//     phases: first the leading 7/8 of every row's pages in equal large
//     splits, about one per warp, then the remaining 1/8 in small splits.
//     Warp w of W starts with item w; every later item is drawn in index
//     order from a global atomic counter (large items first), so the last
//     items are short and the warps finish together.  Launched beside a
//     prefill grid (whose CTAs hold most SMs at first), every item comes
//     from the counter and phase A is cut finer.  Split sizes are chosen in
//     the kernel from the total page count, and doubled until the splits
//     fit the caller's partial slots.
//   * Every WARP is an independent worker with its own pipeline: lane 0 issues
//     the copies of the (block, head) K page and V page into a ring of
//     kStages shared-memory stages, each tracked by an mbarrier; the ring
//     runs across item boundaries, so the next item's pages are already in
//     flight when one item ends.
//   * bf16 caches: the G query heads that share KV head g form a real
//     [G x D] . [D x 16] product per page, so both products of a page run as
//     warp-level bf16 matrix instructions (mma.sync m16n8k16, fp32
//     accumulate): S^T = K Q^T (16 tokens x 8 heads per n-tile), then
//     O^T += V^T P^T.  The TMA engine lands each page as 64-dim boxes in the
//     128-byte-swizzled layout, so the operand loads (ldmatrix, transposed
//     for V) are free of bank conflicts; P^T is formed from the score
//     fragments in registers (movmatrix).  The roofline stays HBM: the
//     matrix instructions only cut the issue slots per byte, which bound the
//     CUDA-core version of this loop at larger G.
//   * fp32 caches: CUDA-core path.  LG lanes cover one token's D dims,
//     partial dot products of the G heads are combined with a butterfly
//     reduce-scatter, P.V in packed f32x2 FMAs.
//   * Online softmax in base 2; the reference max moves only when a page
//     raises it by more than 2^8, so accumulators are rarely rescaled.
//   * A request with one split writes its output directly.  Otherwise every
//     split writes an (m, l, acc) partial and takes a ticket on its
//     (request, KV head) counter; the warp whose ticket completes the count
//     merges the splits with the log-sum-exp rescale and resets the counter.
//     No warp ever waits for another, so the kernel makes no assumption
//     about which CTAs are resident at the same time.
//
// Sliding-window layers ("Continuous batching architecture", Memory
// management): with window W > 0 the decode token at position seq_len - 1
// attends keys seq_len - W .. seq_len - 1 only.  A row's items then cover
// the pages from the one holding key seq_len - W (pages before it may have
// been recycled and are never read), and keys before the window on that
// first page are masked like the slots past the end on the last page.
#pragma once

#include <cuda.h>

#include <cstdint>
#include <cuda_bf16.h>
#include <type_traits>

#include "decode_launch.h"
#include "device_utils.cuh"

namespace cb {
namespace decode {

constexpr int kPageTokens = 16;
constexpr int kTailDiv = 8;         // the last 1/kTailDiv of each row's pages: phase B
constexpr int kMinSplitPages = 8;   // phase-A split size floor
// shared memory of the plan: split-count prefixes of both phases, and each
// row's sequence length (0 for a row that is skipped) and query token
constexpr int kPlanSmemBytes = (2 * (kPlanMax + 1) + 2 * kPlanMax) * (int)sizeof(int32_t);

struct Params {
  // bf16 caches: 2-D views [num_blocks * Hkv * 16 rows][D] of K and V, box
  // 16 rows x 64 dims, 128-byte swizzle (unused for fp32 caches)
  CUtensorMap tmap_k;
  CUtensorMap tmap_v;
  const void* q;
  void* out;
  const void* k_cache;
  const void* v_cache;
  const int32_t* cu_seqlens_q;
  const int32_t* seq_lens;
  const int32_t* block_tables;
  int32_t row_begin;       // first decode row handled by this launch
  int32_t num_rows;        // decode rows in this launch (<= kPlanMax)
  int32_t num_tokens;      // rows of q/out
  int32_t num_blocks;
  int32_t max_blocks_per_seq;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  float scale_log2;        // softmax scale * log2(e)
  int32_t window;          // sliding window (0: full attention)
  uint32_t* error_word;
  uint32_t* work_counter;  // zero between launches (the last grab resets it)
  uint32_t* done;          // [num_rows * Hkv] split tickets; zero between launches
  int32_t max_slots;       // partial slots available (>= 2 * num_rows)
  float* part_ml;          // [slots][Hkv][G][2]
  float* part_acc;         // [slots][Hkv][G][D]
  uint64_t wait_ns;        // limit of every bounded wait
  int32_t pdl_mode;        // After: 1 wait for the grid before (the append)
                           // before reading the cache; 2 only the grid's
                           // completion waits for the one before (prefill)
  int32_t withhold_item;   // test hook: the item with this global index
                           // never gets its first page's copies (-1: none)
};

// How a row of `pages` pages is cut, given the launch-wide split sizes spa
// (phase A) and spb (phase B): phase A covers pages [0, bp) in na full
// splits of spa pages, na = floor(leading (1 - 1/kTailDiv) of the row / spa);
// phase B covers the rest, [bp, pages), in nb splits of spb pages (the last
// one shorter).
struct RowSplit {
  int na, bp, nb;
};

// First key and first page a decode row of length L reads (window W, 0 = all).
__device__ __forceinline__ int first_key(int L, int W) { return W > 0 && L > W ? L - W : 0; }
__device__ __forceinline__ int first_page(int L, int W) { return first_key(L, W) / kPageTokens; }

__device__ __forceinline__ RowSplit row_split(int pages, int spa, int spb) {
  RowSplit s;
  const int big = pages - pages / kTailDiv;
  s.na = big / spa;
  s.bp = s.na * spa;
  s.nb = (pages - s.bp + spb - 1) / spb;
  return s;
}

// CUDA-core geometry (fp32 caches)
template <typename T, int D, int G>
struct Cfg {
  static constexpr int kElem = sizeof(T);
  static constexpr int kRowBytes = D * kElem;
  static constexpr int kChunks = kRowBytes / 16;  // 16-byte vectors per row
  static constexpr int kLG0 = (G >= 8) ? 16 : 8;
  static constexpr int kLG = kLG0 < kChunks ? kLG0 : kChunks;  // lanes per token
  static constexpr int kCPL = kChunks / kLG;                   // vectors per lane
  static constexpr int kEPC = 16 / kElem;                      // elements per vector
  static constexpr int kDPL = kCPL * kEPC;                     // dims per lane
  static constexpr int kTPI = 32 / kLG;                        // tokens per iteration
  static constexpr int kNIT = kPageTokens / kTPI;              // iterations per page
  static constexpr int kDup = kLG / G;                         // lanes holding one head's score
  static_assert(kRowBytes % 16 == 0, "row must be a multiple of 16 bytes");
  static_assert(kLG >= G && kLG % G == 0, "group must divide lanes per token");
  static_assert(kChunks % kLG == 0, "vectors must split evenly over lanes");
};

// Matrix-instruction geometry (bf16 caches)
template <int D, int G>
struct MmaCfg {
  static constexpr int kNT = (G + 7) / 8;  // n-tiles of 8 query heads
  static constexpr int kKS = D / 16;       // k-steps of K Q^T
  static constexpr int kMT = D / 16;       // m-tiles of V^T P^T
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static_assert(G == 1 || G == 2 || G == 4 || G == 8 || G == 16, "group 1..16");
};

struct ItemDesc {
  int32_t r, g, split, nsplit, page0, page1, seq_len, token, slot;
  int32_t pad[3];
};

template <typename T, int D, int G, int kStages>
struct WarpSmem {
  static constexpr int kPageBytes = kPageTokens * D * (int)sizeof(T);
  static constexpr int kQBytes = G * D * (int)sizeof(T);
  static constexpr int kRing = kStages + 1;
  // K page | V page of every stage; 1024-byte aligned for the swizzled boxes
  alignas(1024) uint8_t kv[kStages][2][kPageBytes];
  alignas(16) uint8_t q[kRing][kQBytes];
  ItemDesc items[kRing];
  uint64_t full[kStages];
  int32_t stage_item[kStages];
  int32_t stage_page[kStages];
};

// Dynamic shared memory of a launch (the extra 1 KB aligns the base).
template <typename T, int D, int G, int kWarps, int kStages>
constexpr size_t smem_bytes() {
  return sizeof(WarpSmem<T, D, G, kStages>) * kWarps + kPlanSmemBytes + 1024;
}

// ---- matrix-instruction helpers -------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
// transpose of an 8x8 b16 matrix held one 32-bit pair per lane
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}
// c += a . b, m16n8k16, bf16 inputs, fp32 accumulate
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// 2-D TMA box load with an L2 eviction hint, completion on an mbarrier
__device__ __forceinline__ void tma_load_2d_hint(void* smem_dst, const CUtensorMap* tmap, int32_t x,
                                                 int32_t y, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(smem_dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}
// byte offset of 16-byte chunk `gc` (0 .. D/8-1) of page row `t` in a page
// landed as 64-dim boxes of 16 rows x 128 bytes with the 128-byte swizzle
__device__ __forceinline__ uint32_t swz_off(int t, int gc) {
  return (uint32_t)((gc >> 3) * 2048 + t * 128 + (((gc & 7) ^ (t & 7)) << 4));
}

// Unpack one 16-byte vector into kEPC floats.
template <typename T>
__device__ __forceinline__ void unpack16(const uint4& w, float* f);

template <>
__device__ __forceinline__ void unpack16<__nv_bfloat16>(const uint4& w, float* f) {
  float2 a = bf16x2_to_float2(w.x), b = bf16x2_to_float2(w.y);
  float2 c = bf16x2_to_float2(w.z), d = bf16x2_to_float2(w.w);
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
  f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}

template <>
__device__ __forceinline__ void unpack16<float>(const uint4& w, float* f) {
  f[0] = __uint_as_float(w.x); f[1] = __uint_as_float(w.y);
  f[2] = __uint_as_float(w.z); f[3] = __uint_as_float(w.w);
}

// Store kDPL floats (one lane's dims of one head row) to a T row.
template <typename T, int D, int G>
__device__ __forceinline__ void store_row(T* row, int j, const float* v) {
  using C = Cfg<T, D, G>;
#pragma unroll
  for (int c = 0; c < C::kCPL; ++c) {
    const float* f = v + c * C::kEPC;
    uint4 w;
    if constexpr (sizeof(T) == 2) {
      w.x = float2_to_bf16x2(f[0], f[1]);
      w.y = float2_to_bf16x2(f[2], f[3]);
      w.z = float2_to_bf16x2(f[4], f[5]);
      w.w = float2_to_bf16x2(f[6], f[7]);
    } else {
      w.x = __float_as_uint(f[0]); w.y = __float_as_uint(f[1]);
      w.z = __float_as_uint(f[2]); w.w = __float_as_uint(f[3]);
    }
    reinterpret_cast<uint4*>(row)[j + C::kLG * c] = w;
  }
}

// Merge the n >= 2 split partials of (decode row i, KV head g), whose slots
// start at s0, into the output rows of query token q0: for each of the G
// heads, o = sum_s w_s acc_s / sum_s w_s l_s with w_s = 2^(m_s - max m).
// One warp; per batch of 32 splits, lane k reads the (m, l) of every head of
// split k, and lanes [0, D/4) each own 4 output elements of every head;
// the accumulator loads of kU splits x G heads are in flight together.
template <typename T, int D, int G>
__device__ __noinline__ void merge_splits(const Params& p, int g, int s0, int n, int q0, int lane) {
  constexpr int kV = D / 4;
  constexpr int kU = G >= 16 ? 1 : 16 / G;
  static_assert(kV <= 32, "head row must fit one warp");
  const int Hkv = p.num_kv_heads;
  const int64_t base = (int64_t)s0 * Hkv + g;  // partial index of split 0
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml) + base * G;
  const int64_t ml_stride = (int64_t)Hkv * G;
  const float4* pa = reinterpret_cast<const float4*>(p.part_acc) + base * G * kV + lane;
  const int64_t acc_stride = (int64_t)Hkv * G * kV;
  float M[G], Ls[G];
  float4 o[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    M[h] = -INFINITY;
    Ls[h] = 0.f;
    o[h] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int b0 = 0; b0 < n; b0 += 32) {
    const int cnt = min(32, n - b0);
    float wl[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float2 v = lane < cnt ? __ldcg(ml + (int64_t)(b0 + lane) * ml_stride + h)
                                  : make_float2(-INFINITY, 0.f);
      float bm = v.x;
#pragma unroll
      for (int k = 16; k > 0; k >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, k));
      const float Mn = fmaxf(M[h], bm);
      wl[h] = lane < cnt ? exp2f(v.x - Mn) : 0.f;
      float lsum = wl[h] * v.y;
#pragma unroll
      for (int k = 16; k > 0; k >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, k);
      const float a_old = exp2f(M[h] - Mn);  // 0 on the first batch
      Ls[h] = Ls[h] * a_old + lsum;
      o[h].x *= a_old; o[h].y *= a_old; o[h].z *= a_old; o[h].w *= a_old;
      M[h] = Mn;
    }
    for (int k0 = 0; k0 < cnt; k0 += kU) {
      float4 av[kU][G];
#pragma unroll
      for (int u = 0; u < kU; ++u)
#pragma unroll
        for (int h = 0; h < G; ++h)
          av[u][h] = (k0 + u < cnt && lane < kV)
                         ? __ldcg(pa + (int64_t)(b0 + k0 + u) * acc_stride + h * kV)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u = 0; u < kU; ++u)
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float w = __shfl_sync(0xffffffffu, wl[h], (k0 + u) & 31);
          o[h].x += w * av[u][h].x; o[h].y += w * av[u][h].y;
          o[h].z += w * av[u][h].z; o[h].w += w * av[u][h].w;
        }
    }
  }
  if (lane < kV) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float inv = 1.f / Ls[h];
      T* orow = static_cast<T*>(p.out) + ((int64_t)q0 * p.num_q_heads + (int64_t)g * G + h) * D +
                4 * lane;
      if constexpr (sizeof(T) == 2) {
        uint2 w2;
        w2.x = float2_to_bf16x2(o[h].x * inv, o[h].y * inv);
        w2.y = float2_to_bf16x2(o[h].z * inv, o[h].w * inv);
        *reinterpret_cast<uint2*>(orow) = w2;
      } else {
        *reinterpret_cast<float4*>(orow) =
            make_float4(o[h].x * inv, o[h].y * inv, o[h].z * inv, o[h].w * inv);
      }
    }
  }
}

// kWindow: the launch has a sliding window (p.window > 0); the full-attention
// instantiation compiles the window arithmetic away.
template <typename T, int D, int G, int kWarps, int kStages, bool kWindow>
__global__ void __launch_bounds__(kWarps * 32, 1) decode_kernel(const __grid_constant__ Params p) {
  constexpr bool kMma = std::is_same<T, __nv_bfloat16>::value;
  using WS = WarpSmem<T, D, G, kStages>;
  constexpr int kRing = WS::kRing;
  constexpr int kPageBytes = WS::kPageBytes;
  constexpr int kQBytes = WS::kQBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  WS* wsm_all = reinterpret_cast<WS*>(smem);
  int32_t* plan_a = reinterpret_cast<int32_t*>(smem + sizeof(WS) * kWarps);  // [num_rows + 1]
  int32_t* plan_b = plan_a + (kPlanMax + 1);                                  // [num_rows + 1]
  int32_t* row_len = plan_b + (kPlanMax + 1);                                 // [num_rows]
  int32_t* row_tok = row_len + kPlanMax;                                      // [num_rows]
  __shared__ int32_t s_red[kWarps];
  __shared__ int32_t s_red2[kWarps];
  __shared__ int32_t s_spa, s_spb;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nthreads = kWarps * 32;
  const int Hkv = p.num_kv_heads;
  const int Hq = p.num_q_heads;
  const int W = p.max_blocks_per_seq;
  const int win = kWindow ? p.window : 0;

  // ---- plan: pages per row -> split sizes -> prefixes of split counts -----
  // Rows are checked once here and kept in shared memory; a row that fails a
  // check gets length 0 (no items) and its error bit.
  int64_t my_pages = 0;
  for (int i = threadIdx.x; i < p.num_rows; i += nthreads) {
    const int r = p.row_begin + i;
    int L = p.seq_lens[r];
    const int q0 = p.cu_seqlens_q[r];
    const int q1 = p.cu_seqlens_q[r + 1];
    int pages = (L + kPageTokens - 1) / kPageTokens;
    if (L == 0 && q1 == q0) {
      // a padding row (no query, no context): nothing to do
    } else {
      if (L < 1 || pages > W) {
        L = 0;
        if (blockIdx.x == 0) set_error(p.error_word, CB_DEVERR_SEQ_RANGE);
      }
      if (q1 - q0 != 1 || q0 < 0 || q0 >= p.num_tokens) {
        L = 0;
        if (blockIdx.x == 0) set_error(p.error_word, CB_DEVERR_DECODE_QLEN);
      }
    }
    pages = (L + kPageTokens - 1) / kPageTokens - first_page(L, win);
    row_len[i] = L;
    row_tok[i] = q0;
    my_pages += pages;
  }
  for (int o = 16; o > 0; o >>= 1) my_pages += __shfl_xor_sync(0xffffffffu, my_pages, o);
  if (lane == 0) s_red[warp] = (int32_t)(my_pages < 0x3fffffff ? my_pages : 0x3fffffff);
  __syncthreads();
  if (threadIdx.x == 0) {
    int64_t tot = 0;
    for (int w = 0; w < kWarps; ++w) tot += s_red[w];
    const int64_t units = tot * Hkv;
    const int64_t units_b = units / kTailDiv;
    const int64_t workers = (int64_t)gridDim.x * kWarps;
    // beside a prefill grid (pdl_mode 2) the CTAs start at different times
    // and draw every item from the counter: smaller items keep their finish
    // together
    const int64_t items_a = p.pdl_mode == 2 ? kItemsABeside : kItemsA;
    int64_t spa = (units - units_b + workers * items_a - 1) / (workers * items_a);
    int64_t spb = (units_b + workers * kItemsB - 1) / (workers * kItemsB);
    if (spa < kMinSplitPages) spa = kMinSplitPages;
    if (spb < 1) spb = 1;
    s_spa = (int32_t)(spa < (1 << 20) ? spa : (1 << 20));
    s_spb = (int32_t)(spb < (1 << 20) ? spb : (1 << 20));
  }
  __syncthreads();
  int spa0 = s_spa, spb0 = s_spb;
  // per row split counts of both phases and their prefixes (serial segments
  // per thread + a block scan of the segment sums); if the splits exceed the
  // partial slots, double both split sizes and plan again
  for (int attempt = 0;; ++attempt) {
    const int seg = (p.num_rows + nthreads - 1) / nthreads;
    const int b = threadIdx.x * seg;
    const int e = min(b + seg, p.num_rows);
    int sum_a = 0, sum_b = 0;
    for (int i = b; i < e; ++i) {
      const int Li = row_len[i];
      const RowSplit rs =
          row_split((Li + kPageTokens - 1) / kPageTokens - first_page(Li, win), spa0, spb0);
      const int na = rs.na, nb = rs.nb;
      plan_a[i + 1] = na;
      plan_b[i + 1] = nb;
      sum_a += na;
      sum_b += nb;
    }
    int inc_a = sum_a, inc_b = sum_b;
    for (int o = 1; o < 32; o <<= 1) {
      const int va = __shfl_up_sync(0xffffffffu, inc_a, o);
      const int vb = __shfl_up_sync(0xffffffffu, inc_b, o);
      if (lane >= o) {
        inc_a += va;
        inc_b += vb;
      }
    }
    if (lane == 31) {
      s_red[warp] = inc_a;
      s_red2[warp] = inc_b;
    }
    __syncthreads();
    int off_a = 0, off_b = 0;
    for (int w = 0; w < warp; ++w) {
      off_a += s_red[w];
      off_b += s_red2[w];
    }
    int run_a = off_a + inc_a - sum_a, run_b = off_b + inc_b - sum_b;
    if (threadIdx.x == 0) {
      plan_a[0] = 0;
      plan_b[0] = 0;
    }
    for (int i = b; i < e; ++i) {
      run_a += plan_a[i + 1];
      run_b += plan_b[i + 1];
      plan_a[i + 1] = run_a;
      plan_b[i + 1] = run_b;
    }
    __syncthreads();
    if (plan_a[p.num_rows] + plan_b[p.num_rows] <= p.max_slots || attempt >= 40) break;
    if (spa0 < (1 << 29)) spa0 *= 2;
    if (spb0 < (1 << 29)) spb0 *= 2;
    __syncthreads();  // everyone has read the totals before they are rewritten
  }
  // unreachable with max_slots >= 2 * num_rows; refuse rather than overrun
  const bool plan_ok = plan_a[p.num_rows] + plan_b[p.num_rows] <= p.max_slots &&
                       (int64_t)(plan_a[p.num_rows] + plan_b[p.num_rows]) * Hkv < (1 << 26);
  if (!plan_ok && blockIdx.x == 0 && threadIdx.x == 0) set_error(p.error_word, CB_DEVERR_PLAN);
  const int num_a = plan_a[p.num_rows];
  const int num_b = plan_b[p.num_rows];
  const int total_items = plan_ok ? (num_a + num_b) * Hkv : 0;
  const uint32_t total_workers = gridDim.x * kWarps;

  // ---- per-warp pipeline --------------------------------------------------
  WS& ws = wsm_all[warp];
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&ws.full[s], 1);
    fence_barrier_init();
  }
  __syncwarp();

  const uint64_t pol = l2_policy_evict_first();
  const uint8_t* kbase = static_cast<const uint8_t*>(p.k_cache);
  const uint8_t* vbase = static_cast<const uint8_t*>(p.v_cache);

  // producer cursor (uniform across the warp)
  int prod_slot = -1;      // ring slot of the producer's current item
  int prod_page = 0, prod_end = 0;
  int prod_items = 0;      // items started by the producer
  int cons_items = 0;      // items whose last page the consumer has processed
  int win_base = 0;        // first page covered by blk_win
  int blk_win = -1;        // lane i holds the block id of page win_base + i
  int blk_win2 = -1;       // lane i: block id of page win_base + 32 + i
  bool exhausted = false;
  bool aborted = false;
  int prod_row = 0, prod_g = 0;
  uint32_t phases = 0;     // parity bit per stage
  int issued = 0, consumed = 0;

  // Look-ahead: the item after the producer's current one is decoded, and
  // its first block ids requested, one item early, so that the block-table
  // load does not stall an item change.  Indices after a warp's first come
  // from the counter, whose next value lane 0 keeps in flight.
  const int items_a = num_a * Hkv;
  const uint32_t worker = blockIdx.x * kWarps + warp;
  // a warp's first item is dealt statically (item w); every later one is
  // drawn from the counter in index order, phase A's large items first.
  // Beside a prefill grid most CTAs start only as its CTAs end, so there
  // every item is drawn from the counter: the CTAs that start first take
  // more.
  const uint32_t n_static =
      p.pdl_mode == 2 ? 0u : (uint32_t)min((int64_t)items_a, (int64_t)total_workers);
  bool first_static = worker < n_static;
  uint32_t pref_idx = 0;
  lane0_fetch_add1(p.work_counter, pref_idx, lane);
  // idx / Hkv without a division: floor(idx * ceil(2^32 / Hkv) / 2^32) is
  // exact for idx < 2^26 and Hkv <= 64 (the plan keeps total_items below)
  const uint64_t hkv_magic = (0x100000000ull + Hkv - 1) / Hkv;
  bool nx_ok = false;
  int nx_i = 0, nx_g = 0, nx_split = 0, nx_nsplit = 0, nx_page0 = 0, nx_page1 = 0, nx_len = 0,
      nx_tok = 0, nx_slot = 0, nx_idx = 0;
  int nx_blk = -1;         // lane i: block id of page nx_page0 + i
  int prod_idx = -1;       // global index of the producer's current item

  // Largest row i in [0, num_rows) with plan[i] <= u (plan is a prefix sum,
  // plan[0] = 0 <= u), i.e. the number of rows with plan[i] <= u, minus one.
  // Warp-parallel in two levels of ballots: which of 32 segments of `step`
  // rows holds it, then which row of that segment (num_rows <= 1024).
  const int fr_step = (p.num_rows + 31) >> 5;
  auto find_row = [&](const int32_t* plan, int u) -> int {
    const int i1 = lane * fr_step;
    const bool le1 = i1 < p.num_rows && plan[i1] <= u;
    const int seg = __popc(__ballot_sync(0xffffffffu, le1)) - 1;
    const int base = seg * fr_step;
    const int i2 = base + lane;
    const bool le2 = lane < fr_step && i2 < p.num_rows && plan[i2] <= u;
    return base + __popc(__ballot_sync(0xffffffffu, le2)) - 1;
  };

  // decode the prefetched index into the look-ahead item and fetch the next
  // index; nx_ok = false once the items are exhausted
  auto fetch_ahead = [&]() {
    nx_ok = false;
    uint32_t idx;
    if (first_static) {
      idx = worker;
      first_static = false;
    } else {
      const uint32_t b = __shfl_sync(0xffffffffu, pref_idx, 0);
      const uint32_t items_dyn = (uint32_t)total_items - n_static;
      if (b >= items_dyn) {
        if (b == items_dyn + total_workers - 1 && lane == 0) atomicExch(p.work_counter, 0u);
        return;
      }
      lane0_fetch_add1(p.work_counter, pref_idx, lane);
      idx = n_static + b;
    }
    const uint32_t u = (uint32_t)(((uint64_t)idx * hkv_magic) >> 32);
    const int g = (int)(idx - u * (uint32_t)Hkv);
    const bool phase_a = (int)u < num_a;
    const int i = phase_a ? find_row(plan_a, (int)u) : find_row(plan_b, (int)u - num_a);
    const int a0 = plan_a[i], a1 = plan_a[i + 1], b0 = plan_b[i], b1 = plan_b[i + 1];
    const int split = phase_a ? (int)u - a0 : (int)u - num_a - b0;
    const int r = p.row_begin + i;
    const int L = row_len[i];
    const int pages = (L + kPageTokens - 1) / kPageTokens;
    const int fp = first_page(L, win);
    const int na = a1 - a0;
    const int bp = fp + na * spa0;
    nx_ok = true;
    nx_idx = (int)idx;
    nx_i = i;
    nx_g = g;
    nx_split = split;
    nx_nsplit = na + (b1 - b0);
    if (phase_a) {
      nx_page0 = fp + split * spa0;
      nx_page1 = nx_page0 + spa0;
    } else {
      nx_page0 = bp + split * spb0;
      nx_page1 = min(pages, nx_page0 + spb0);
    }
    nx_len = L;
    nx_tok = row_tok[i];
    nx_slot = a0 + b0 + (phase_a ? split : na + split);
    const int pg = nx_page0 + lane;
    nx_blk = (pg < nx_page1) ? __ldg(p.block_tables + (int64_t)r * W + pg) : -1;
  };

  // make the look-ahead item the producer's current one (describing it in
  // the ring) and look one further ahead; false when none is left
  auto next_item = [&]() -> bool {
    if (!nx_ok) return false;
    const int slot_i = (prod_items) % kRing;
    ++prod_items;
    prod_slot = slot_i;
    prod_row = p.row_begin + nx_i;
    prod_g = nx_g;
    prod_page = nx_page0;
    prod_end = nx_page1;
    prod_idx = nx_idx;
    win_base = nx_page0;
    blk_win = nx_blk;
    if (lane == 0) {
      ItemDesc& d = ws.items[slot_i];
      d.r = nx_i; d.g = nx_g; d.split = nx_split; d.nsplit = nx_nsplit;
      d.page0 = nx_page0; d.page1 = nx_page1; d.seq_len = nx_len; d.token = nx_tok;
      d.slot = nx_slot;
    }
    __syncwarp();
    fetch_ahead();
    return true;
  };
  fetch_ahead();

  // refill one stage with the producer's next page (whole warp calls this)
  auto produce = [&](int st) {
    if (exhausted || aborted) return;
    bool first = false;
    if (prod_slot < 0 || prod_page >= prod_end) {
      if (!next_item()) { exhausted = true; return; }
      first = true;
    }
    // block ids come 32 pages at a time; the next 32 are requested half way
    // through the current window
    if (prod_page - win_base == 16 && win_base + 32 < prod_end) {
      const int pg = win_base + 32 + lane;
      blk_win2 = (pg < prod_end) ? __ldg(p.block_tables + (int64_t)prod_row * W + pg) : -1;
    }
    if (prod_page - win_base >= 32) {
      win_base += 32;
      blk_win = blk_win2;
    }
    const int blk = __shfl_sync(0xffffffffu, blk_win, prod_page - win_base);
    if (lane == 0) {
      ws.stage_item[st] = prod_slot;
      ws.stage_page[st] = prod_page;
      uint32_t bytes = 2u * kPageBytes + (first ? (uint32_t)kQBytes : 0u);
      const bool ok_blk = blk >= 0 && blk < p.num_blocks;
      if (!ok_blk) {
        set_error(p.error_word, CB_DEVERR_BLOCK_RANGE);
        bytes = first ? (uint32_t)kQBytes : 0u;
      }
      // the stage's previous contents were read (generic proxy) before the
      // __syncwarp that precedes this call; the copies below only write it
      mbar_arrive_expect_tx(&ws.full[st], bytes);
      // test hook: the withheld item's first page is announced but never
      // copied, so the consumer's bounded wait on it runs out
      const bool withhold = first && prod_idx == p.withhold_item;
      if (first && !withhold) {
        const ItemDesc& d = ws.items[prod_slot];
        const uint8_t* qsrc = static_cast<const uint8_t*>(p.q) +
                              ((int64_t)d.token * Hq + (int64_t)prod_g * G) * D * sizeof(T);
        bulk_copy_g2s(ws.q[prod_slot], qsrc, kQBytes, &ws.full[st]);
      }
      if (ok_blk && !withhold) {
        if constexpr (kMma) {
          const int row = (blk * Hkv + prod_g) * kPageTokens;
#pragma unroll
          for (int hf = 0; hf < D / 64; ++hf) {
            tma_load_2d_hint(ws.kv[st][0] + hf * 2048, &p.tmap_k, hf * 64, row, &ws.full[st], pol);
            tma_load_2d_hint(ws.kv[st][1] + hf * 2048, &p.tmap_v, hf * 64, row, &ws.full[st], pol);
          }
        } else {
          const int64_t off = ((int64_t)blk * Hkv + prod_g) * kPageBytes;
          bulk_copy_g2s_hint(ws.kv[st][0], kbase + off, kPageBytes, &ws.full[st], pol);
          bulk_copy_g2s_hint(ws.kv[st][1], vbase + off, kPageBytes, &ws.full[st], pol);
        }
      } else if (!ok_blk) {
        // unreadable page: zero it so the math stays finite
        uint4* z = reinterpret_cast<uint4*>(ws.kv[st][0]);
        for (int k = 0; k < 2 * kPageBytes / 16; ++k) z[k] = make_uint4(0, 0, 0, 0);
      }
    }
    ++prod_page;
    ++issued;
    __syncwarp();
  };

  // ---- split tickets ----------------------------------------------------------
  // Count one split of (row i, KV head g) done; the warp whose ticket
  // completes the count of n merges the row's splits and leaves the counter
  // zero.  The count follows a fence, so the merging warp sees every
  // partial.  A warp that aborted still counts its splits (so counters
  // return to zero) but merges nothing.
  auto ticket = [&](int i, int g, int n) {
    __threadfence();
    __syncwarp();
    uint32_t* cnt = p.done + (int64_t)i * Hkv + g;
    uint32_t old = 0;
    if (lane == 0) old = atomicAdd(cnt, 1u);
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old == (uint32_t)n - 1) {
      __threadfence();
      if (!aborted) merge_splits<T, D, G>(p, g, plan_a[i] + plan_b[i], n, row_tok[i], lane);
      __syncwarp();
      if (lane == 0) *cnt = 0u;
    }
  };
  // (row, KV head, splits) of this warp's last partial, not yet counted
  // done: counted when the warp writes its next partial (or finishes), by
  // when the stores are long complete and the fence rarely waits
  int pend_i = -1, pend_g = 0, pend_n = 0;
  auto flush_pending = [&]() {
    if (pend_i >= 0) {
      ticket(pend_i, pend_g, pend_n);
      pend_i = -1;
    }
  };

  // The cache is read from here on.  Launched right after the step's K/V
  // append (programmatic dependent launch), the grid planned while the
  // append finished and waits for it here (a no-op without such a launch;
  // skipped when the grid before is the prefill rows of the same call, which
  // write nothing it reads).  Only then may a kernel launched after this one
  // with programmatic serialization (the prefill rows of the same call,
  // which read nothing this kernel writes but do read the appended K/V)
  // start on the SMs this grid leaves.
  if (p.pdl_mode != 2) asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int s = 0; s < kStages; ++s) produce(s);

  if constexpr (kMma) {
    // ======================= matrix-instruction path (bf16) =====================
    using M = MmaCfg<D, G>;
    constexpr int kNT = M::kNT, kKS = M::kKS, kMT = M::kMT;
    // lane roles in the m16n8k16 fragments: rows (tokens / dims) grp and
    // grp + 8, columns (heads / tokens) 2 * qd and 2 * qd + 1
    const int grp = lane >> 2;
    const int qd = lane & 3;
    // ldmatrix row addresses: matrix mi = lane / 8, row rr = lane % 8
    const int mi = lane >> 3;
    const int rr = lane & 7;
    const int k_tok = rr + ((mi & 1) << 3);   // K: matrices (tokens 0-7 | 8-15) x (dims lo | hi)
    const int k_gc = mi >> 1;
    const int v_tok = rr + ((mi >> 1) << 3);  // V^T: matrices (dims lo | hi) x (tokens 0-7 | 8-15)
    const int v_gc = mi & 1;

    uint32_t qb[kNT][kKS][2];      // Q^T B fragments of the current item
    float acc[kNT][kMT][4];        // O^T accumulators (dims x heads)
    float m_run[kNT][2], l_run[kNT][2];
    int cur_slot = -1;

    int st = 0;
    while (consumed < issued) {
      {
        // always wait (bounded) so no copy is still landing when the CTA exits
        const bool ok = mbar_wait(&ws.full[st], (phases >> st) & 1u, p.wait_ns);
        if (!__all_sync(0xffffffffu, ok)) {
          if (!aborted && lane == 0) set_error(p.error_word, CB_DEVERR_TIMEOUT);
          aborted = true;
        }
      }
      phases ^= 1u << st;
      ++consumed;
      const int slot = ws.stage_item[st];
      const int page = ws.stage_page[st];
      const ItemDesc d = ws.items[slot];
      if (!aborted) {
        if (slot != cur_slot || page == d.page0) {
          // new item: load Q^T, reset the state
          cur_slot = slot;
          const uint32_t qs = smem_addr(ws.q[slot]);
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt) {
            const int head = nt * 8 + rr;
            const int hrow = head < G ? head : 0;
#pragma unroll
            for (int kk = 0; kk < kKS; kk += 2) {
              uint32_t f[4];
              ldsm_x4(qs + hrow * (D * 2) + (2 * kk + mi) * 16, f);
              const bool live = nt * 8 + grp < G;
              qb[nt][kk][0] = live ? f[0] : 0u;
              qb[nt][kk][1] = live ? f[1] : 0u;
              qb[nt][kk + 1][0] = live ? f[2] : 0u;
              qb[nt][kk + 1][1] = live ? f[3] : 0u;
            }
#pragma unroll
            for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
              for (int e = 0; e < 4; ++e) acc[nt][mt][e] = 0.f;
            m_run[nt][0] = m_run[nt][1] = -INFINITY;
            l_run[nt][0] = l_run[nt][1] = 0.f;
          }
        }
        // keys [lo_t, valid) of this page are read: the sequence end on the
        // last page, the window start on the first
        const int valid = min(kPageTokens, d.seq_len - page * kPageTokens);
        const int lo_t = first_key(d.seq_len, win) - page * kPageTokens;
        const uint32_t kp = smem_addr(ws.kv[st][0]);
        const uint32_t vp = smem_addr(ws.kv[st][1]);

        // ---- S^T = K Q^T: two accumulator chains over the k-steps --------------
        float s[kNT][4], s2[kNT][4];
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) s[nt][e] = s2[nt][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < kKS; ++kk) {
          uint32_t a[4];
          ldsm_x4(kp + swz_off(k_tok, 2 * kk + k_gc), a);
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt) {
            if (kk & 1)
              mma_bf16(s2[nt], a, qb[nt][kk][0], qb[nt][kk][1]);
            else
              mma_bf16(s[nt], a, qb[nt][kk][0], qb[nt][kk][1]);
          }
        }
        // ---- online softmax (base 2) per head ------------------------------------
        // this lane: tokens grp and grp + 8, heads nt*8 + 2qd and nt*8 + 2qd + 1
        const bool v0 = grp < valid && grp >= lo_t;
        const bool v1 = grp + 8 < valid && grp + 8 >= lo_t;
        const float sl = p.scale_log2;
        uint32_t pb[kNT][2];
        bool resc = false;
        float alpha[kNT][2];
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          float x[4];
          x[0] = v0 ? (s[nt][0] + s2[nt][0]) * sl : -INFINITY;
          x[1] = v0 ? (s[nt][1] + s2[nt][1]) * sl : -INFINITY;
          x[2] = v1 ? (s[nt][2] + s2[nt][2]) * sl : -INFINITY;
          x[3] = v1 ? (s[nt][3] + s2[nt][3]) * sl : -INFINITY;
          float pm0 = fmaxf(x[0], x[2]), pm1 = fmaxf(x[1], x[3]);
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) {
            pm0 = fmaxf(pm0, __shfl_xor_sync(0xffffffffu, pm0, o));
            pm1 = fmaxf(pm1, __shfl_xor_sync(0xffffffffu, pm1, o));
          }
          // the reference max moves only when a page raises it by more than 8
          // (weights stay <= 2^8); a partial's (m, l, acc) share whatever
          // reference it ends with
          float mu[2];
          const float pmv[2] = {pm0, pm1};
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const float mn = fmaxf(m_run[nt][c], pmv[c]);
            mu[c] = (mn - m_run[nt][c] > 8.f) ? mn : m_run[nt][c];
            alpha[nt][c] = (mu[c] == m_run[nt][c]) ? 1.f : ex2_approx(m_run[nt][c] - mu[c]);
            resc |= alpha[nt][c] != 1.f;
            m_run[nt][c] = mu[c];
          }
          // P rounded to bf16 (the MMA operand); l adds the rounded values
          const uint32_t p0 = float2_to_bf16x2(ex2_approx(x[0] - mu[0]), ex2_approx(x[1] - mu[1]));
          const uint32_t p1 = float2_to_bf16x2(ex2_approx(x[2] - mu[0]), ex2_approx(x[3] - mu[1]));
          const float2 f0 = bf16x2_to_float2(p0), f1 = bf16x2_to_float2(p1);
          l_run[nt][0] = l_run[nt][0] * alpha[nt][0] + (f0.x + f1.x);
          l_run[nt][1] = l_run[nt][1] * alpha[nt][1] + (f0.y + f1.y);
          // P^T as the B operand: (tokens 2qd.., head grp) from (token grp, heads 2qd..)
          pb[nt][0] = movmatrix_trans(p0);
          pb[nt][1] = movmatrix_trans(p1);
        }
        if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
            for (int mt = 0; mt < kMT; ++mt) {
              acc[nt][mt][0] *= alpha[nt][0];
              acc[nt][mt][1] *= alpha[nt][1];
              acc[nt][mt][2] *= alpha[nt][0];
              acc[nt][mt][3] *= alpha[nt][1];
            }
        }
        // ---- O^T += V^T P^T ----------------------------------------------------------
        // Slots past the sequence end hold whatever the pool held (possibly
        // not finite), so on a partial page the V values of masked tokens
        // are zeroed in the fragments; full pages skip the masking.
        const bool partial = valid < kPageTokens || lo_t > 0;
        uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
        if (partial) {
          const int t0 = 2 * qd, t1 = 2 * qd + 8;
          mlo = ((t0 < valid && t0 >= lo_t) ? 0x0000ffffu : 0u) |
                ((t0 + 1 < valid && t0 + 1 >= lo_t) ? 0xffff0000u : 0u);
          mhi = ((t1 < valid && t1 >= lo_t) ? 0x0000ffffu : 0u) |
                ((t1 + 1 < valid && t1 + 1 >= lo_t) ? 0xffff0000u : 0u);
        }
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt) {
          uint32_t a[4];
          ldsm_x4_trans(vp + swz_off(v_tok, 2 * mt + v_gc), a);
          a[0] &= mlo; a[1] &= mlo; a[2] &= mhi; a[3] &= mhi;
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt) mma_bf16(acc[nt][mt], a, pb[nt][0], pb[nt][1]);
        }
      }
      // ---- item end ------------------------------------------------------------------
      if (page + 1 == d.page1) {
        ++cons_items;
        if (!aborted) {
          float lsum[kNT][2];
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              float l = l_run[nt][c];
#pragma unroll
              for (int o = 4; o < 32; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
              lsum[nt][c] = l;
            }
          if (d.nsplit == 1) {
            T* orow = static_cast<T*>(p.out) + ((int64_t)d.token * Hq + (int64_t)d.g * G) * D;
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
              for (int c = 0; c < 2; ++c) {
                const int h = nt * 8 + 2 * qd + c;
                if (h < G) {
                  const float inv = 1.f / lsum[nt][c];
                  T* hrow = orow + h * D;
#pragma unroll
                  for (int mt = 0; mt < kMT; ++mt) {
                    hrow[mt * 16 + grp] = __float2bfloat16_rn(acc[nt][mt][c] * inv);
                    hrow[mt * 16 + grp + 8] = __float2bfloat16_rn(acc[nt][mt][c + 2] * inv);
                  }
                }
              }
          } else {
            // count the previous partial of this warp done first: its stores
            // were issued an item ago, so the fence rarely waits
            flush_pending();
            const int64_t pslot = (int64_t)d.slot * Hkv + d.g;
            float* pacc = p.part_acc + pslot * G * D;
            float* pml = p.part_ml + pslot * G * 2;
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
              for (int c = 0; c < 2; ++c) {
                const int h = nt * 8 + 2 * qd + c;
                if (h < G) {
                  float* hrow = pacc + h * D;
#pragma unroll
                  for (int mt = 0; mt < kMT; ++mt) {
                    hrow[mt * 16 + grp] = acc[nt][mt][c];
                    hrow[mt * 16 + grp + 8] = acc[nt][mt][c + 2];
                  }
                  if (grp == 0) {
                    pml[h * 2 + 0] = m_run[nt][c];
                    pml[h * 2 + 1] = lsum[nt][c];
                  }
                }
              }
            pend_i = d.r;
            pend_g = d.g;
            pend_n = d.nsplit;
          }
        } else if (d.nsplit > 1) {
          ticket(d.r, d.g, d.nsplit);
        }
      }
      __syncwarp();
      produce(st);
      st = (st + 1 == kStages) ? 0 : st + 1;
    }
  } else {
    // ========================= CUDA-core path (fp32) ============================
    using C = Cfg<T, D, G>;
    // lane geometry
    const int tok = lane / C::kLG;
    const int j = lane - tok * C::kLG;

    float qf[G][C::kDPL];
    float acc[G][C::kDPL];
    float m_own = -INFINITY, l_own = 0.f;
    int cur_slot = -1;

    int st = 0;
    while (consumed < issued) {
      {
        const bool ok = mbar_wait(&ws.full[st], (phases >> st) & 1u, p.wait_ns);
        if (!__all_sync(0xffffffffu, ok)) {
          if (!aborted && lane == 0) set_error(p.error_word, CB_DEVERR_TIMEOUT);
          aborted = true;
        }
      }
      phases ^= 1u << st;
      ++consumed;
      const int slot = ws.stage_item[st];
      const int page = ws.stage_page[st];
      const ItemDesc d = ws.items[slot];
      if (!aborted) {
        if (slot != cur_slot || page == d.page0) {
          // new item: load and pre-scale q, reset the online-softmax state
          cur_slot = slot;
          const T* qrow = reinterpret_cast<const T*>(ws.q[slot]);
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const uint4* qv = reinterpret_cast<const uint4*>(qrow + h * D);
#pragma unroll
            for (int c = 0; c < C::kCPL; ++c) {
              float f[C::kEPC];
              unpack16<T>(qv[j + C::kLG * c], f);
#pragma unroll
              for (int e = 0; e < C::kEPC; ++e) qf[h][c * C::kEPC + e] = f[e] * p.scale_log2;
            }
#pragma unroll
            for (int e = 0; e < C::kDPL; ++e) acc[h][e] = 0.f;
          }
          m_own = -INFINITY;
          l_own = 0.f;
        }
        const int valid = min(kPageTokens, d.seq_len - page * kPageTokens);
        const int lo_t = first_key(d.seq_len, win) - page * kPageTokens;
        const uint8_t* kp = ws.kv[st][0];
        const uint8_t* vp = ws.kv[st][1];

        // ---- scores -----------------------------------------------------------
        float sc[C::kNIT];
#pragma unroll
        for (int it = 0; it < C::kNIT; ++it) {
          const int t = it * C::kTPI + tok;
          const uint4* krow = reinterpret_cast<const uint4*>(kp + t * C::kRowBytes);
          float2 part2[G];
#pragma unroll
          for (int h = 0; h < G; ++h) part2[h] = make_float2(0.f, 0.f);
#pragma unroll
          for (int c = 0; c < C::kCPL; ++c) {
            float kf[C::kEPC];
            unpack16<T>(krow[j + C::kLG * c], kf);
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
              for (int e = 0; e < C::kEPC; e += 2)
                part2[h] = __ffma2_rn(make_float2(qf[h][c * C::kEPC + e], qf[h][c * C::kEPC + e + 1]),
                                      make_float2(kf[e], kf[e + 1]), part2[h]);
          }
          float v[G];
#pragma unroll
          for (int h = 0; h < G; ++h) v[h] = part2[h].x + part2[h].y;
          // butterfly reduce-scatter over the LG lanes of this token
          int cnt = G;
#pragma unroll
          for (int o = C::kLG / 2; o >= 1; o >>= 1) {
            if (cnt > 1) {
              const int half = cnt / 2;
              const bool upper = (j & o) != 0;
#pragma unroll
              for (int k = 0; k < G / 2; ++k) {
                if (k < half) {
                  const float send = upper ? v[k] : v[k + half];
                  const float keep = upper ? v[k + half] : v[k];
                  v[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
              }
              cnt = half;
            } else {
              v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
            }
          }
          sc[it] = (t < valid && t >= lo_t) ? v[0] : -INFINITY;
        }

        // ---- online softmax (base 2) -------------------------------------------
        float pm = sc[0];
#pragma unroll
        for (int it = 1; it < C::kNIT; ++it) pm = fmaxf(pm, sc[it]);
#pragma unroll
        for (int o = C::kLG; o < 32; o <<= 1) pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, o));
        const float m_new = fmaxf(m_own, pm);
        const float m_use = (m_new - m_own > 8.f) ? m_new : m_own;
        const float a_own = (m_use == m_own) ? 1.f : ex2_approx(m_own - m_use);
        m_own = m_use;
        float pr[C::kNIT];
        float psum = 0.f;
#pragma unroll
        for (int it = 0; it < C::kNIT; ++it) {
          pr[it] = ex2_approx(sc[it] - m_own);
          psum += pr[it];
        }
        l_own = l_own * a_own + psum;
        if (!__all_sync(0xffffffffu, a_own == 1.f)) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float a = __shfl_sync(0xffffffffu, a_own, h * C::kDup);
#pragma unroll
            for (int e = 0; e < C::kDPL; ++e) acc[h][e] *= a;
          }
        }

        // ---- P.V ------------------------------------------------------------------
        auto pv = [&](auto mask_tag) {
          constexpr bool kMask = decltype(mask_tag)::value;
#pragma unroll
          for (int it = 0; it < C::kNIT; ++it) {
            const int t = it * C::kTPI + tok;
            const uint4* vrow = reinterpret_cast<const uint4*>(vp + t * C::kRowBytes);
            float ph[G];
#pragma unroll
            for (int h = 0; h < G; ++h) ph[h] = __shfl_sync(0xffffffffu, pr[it], tok * C::kLG + h * C::kDup);
            const bool tv = t < valid && t >= lo_t;
#pragma unroll
            for (int c = 0; c < C::kCPL; ++c) {
              float vf[C::kEPC];
              unpack16<T>(vrow[j + C::kLG * c], vf);
              if constexpr (kMask) {
#pragma unroll
                for (int e = 0; e < C::kEPC; ++e) vf[e] = tv ? vf[e] : 0.f;
              }
#pragma unroll
              for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < C::kEPC; e += 2) {
                  float2 a2 = make_float2(acc[h][c * C::kEPC + e], acc[h][c * C::kEPC + e + 1]);
                  a2 = __ffma2_rn(make_float2(ph[h], ph[h]), make_float2(vf[e], vf[e + 1]), a2);
                  acc[h][c * C::kEPC + e] = a2.x;
                  acc[h][c * C::kEPC + e + 1] = a2.y;
                }
            }
          }
        };
        if (valid == kPageTokens && lo_t <= 0)
          pv(std::false_type{});
        else
          pv(std::true_type{});
      }

      // ---- item end -------------------------------------------------------------
      if (page + 1 == d.page1) {
        ++cons_items;
        if (!aborted) {
#pragma unroll
          for (int o = C::kLG; o < 32; o <<= 1) {
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
              for (int e = 0; e < C::kDPL; ++e) acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], o);
            l_own += __shfl_xor_sync(0xffffffffu, l_own, o);
          }
          if (d.nsplit == 1) {
            T* orow = static_cast<T*>(p.out) + ((int64_t)d.token * Hq + (int64_t)d.g * G) * D;
#pragma unroll
            for (int h = 0; h < G; ++h) {
              const float l = __shfl_sync(0xffffffffu, l_own, h * C::kDup);
              if (h % C::kTPI == tok) {
                float o[C::kDPL];
                const float inv = 1.f / l;
#pragma unroll
                for (int e = 0; e < C::kDPL; ++e) o[e] = acc[h][e] * inv;
                store_row<T, D, G>(orow + h * D, j, o);
              }
            }
          } else {
            flush_pending();
            const int64_t pslot = (int64_t)d.slot * Hkv + d.g;
            float* pacc = p.part_acc + pslot * G * D;
            float* pml = p.part_ml + pslot * G * 2;
#pragma unroll
            for (int h = 0; h < G; ++h) {
              const float l = __shfl_sync(0xffffffffu, l_own, h * C::kDup);
              const float m = __shfl_sync(0xffffffffu, m_own, h * C::kDup);
              if (h % C::kTPI == tok) {
#pragma unroll
                for (int c = 0; c < C::kCPL; ++c) {
                  float4* dst = reinterpret_cast<float4*>(pacc + h * D);
#pragma unroll
                  for (int e = 0; e < C::kEPC; e += 4) {
                    const int fi = (j + C::kLG * c) * C::kEPC + e;
                    dst[fi / 4] = make_float4(acc[h][c * C::kEPC + e], acc[h][c * C::kEPC + e + 1],
                                              acc[h][c * C::kEPC + e + 2],
                                              acc[h][c * C::kEPC + e + 3]);
                  }
                }
                if (j == 0) {
                  pml[h * 2 + 0] = m;
                  pml[h * 2 + 1] = l;
                }
              }
            }
            pend_i = d.r;
            pend_g = d.g;
            pend_n = d.nsplit;
          }
        } else if (d.nsplit > 1) {
          ticket(d.r, d.g, d.nsplit);
        }
      }
      __syncwarp();
      produce(st);
      st = (st + 1 == kStages) ? 0 : st + 1;
    }
  }

  // ---- finish -------------------------------------------------------------------
  // count the last partial; after an abort, also every split this warp
  // started but did not finish and every split still dealt to it, so each
  // (row, KV head) counter still reaches its count and returns to zero
  flush_pending();
  if (aborted) {
    for (int k = cons_items; k < prod_items; ++k) {
      const ItemDesc d = ws.items[k % kRing];
      if (d.nsplit > 1) ticket(d.r, d.g, d.nsplit);
    }
    while (nx_ok) {
      const int i = nx_i, g = nx_g, n = nx_nsplit;
      fetch_ahead();
      if (n > 1) ticket(i, g, n);
    }
  }
  // beside the prefill grid before it: this grid completes only after it
  if (p.pdl_mode == 2 && blockIdx.x == 0 && threadIdx.x == 0)
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace decode
}  // namespace cb
