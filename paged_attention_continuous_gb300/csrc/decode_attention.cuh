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
//     16-token pages of one request and one KV head.  Items are handed out
//     through a global atomic counter (dynamic load balance).  The split
//     size is chosen in the kernel from the total page count so every warp
//     gets several items; a request gets at most kMaxSplits splits.
//   * Every WARP is an independent worker with its own pipeline: lane 0 issues
//     cp.async.bulk copies (TMA engine, 1-D) of the (block, head) K page and V
//     page -- each one contiguous block_size*D run in the cache layout
//     [num_blocks][Hkv][16][D] -- into a ring of kStages shared-memory stages,
//     each tracked by an mbarrier.  The ring runs across item boundaries, so
//     the next item's pages are already in flight when one item ends.
//   * The GQA group's G query heads share each K/V byte.  LG lanes cover one
//     token's D dims (16-byte vectors, conflict-free), 32/LG tokens per warp
//     iteration; partial dot products of the G heads are combined with a
//     butterfly reduce-scatter (warp shuffles), so each lane ends with one
//     (token, head) score.  Online softmax in base 2 with the scale folded
//     into q; P.V accumulates in fp32 registers (packed f32x2 FMAs).
//   * Splits write (m, l, acc) partials; the last split of a (request, head)
//     to finish -- an atomic ticket, no spin-wait -- merges them with the
//     log-sum-exp rescale and writes the output.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "device_utils.cuh"

namespace cb {
namespace decode {

constexpr int kPageTokens = 16;
constexpr int kMaxSplits = 32;
constexpr int kMinSplitPages = 8;
constexpr int kItemsPerWarp = 6;
constexpr int kPlanMax = 1024;  // decode rows planned per launch

struct Params {
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
  uint32_t* error_word;
  uint32_t* work_counter;
  uint32_t* tickets;       // [num_rows * Hkv], zero between launches
  float* part_ml;          // [slots][Hkv][G][2]
  float* part_acc;         // [slots][Hkv][G][D]
};

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
  static constexpr int kPageBytes = kPageTokens * kRowBytes;
  static constexpr int kQBytes = G * D * kElem;
  static_assert(kRowBytes % 16 == 0, "row must be a multiple of 16 bytes");
  static_assert(kLG >= G && kLG % G == 0, "group must divide lanes per token");
  static_assert(kChunks % kLG == 0, "vectors must split evenly over lanes");
};

struct ItemDesc {
  int32_t r, g, split, nsplit, page0, page1, seq_len, token, slot;
  int32_t pad[3];
};

template <typename T, int D, int G, int kStages>
struct WarpSmem {
  using C = Cfg<T, D, G>;
  static constexpr int kRing = kStages + 1;
  alignas(128) uint8_t kv[kStages][2][C::kPageBytes];
  alignas(16) uint8_t q[kRing][C::kQBytes];
  ItemDesc items[kRing];
  uint64_t full[kStages];
  int32_t stage_item[kStages];
  int32_t stage_page[kStages];
};

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

__device__ __forceinline__ int split_pages_for(int pages, int base_split) {
  const int need = (pages + kMaxSplits - 1) / kMaxSplits;
  return base_split > need ? base_split : need;
}

template <typename T, int D, int G, int kWarps, int kStages>
__global__ void __launch_bounds__(kWarps * 32, 1) decode_kernel(const Params p) {
  using C = Cfg<T, D, G>;
  using WS = WarpSmem<T, D, G, kStages>;
  constexpr int kRing = WS::kRing;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  WS* wsm_all = reinterpret_cast<WS*>(smem_raw);
  int32_t* plan = reinterpret_cast<int32_t*>(smem_raw + sizeof(WS) * kWarps);  // [num_rows + 1]
  __shared__ int32_t s_red[kWarps];
  __shared__ int32_t s_split_pages;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nthreads = kWarps * 32;
  const int Hkv = p.num_kv_heads;
  const int Hq = p.num_q_heads;
  const int W = p.max_blocks_per_seq;

  // ---- plan: pages per row -> split size -> prefix of split counts --------
  int64_t my_pages = 0;
  for (int i = threadIdx.x; i < p.num_rows; i += nthreads) {
    const int r = p.row_begin + i;
    const int L = p.seq_lens[r];
    int pages = (L + kPageTokens - 1) / kPageTokens;
    if (L < 1 || pages > W) {
      pages = 0;
      if (blockIdx.x == 0) set_error(p.error_word, CB_DEVERR_SEQ_RANGE);
    }
    my_pages += pages;
  }
  for (int o = 16; o > 0; o >>= 1) my_pages += __shfl_xor_sync(0xffffffffu, my_pages, o);
  if (lane == 0) s_red[warp] = (int32_t)(my_pages < 0x3fffffff ? my_pages : 0x3fffffff);
  __syncthreads();
  if (threadIdx.x == 0) {
    int64_t tot = 0;
    for (int w = 0; w < kWarps; ++w) tot += s_red[w];
    const int64_t workers = (int64_t)gridDim.x * kWarps * kItemsPerWarp;
    int64_t sp = (tot * Hkv + workers - 1) / workers;
    if (sp < kMinSplitPages) sp = kMinSplitPages;
    s_split_pages = (int32_t)(sp < (1 << 20) ? sp : (1 << 20));
  }
  __syncthreads();
  const int base_split = s_split_pages;
  // serial-per-thread segments + shared scan of segment sums
  {
    const int seg = (p.num_rows + nthreads - 1) / nthreads;
    const int b = threadIdx.x * seg;
    const int e = min(b + seg, p.num_rows);
    int sum = 0;
    for (int i = b; i < e; ++i) {
      const int r = p.row_begin + i;
      const int L = p.seq_lens[r];
      int pages = (L + kPageTokens - 1) / kPageTokens;
      int ns = 0;
      if (L >= 1 && pages <= W) {
        const int sp = split_pages_for(pages, base_split);
        ns = (pages + sp - 1) / sp;
      }
      plan[i + 1] = ns;
      sum += ns;
    }
    // inclusive scan of per-thread sums
    int incl = sum;
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) s_red[warp] = incl;
    __syncthreads();
    int warp_off = 0;
    for (int w = 0; w < warp; ++w) warp_off += s_red[w];
    int run = warp_off + incl - sum;  // exclusive prefix of this thread's segment
    if (threadIdx.x == 0) plan[0] = 0;
    for (int i = b; i < e; ++i) {
      run += plan[i + 1];
      plan[i + 1] = run;
    }
  }
  __syncthreads();
  const int total_items = plan[p.num_rows] * Hkv;
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
  int win_base = 0;        // first page covered by blk_win
  int blk_win = -1;        // lane i holds the block id of page win_base + i
  bool exhausted = false;
  bool aborted = false;
  int prod_row = 0, prod_g = 0;
  uint32_t phases = 0;     // parity bit per stage
  int issued = 0, consumed = 0;

  // grab the next item and describe it in the ring; false when none is left
  auto next_item = [&]() -> bool {
    while (true) {
      uint32_t idx = 0;
      if (lane == 0) idx = atomicAdd(p.work_counter, 1u);
      idx = __shfl_sync(0xffffffffu, idx, 0);
      if (idx >= (uint32_t)total_items) {
        if (idx == (uint32_t)total_items + total_workers - 1 && lane == 0) atomicExch(p.work_counter, 0u);
        return false;
      }
      // row: largest i with plan[i] * Hkv <= idx
      int lo = 0, hi = p.num_rows - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (plan[mid] * Hkv <= (int)idx) lo = mid; else hi = mid - 1;
      }
      const int i = lo;
      const int local = (int)idx - plan[i] * Hkv;
      const int split = local / Hkv;
      const int g = local - split * Hkv;
      const int r = p.row_begin + i;
      const int L = p.seq_lens[r];
      const int pages = (L + kPageTokens - 1) / kPageTokens;
      const int sp = split_pages_for(pages, base_split);
      const int nsplit = plan[i + 1] - plan[i];
      const int q0 = p.cu_seqlens_q[r];
      const int q1 = p.cu_seqlens_q[r + 1];
      if (q1 - q0 != 1 || q0 < 0 || q0 >= p.num_tokens) {
        if (lane == 0 && split == 0 && g == 0) set_error(p.error_word, CB_DEVERR_DECODE_QLEN);
        continue;
      }
      const int slot_i = (prod_items) % kRing;
      ++prod_items;
      prod_slot = slot_i;
      prod_row = r;
      prod_g = g;
      prod_page = split * sp;
      prod_end = min(pages, prod_page + sp);
      if (lane == 0) {
        ItemDesc& d = ws.items[slot_i];
        d.r = i; d.g = g; d.split = split; d.nsplit = nsplit;
        d.page0 = prod_page; d.page1 = prod_end; d.seq_len = L; d.token = q0;
        d.slot = plan[i] + split;
      }
      win_base = prod_page;
      const int pg = win_base + lane;
      blk_win = (pg < prod_end) ? p.block_tables[(int64_t)r * W + pg] : -1;
      return true;
    }
  };

  // refill one stage with the producer's next page (whole warp calls this)
  auto produce = [&](int st) {
    if (exhausted || aborted) return;
    bool first = false;
    if (prod_slot < 0 || prod_page >= prod_end) {
      if (!next_item()) { exhausted = true; return; }
      first = true;
    }
    if (prod_page - win_base >= 32) {
      win_base = prod_page;
      const int pg = win_base + lane;
      blk_win = (pg < prod_end) ? p.block_tables[(int64_t)prod_row * W + pg] : -1;
    }
    const int blk = __shfl_sync(0xffffffffu, blk_win, prod_page - win_base);
    if (lane == 0) {
      ws.stage_item[st] = prod_slot;
      ws.stage_page[st] = prod_page;
      uint32_t bytes = 2u * C::kPageBytes + (first ? (uint32_t)C::kQBytes : 0u);
      const bool ok_blk = blk >= 0 && blk < p.num_blocks;
      if (!ok_blk) {
        set_error(p.error_word, CB_DEVERR_BLOCK_RANGE);
        bytes = first ? (uint32_t)C::kQBytes : 0u;
      }
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&ws.full[st], bytes);
      if (first) {
        const ItemDesc& d = ws.items[prod_slot];
        const uint8_t* qsrc = static_cast<const uint8_t*>(p.q) +
                              ((int64_t)d.token * Hq + (int64_t)prod_g * G) * D * C::kElem;
        bulk_copy_g2s(ws.q[prod_slot], qsrc, C::kQBytes, &ws.full[st]);
      }
      if (ok_blk) {
        const int64_t off = ((int64_t)blk * Hkv + prod_g) * C::kPageBytes;
        bulk_copy_g2s_hint(ws.kv[st][0], kbase + off, C::kPageBytes, &ws.full[st], pol);
        bulk_copy_g2s_hint(ws.kv[st][1], vbase + off, C::kPageBytes, &ws.full[st], pol);
      } else {
        // unreadable page: zero it so the math stays finite
        uint4* z = reinterpret_cast<uint4*>(ws.kv[st][0]);
        for (int k = 0; k < 2 * C::kPageBytes / 16; ++k) z[k] = make_uint4(0, 0, 0, 0);
      }
    }
    ++prod_page;
    ++issued;
    __syncwarp();
  };

  // lane geometry
  const int tok = lane / C::kLG;
  const int j = lane - tok * C::kLG;
  const int hh = j / C::kDup;                // head whose score this lane ends with

  float qf[G][C::kDPL];
  float acc[G][C::kDPL];
  float m_own = -INFINITY, l_own = 0.f;
  int cur_slot = -1;

  for (int s = 0; s < kStages; ++s) produce(s);

  int st = 0;
  while (consumed < issued) {
    {
      // always wait (bounded) so no copy is still landing when the CTA exits
      const bool ok = mbar_wait(&ws.full[st], (phases >> st) & 1u);
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
        sc[it] = (t < valid) ? v[0] : -INFINITY;
      }

      // ---- online softmax (base 2) -------------------------------------------
      float pm = sc[0];
#pragma unroll
      for (int it = 1; it < C::kNIT; ++it) pm = fmaxf(pm, sc[it]);
#pragma unroll
      for (int o = C::kLG; o < 32; o <<= 1) pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, o));
      const float m_new = fmaxf(m_own, pm);
      const float a_own = exp2f(m_own - m_new);
      m_own = m_new;
      float pr[C::kNIT];
      float psum = 0.f;
#pragma unroll
      for (int it = 0; it < C::kNIT; ++it) {
        pr[it] = exp2f(sc[it] - m_new);
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
#pragma unroll
      for (int it = 0; it < C::kNIT; ++it) {
        const int t = it * C::kTPI + tok;
        const uint4* vrow = reinterpret_cast<const uint4*>(vp + t * C::kRowBytes);
        float ph[G];
#pragma unroll
        for (int h = 0; h < G; ++h) ph[h] = __shfl_sync(0xffffffffu, pr[it], tok * C::kLG + h * C::kDup);
        const bool tv = t < valid;
#pragma unroll
        for (int c = 0; c < C::kCPL; ++c) {
          float vf[C::kEPC];
          unpack16<T>(vrow[j + C::kLG * c], vf);
#pragma unroll
          for (int e = 0; e < C::kEPC; ++e) vf[e] = tv ? vf[e] : 0.f;
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

      // ---- item end -------------------------------------------------------------
      if (page + 1 == d.page1) {
#pragma unroll
        for (int o = C::kLG; o < 32; o <<= 1) {
#pragma unroll
          for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < C::kDPL; ++e) acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], o);
          l_own += __shfl_xor_sync(0xffffffffu, l_own, o);
        }
        const int r = p.row_begin + d.r;
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
                float4* dst = reinterpret_cast<float4*>(pacc + h * D) ;
                // element index of vector (j + LG*c) in floats: (j + LG*c) * kEPC
#pragma unroll
                for (int e = 0; e < C::kEPC; e += 4) {
                  const int fi = (j + C::kLG * c) * C::kEPC + e;
                  dst[fi / 4] = make_float4(acc[h][c * C::kEPC + e], acc[h][c * C::kEPC + e + 1],
                                            acc[h][c * C::kEPC + e + 2], acc[h][c * C::kEPC + e + 3]);
                }
              }
              if (j == 0) {
                pml[h * 2 + 0] = m;
                pml[h * 2 + 1] = l;
              }
            }
          }
          __threadfence();
          __syncwarp();
          uint32_t ticket = 0;
          if (lane == 0) ticket = atomicAdd(p.tickets + (int64_t)d.r * Hkv + d.g, 1u);
          ticket = __shfl_sync(0xffffffffu, ticket, 0);
          if (ticket == (uint32_t)d.nsplit - 1) {
            // last split of (row, head): merge partials
            __threadfence();
            if (lane == 0) p.tickets[(int64_t)d.r * Hkv + d.g] = 0u;
            const int64_t base = (int64_t)(d.slot - d.split) * Hkv + d.g;
            constexpr int kVec = G * D / 4;  // float4 outputs per (row, head group)
            T* orow = static_cast<T*>(p.out) + ((int64_t)d.token * Hq + (int64_t)d.g * G) * D;
            for (int v4 = lane; v4 < kVec; v4 += 32) {
              const int h = v4 / (D / 4);
              float M = -INFINITY;
              for (int s = 0; s < d.nsplit; ++s)
                M = fmaxf(M, __ldcg(p.part_ml + ((base + (int64_t)s * Hkv) * G + h) * 2));
              float L = 0.f;
              float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
              for (int s = 0; s < d.nsplit; ++s) {
                const int64_t ps = base + (int64_t)s * Hkv;
                const float ms = __ldcg(p.part_ml + (ps * G + h) * 2);
                const float ls = __ldcg(p.part_ml + (ps * G + h) * 2 + 1);
                const float w = exp2f(ms - M);
                L += w * ls;
                const float4 a = __ldcg(reinterpret_cast<const float4*>(p.part_acc + ps * G * D) + v4);
                o.x += w * a.x; o.y += w * a.y; o.z += w * a.z; o.w += w * a.w;
              }
              const float inv = 1.f / L;
              const int fi = v4 * 4;
              if constexpr (sizeof(T) == 2) {
                uint2 w2;
                w2.x = float2_to_bf16x2(o.x * inv, o.y * inv);
                w2.y = float2_to_bf16x2(o.z * inv, o.w * inv);
                *reinterpret_cast<uint2*>(orow + fi) = w2;
              } else {
                *reinterpret_cast<float4*>(orow + fi) = make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
              }
            }
          }
        }
        (void)r;
      }
    }
    __syncwarp();
    produce(st);
    st = (st + 1 == kStages) ? 0 : st + 1;
  }
  // a warp that stopped early still drains the item counter so it resets
  if (aborted) {
    while (!exhausted) {
      if (!next_item()) exhausted = true;
    }
  }
}

}  // namespace decode
}  // namespace cb
