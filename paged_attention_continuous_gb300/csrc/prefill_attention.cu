// Prefill-chunk paged attention on tcgen05 tensor cores (bf16, head_dim 128).
//
// What it computes ("Chunked Prefill", Ultralytics glossary, How chunked
// prefill works): a chunk of q_len query tokens that starts at absolute
// position s = seq_len - q_len attends, under a causal mask over absolute
// positions, to every cached key of its request -- query i sees keys
// 0..s+i, i.e. all earlier chunks plus its own prefix.  Prefill does many
// operations per byte ("Chunked Prefill", Prefill, decode and generation
// stalls), and both Q.K^T and P.V are dense contractions, so they run on the
// tensor cores.
//
// One CTA = (prefill row r, KV head g, a PAIR of 128-row query tiles).  A
// query tile packs 128/G tokens x the G query heads that share KV head g, so
// each K/V byte feeds G heads, and both tiles of the pair share every K/V
// tile staged in shared memory.  Keys stream in tiles of 128 (eight 16-token
// pages), gathered through the block table by TMA: each page is two 2-D
// tensor-map loads (dims 0-63 and 64-127, 128-byte swizzle) that land in the
// canonical UMMA layout; one warp instruction issues a tile's 32 loads.
//
// Tensor memory (512 columns): S0 | S1 | O0 | O1, 128 fp32 columns each.  The
// softmax of tile t overwrites the first 64 columns of S_t with P_t as bf16
// pairs, and P_t.V reads its A operand straight from tensor memory, so P never
// touches shared memory.
//
// Warp roles (320 threads):
//   warps 0-3 / 4-7  softmax for query tile 0 / 1: thread i owns row i (TMEM
//              lane i).  Loads its Q row into shared memory; per KV tile reads
//              its S row, masks, runs the online softmax in base 2 (O_t is
//              rescaled in tensor memory only when the running max grows by
//              more than 2^8), writes P_t back to tensor memory; at the end
//              normalises O_t and stores it.
//   warp 8     TMA producer: K/V tiles into a 2-stage ring.
//   warp 9     MMA issuer: allocates tensor memory and issues, per KV tile j,
//              P0.V(j-1), Q0.K(j), P1.V(j-1), Q1.K(j) -- so each softmax
//              warpgroup works while the tensor core serves the other.
// Every wait is bounded (CB_DEVERR_TIMEOUT) and nothing spins forever.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "cb_error.h"
#include "device_utils.cuh"
#include "prefill_dispatch.h"
#include "tcgen05.cuh"

namespace cb {
namespace prefill {

constexpr int kBM = 128;            // query rows per tile
constexpr int kBN = 128;            // keys per KV tile
constexpr int kD = 128;             // head dim
constexpr int kPage = 16;           // tokens per block
constexpr int kStages = 2;          // K/V tile ring
constexpr int kThreads = 320;
constexpr uint32_t kTileBytes = kBN * kD * 2;       // 32 KB (one Q, K or V tile)
constexpr uint32_t kHalf = kTileBytes / 2;          // dims 0-63 | dims 64-127
constexpr uint32_t kTmemCols = 512;
// tensor-memory column of S_t and O_t for query tile t
__host__ __device__ constexpr uint32_t col_s(int t) { return t ? 128u : 0u; }
__host__ __device__ constexpr uint32_t col_o(int t) { return t ? 384u : 256u; }

struct SmemLayout {
  static constexpr uint32_t q = 0;                              // Q0 | Q1
  static constexpr uint32_t k = q + 2 * kTileBytes;
  static constexpr uint32_t v = k + kStages * kTileBytes;
  static constexpr uint32_t bars = v + kStages * kTileBytes;
  static constexpr uint32_t total = bars + 256;
};

struct Bars {
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[2];     // per query tile: S_t of the current KV tile ready
  uint64_t p_full[2];     // per query tile: P_t written (and O_t rescaled)
  uint64_t o_done[2];     // per query tile: last P_t.V complete
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort;
};

struct Params {
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  const int32_t* cu_seqlens_q;
  const int32_t* seq_lens;
  const int32_t* block_tables;
  int32_t row_begin;          // first prefill row
  int32_t num_blocks, max_blocks_per_seq, num_q_heads, num_kv_heads, group;
  float scale_log2;
  uint32_t* error_word;
};

__device__ __forceinline__ void abort_cta(Bars* B, uint32_t* error_word) {
  if (atomicExch(&B->abort, 1u) == 0u) set_error(error_word, CB_DEVERR_TIMEOUT);
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Bars* B,
                                              uint32_t* error_word) {
  if (mbar_wait(bar, parity)) return true;
  abort_cta(B, error_word);
  return false;
}

// 2^x with the hardware approximation (ex2.approx.ftz.f32): relative error
// about 2^-22, 2^-inf = 0; used for softmax weights that are rounded to bf16.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t chunk) {
  // byte offset of 16-byte chunk `chunk` (0..7) of 128-byte row `row` under
  // the 128-byte swizzle (chunk index XOR row mod 8)
  return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Bars* B = reinterpret_cast<Bars*>(smem + SmemLayout::bars);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int G = p.group;
  const int tpt = kBM / G;                       // tokens per query tile
  const int r = p.row_begin + blockIdx.z;
  const int g = blockIdx.y;
  const int mp = gridDim.x - 1 - blockIdx.x;     // tile pair; heavy (late) pairs first
  const int q0 = p.cu_seqlens_q[r];
  const int q_len = p.cu_seqlens_q[r + 1] - q0;
  const int L = p.seq_lens[r];
  const int W = p.max_blocks_per_seq;
  if (q_len < 1 || L < q_len || (L + kPage - 1) / kPage > W) {
    if (threadIdx.x == 0 && blockIdx.x == gridDim.x - 1 && g == 0)
      set_error(p.error_word, CB_DEVERR_SEQ_RANGE);
    return;
  }
  const int tok0 = mp * 2 * tpt;                 // first token of query tile 0
  if (tok0 >= q_len) return;                     // this pair is past the chunk
  const bool has_t1 = tok0 + tpt < q_len;        // query tile 1 holds tokens
  const int start = L - q_len;
  const int last_tok = min(tok0 + 2 * tpt - 1, q_len - 1);
  const int n_tiles = (start + last_tok) / kBN + 1;
  const int npages = (L + kPage - 1) / kPage;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&B->kv_full[s], 1);
      mbar_init(&B->kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&B->s_full[t], 1);
      mbar_init(&B->p_full[t], 4);
      mbar_init(&B->o_done[t], 1);
    }
    mbar_init(&B->drain, 1);
    B->abort = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tc::tmem_alloc(&B->tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = B->tmem_base;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    // Lane l moves one 16-row x 64-dim box: page l/4 of the tile, part l%4
    // (K dims 0-63, K dims 64-127, V dims 0-63, V dims 64-127), so one warp
    // instruction issues all 32 loads of a tile.  Block ids of the next tile
    // are fetched while waiting for a free stage.
    const int oob_row = p.num_blocks * p.num_kv_heads * kPage;  // reads as zeros
    const int part = lane & 3;
    const int pg = lane >> 2;
    const CUtensorMap* tmap = part < 2 ? &tmap_k : &tmap_v;
    const uint32_t dst_off = (part < 2 ? SmemLayout::k : SmemLayout::v) + (part & 1) * kHalf +
                             pg * (kPage * 128);
    const int x = (part & 1) * 64;
    auto fetch_blk = [&](int j) -> int {
      const int page = j * (kBN / kPage) + lane;
      return (lane < kBN / kPage && j < n_tiles && page < npages)
                 ? __ldg(p.block_tables + (int64_t)r * W + page)
                 : -1;
    };
    auto to_row = [&](int blk, int j) -> int {
      const int page = j * (kBN / kPage) + lane;
      if (lane >= kBN / kPage || page >= npages) return oob_row;
      if (blk < 0 || blk >= p.num_blocks) {
        set_error(p.error_word, CB_DEVERR_BLOCK_RANGE);
        return oob_row;
      }
      return (blk * p.num_kv_heads + g) * kPage;
    };
    int issued = 0;
    int blk_next = fetch_blk(0);
    for (int j = 0; j < n_tiles; ++j) {
      const int s = j % kStages;
      const int blk_cur = blk_next;
      blk_next = fetch_blk(j + 1);  // in flight while we wait
      if (j >= kStages) {
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&B->kv_empty[s], ((j / kStages) - 1) & 1));
        if (!ok) { abort_cta(B, p.error_word); break; }
      }
      if (*reinterpret_cast<volatile uint32_t*>(&B->abort)) break;
      const int rr = __shfl_sync(0xffffffffu, to_row(blk_cur, j), pg);
      if (lane == 0) mbar_arrive_expect_tx(&B->kv_full[s], 2 * kTileBytes);
      __syncwarp();
      tc::tma_load_2d(smem + dst_off + s * kTileBytes, tmap, x, rr, &B->kv_full[s]);
      issued = j + 1;
    }
    // drain: every issued load lands before the CTA may exit
    if (lane == 0) {
      for (int j = (issued > kStages ? issued - kStages : 0); j < issued; ++j)
        mbar_wait(&B->kv_full[j % kStages], (j / kStages) & 1);
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------------- MMA
    asm volatile("bar.sync 1, 288;" ::: "memory");  // Q0, Q1 are in shared memory
    tc::fence_after_sync();
    if (lane == 0) {
      constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(kBM, kBN, 0);
      constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(kBM, kD, 1);
      const uint32_t sQ = smem_addr(smem + SmemLayout::q);
      const uint32_t sK = smem_addr(smem + SmemLayout::k);
      const uint32_t sV = smem_addr(smem + SmemLayout::v);
      const int nt = has_t1 ? 2 : 1;
      bool ok = true;
      for (int j = 0; j <= n_tiles && ok; ++j) {
        const int s = j % kStages;
        if (j < n_tiles) ok = wait_or_abort(&B->kv_full[s], (j / kStages) & 1, B, p.error_word);
        for (int t = 0; t < nt && ok; ++t) {
          if (j >= 1) {
            // O_t += P_t(j-1) . V(j-1); P_t lives in the first 64 columns of S_t
            const int jp = j - 1;
            const int sp = jp % kStages;
            ok = wait_or_abort(&B->p_full[t], jp & 1, B, p.error_word);
            if (!ok) break;
            tc::fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
              tc::mma_f16_ts(tmem + col_o(t), tmem + col_s(t) + kk * 8,
                             tc::smem_desc_sw128(sV + sp * kTileBytes + kk * 2048, kHalf, 1024),
                             idesc_pv, (jp > 0 || kk > 0) ? 1u : 0u);
            if (t == nt - 1) tc::mma_commit(&B->kv_empty[sp]);
            if (j == n_tiles) tc::mma_commit(&B->o_done[t]);
          }
          if (j < n_tiles) {
            // S_t = Q_t . K(j)^T (after P_t.V(j-1) in issue order)
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
              const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
              tc::mma_f16(tmem + col_s(t),
                          tc::smem_desc_sw128(sQ + t * kTileBytes + off, 16, 1024),
                          tc::smem_desc_sw128(sK + s * kTileBytes + off, 16, 1024), idesc_qk, kk > 0);
            }
            tc::mma_commit(&B->s_full[t]);
          }
        }
      }
      // drain: all issued MMAs complete before tensor memory is released
      tc::mma_commit(&B->drain);
      mbar_wait(&B->drain, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;                     // query tile of this warpgroup
    const int row = threadIdx.x & 127;           // == TMEM lane
    const int tok = tok0 + t * tpt + row / G;
    const int head = g * G + row % G;
    const bool valid = tok < q_len;
    const int pos = start + (valid ? tok : q_len - 1);
    // Q row -> shared memory (128-byte swizzle, two 64-dim halves)
    {
      const uint4* src = reinterpret_cast<const uint4*>(
          p.q + ((int64_t)(q0 + (valid ? tok : q_len - 1)) * p.num_q_heads + head) * kD);
      uint8_t* qs = smem + SmemLayout::q + t * kTileBytes;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        uint4 v = valid ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(qs + (c >> 3) * kHalf + swz(row, c & 7)) = v;
      }
      fence_proxy_async_smem();
      asm volatile("bar.sync 1, 288;" ::: "memory");
    }
    const bool active = t == 0 || has_t1;
    const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t colS = col_s(t), colO = col_o(t);
    float m_run = -INFINITY, l_run = 0.f;
    const float sl = p.scale_log2;
    bool ok = active;
    for (int j = 0; j < n_tiles && ok; ++j) {
      bool w = __all_sync(0xffffffffu, mbar_wait(&B->s_full[t], j & 1));
      if (!w) { abort_cta(B, p.error_word); ok = false; break; }
      tc::fence_after_sync();
      const int kbase = j * kBN;
      // causal mask limit: key kbase+i is visible iff i <= lim
      const int lim = pos - kbase;
      const bool masked = lim < kBN - 1;
      // pass 1: row max of the raw scores (64 columns at a time, 8 chains)
      float mx[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mx[u] = -INFINITY;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float s[64];
        tc::tmem_ld32(trow + colS + 64 * h, s);
        tc::tmem_ld32(trow + colS + 64 * h + 32, s + 32);
        tc::tmem_wait_ld();
        if (masked) {
#pragma unroll
          for (int i = 0; i < 64; ++i) s[i] = (64 * h + i <= lim) ? s[i] : -INFINITY;
        }
#pragma unroll
        for (int i = 0; i < 64; i += 8)
#pragma unroll
          for (int u = 0; u < 8; ++u) mx[u] = fmaxf(mx[u], s[i + u]);
      }
      const float mt_max =
          fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sl;
      const float m_new = fmaxf(m_run, mt_max);
      const bool resc = (m_new - m_run) > 8.f;  // also true on the first tile
      const float m_use = resc ? m_new : m_run;
      const float alpha = resc ? fast_exp2(m_run - m_use) : 1.f;
      m_run = m_use;
      // pass 2: p = 2^(s*scale - m) (one FFMA + one ex2 per score), row sum in
      // 8 chains, P as bf16 pairs written over S columns already read
      const float nm = -m_use;
      float ls[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) ls[u] = 0.f;
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        float s[32];
        tc::tmem_ld32(trow + colS + 32 * h, s);
        tc::tmem_wait_ld();
        if (masked) {
#pragma unroll
          for (int i = 0; i < 32; ++i) s[i] = (32 * h + i <= lim) ? s[i] : -INFINITY;
        }
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float a = fast_exp2(fmaf(s[i], sl, nm));
          const float c = fast_exp2(fmaf(s[i + 1], sl, nm));
          ls[(i >> 1) & 7] += a + c;
          pk[i / 2] = float2_to_bf16x2(a, c);
        }
        tc::tmem_st16(trow + colS + 16 * h, pk);
      }
      const float lsum = ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
      l_run = l_run * alpha + lsum;

      // S_t(j) ready implies P_t.V(j-1) completed (same issuing thread, in
      // order), so O_t is stable here and may be rescaled.
      if (j >= 1 && __any_sync(0xffffffffu, resc)) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float o[32];
          tc::tmem_ld32(trow + colO + 32 * c, o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= alpha;
          tc::tmem_st32(trow + colO + 32 * c, o);
        }
      }
      // keys at or past seq_len in this tile's valid pages hold stale data;
      // zero those V rows (P is 0 there, but 0 * NaN would not be).  Done by
      // tile 0's warpgroup before P_0.V(j), the first reader of V(j).
      if (t == 0 && kbase + kBN > L) {
        const int z0 = L - kbase;
        const int z1 = min(kBN, npages * kPage - kbase);
        const int kr = z0 + row;
        if (kr < z1) {
          uint8_t* vrow = smem + SmemLayout::v + (j % kStages) * kTileBytes + kr * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            *reinterpret_cast<uint4*>(vrow + c * 16) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(vrow + kHalf + c * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&B->p_full[t]);
    }
    // epilogue: O_t / l -> bf16 rows
    if (ok) {
      const bool w = __all_sync(0xffffffffu, mbar_wait(&B->o_done[t], 0));
      if (!w) abort_cta(B, p.error_word);
      if (w) {
        tc::fence_after_sync();
        const float inv = 1.f / l_run;
        uint4* dst = reinterpret_cast<uint4*>(p.out + ((int64_t)(q0 + tok) * p.num_q_heads + head) * kD);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float o[32];
          tc::tmem_ld32(trow + colO + 32 * c, o);
          tc::tmem_wait_ld();
          if (valid) {
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
              uint4 v;
              v.x = float2_to_bf16x2(o[e] * inv, o[e + 1] * inv);
              v.y = float2_to_bf16x2(o[e + 2] * inv, o[e + 3] * inv);
              v.z = float2_to_bf16x2(o[e + 4] * inv, o[e + 5] * inv);
              v.w = float2_to_bf16x2(o[e + 6] * inv, o[e + 7] * inv);
              dst[(32 * c + e) / 8] = v;
            }
          }
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 9) tc::tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------- host
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// 2-D view of a cache [num_blocks * Hkv * 16 rows][128 dims] bf16; box 16
// rows x 64 dims (128 bytes) with the 128-byte swizzle.
cb_status make_cache_map(CUtensorMap* m, const void* base, int64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(CB_ERR_CUDA, "cuTensorMapEncodeTiled entry point not available");
  cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kPage};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(CB_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return CB_OK;
}

}  // namespace prefill

bool prefill_supported(int group) {
  return group == 1 || group == 2 || group == 4 || group == 8 || group == 16;
}

size_t prefill_workspace_bytes(int64_t, int64_t, int64_t) { return 0; }

cb_status launch_prefill_bf16(const cb_attention_args& a, uint32_t* error_word, uint8_t*,
                              cudaStream_t stream) {
  using namespace prefill;
  if (a.head_dim != kD || a.block_size != kPage || a.dtype != CB_DTYPE_BF16) return CB_ERR_UNSUPPORTED;
  const int G = a.num_q_heads / a.num_kv_heads;
  if (!prefill_supported(G)) return CB_ERR_UNSUPPORTED;
  const int64_t rows = (int64_t)a.num_blocks * a.num_kv_heads * kPage;
  if (rows >= (int64_t)1 << 31) return CB_ERR_UNSUPPORTED;
  CUtensorMap mk, mv;
  cb_status st = make_cache_map(&mk, a.k_cache, rows);
  if (st != CB_OK) return st;
  st = make_cache_map(&mv, a.v_cache, rows);
  if (st != CB_OK) return st;
  const size_t smem = SmemLayout::total + 1024;
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [&] {
    attr = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem);
  });
  if (attr != cudaSuccess) return fail(CB_ERR_CUDA, "prefill smem attribute: %s", cudaGetErrorString(attr));
  Params p{};
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.cu_seqlens_q = a.cu_seqlens_q;
  p.seq_lens = a.seq_lens;
  p.block_tables = a.block_tables;
  p.row_begin = a.num_decodes;
  p.num_blocks = a.num_blocks;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = G;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.error_word = error_word;
  const int tpp = 2 * (kBM / G);  // tokens per CTA (a pair of query tiles)
  dim3 grid((a.max_q_len + tpp - 1) / tpp, a.num_kv_heads, a.num_reqs - a.num_decodes);
  prefill_kernel<<<grid, kThreads, smem, stream>>>(mk, mv, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(CB_ERR_CUDA, "prefill kernel launch: %s", cudaGetErrorString(e));
  return CB_OK;
}

}  // namespace cb
