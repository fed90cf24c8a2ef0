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
// One CTA = (prefill row r, KV head g, M tile of 128 query rows).  The 128
// rows pack 128/G tokens x the G query heads that share KV head g, so each
// K/V byte feeds G heads.  Keys stream in tiles of 128 (eight 16-token
// pages), gathered through the block table by TMA: every page is two 2-D
// tensor-map loads (dims 0-63 and 64-127, 128-byte swizzle) straight into the
// canonical UMMA layout.
//
// Warp roles (192 threads):
//   warps 0-3  softmax: thread i owns query row i = TMEM lane i.  Loads Q
//              into shared memory, reads S rows from TMEM, masks, runs the
//              online softmax in base 2 (rescaling O in TMEM only when the
//              running max grows by more than 2^8), writes P (bf16) to shared
//              memory, and finally normalises O and stores it.
//   warp 4     TMA producer: K/V tiles into a 2-stage ring (mbarrier tx).
//   warp 5     MMA issuer: allocates 512 TMEM columns, issues
//              S[b] = Q K^T (S double-buffered, so Q K^T of tile j+1 runs
//              while tile j is in softmax) and O += P V, commits to mbarriers.
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

constexpr int kBM = 128;            // query rows per CTA
constexpr int kBN = 128;            // keys per KV tile
constexpr int kD = 128;             // head dim
constexpr int kPage = 16;           // tokens per block
constexpr int kStages = 2;          // K/V tile ring
constexpr int kThreads = 192;
constexpr uint32_t kTileBytes = kBN * kD * 2;       // 32 KB (one K or V tile)
constexpr uint32_t kHalf = kTileBytes / 2;          // dims 0-63 | dims 64-127
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;

struct SmemLayout {
  static constexpr uint32_t q = 0;
  static constexpr uint32_t k = q + kTileBytes;
  static constexpr uint32_t v = k + kStages * kTileBytes;
  static constexpr uint32_t p = v + kStages * kTileBytes;
  static constexpr uint32_t bars = p + kTileBytes;
  static constexpr uint32_t total = bars + 256;
};

struct Bars {
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[2];
  uint64_t s_empty[2];
  uint64_t p_full;
  uint64_t pv_done;
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

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Bars* B,
                                              uint32_t* error_word) {
  if (mbar_wait(bar, parity)) return true;
  if (atomicExch(&B->abort, 1u) == 0u) set_error(error_word, CB_DEVERR_TIMEOUT);
  return false;
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
  const int tpt = kBM / G;                       // tokens per M tile
  const int r = p.row_begin + blockIdx.z;
  const int g = blockIdx.y;
  const int mt = gridDim.x - 1 - blockIdx.x;     // heavy (late) tiles first
  const int q0 = p.cu_seqlens_q[r];
  const int q_len = p.cu_seqlens_q[r + 1] - q0;
  const int L = p.seq_lens[r];
  const int W = p.max_blocks_per_seq;
  if (q_len < 1 || L < q_len || (L + kPage - 1) / kPage > W) {
    if (threadIdx.x == 0 && blockIdx.x == gridDim.x - 1 && g == 0)
      set_error(p.error_word, CB_DEVERR_SEQ_RANGE);
    return;
  }
  if (mt * tpt >= q_len) return;  // this M tile is past the chunk
  const int start = L - q_len;
  const int last_tok = min(mt * tpt + tpt - 1, q_len - 1);
  const int n_tiles = (start + last_tok) / kBN + 1;
  const int npages = (L + kPage - 1) / kPage;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&B->kv_full[s], 1);
      mbar_init(&B->kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&B->s_full[b], 1);
      mbar_init(&B->s_empty[b], 4);
    }
    mbar_init(&B->p_full, 4);
    mbar_init(&B->pv_done, 1);
    mbar_init(&B->drain, 1);
    B->abort = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tc::tmem_alloc(&B->tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = B->tmem_base;

  const uint32_t sQ = smem_addr(smem + SmemLayout::q);
  const uint32_t sK = smem_addr(smem + SmemLayout::k);
  const uint32_t sV = smem_addr(smem + SmemLayout::v);
  const uint32_t sP = smem_addr(smem + SmemLayout::p);

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    const int oob_row = p.num_blocks * p.num_kv_heads * kPage;  // reads as zeros
    int issued = 0;
    for (int j = 0; j < n_tiles; ++j) {
      const int s = j % kStages;
      if (j >= kStages) {
        bool ok = true;
        if (lane == 0) ok = wait_or_abort(&B->kv_empty[s], ((j / kStages) - 1) & 1, B, p.error_word);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
      if (*reinterpret_cast<volatile uint32_t*>(&B->abort)) break;
      // lanes 0..7 look up the 8 pages of this tile
      int row = oob_row;
      if (lane < kBN / kPage) {
        const int page = j * (kBN / kPage) + lane;
        if (page < npages) {
          const int blk = p.block_tables[(int64_t)r * W + page];
          if (blk >= 0 && blk < p.num_blocks) {
            row = (blk * p.num_kv_heads + g) * kPage;
          } else {
            set_error(p.error_word, CB_DEVERR_BLOCK_RANGE);
          }
        }
      }
      if (lane == 0) mbar_arrive_expect_tx(&B->kv_full[s], 2 * kTileBytes);
      for (int pg = 0; pg < kBN / kPage; ++pg) {
        const int rr = __shfl_sync(0xffffffffu, row, pg);
        if (lane == 0) {
          uint8_t* kd = smem + SmemLayout::k + s * kTileBytes + pg * (kPage * 128);
          uint8_t* vd = smem + SmemLayout::v + s * kTileBytes + pg * (kPage * 128);
          tc::tma_load_2d(kd, &tmap_k, 0, rr, &B->kv_full[s]);
          tc::tma_load_2d(kd + kHalf, &tmap_k, 64, rr, &B->kv_full[s]);
          tc::tma_load_2d(vd, &tmap_v, 0, rr, &B->kv_full[s]);
          tc::tma_load_2d(vd + kHalf, &tmap_v, 64, rr, &B->kv_full[s]);
        }
      }
      __syncwarp();
      issued = j + 1;
    }
    // drain: every issued load lands before the CTA may exit
    if (lane == 0) {
      for (int j = (issued > kStages ? issued - kStages : 0); j < issued; ++j)
        mbar_wait(&B->kv_full[j % kStages], (j / kStages) & 1);
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------------- MMA
    asm volatile("bar.sync 1, 160;" ::: "memory");  // Q is in shared memory
    tc::fence_after_sync();
    if (lane == 0) {
      constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(kBM, kBN, 0);
      constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(kBM, kD, 1);
      bool ok = true;
      for (int j = 0; j <= n_tiles && ok; ++j) {
        if (j < n_tiles) {
          const int s = j % kStages;
          const int b = j & 1;
          ok = wait_or_abort(&B->kv_full[s], (j / kStages) & 1, B, p.error_word);
          if (ok && j >= 2) ok = wait_or_abort(&B->s_empty[b], ((j >> 1) - 1) & 1, B, p.error_word);
          if (!ok) break;
          tc::fence_after_sync();
          const uint32_t d = tmem + (b ? kColS1 : kColS0);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
            tc::mma_f16(d, tc::smem_desc_sw128(sQ + off, 16, 1024),
                        tc::smem_desc_sw128(sK + s * kTileBytes + off, 16, 1024), idesc_qk, kk > 0);
          }
          tc::mma_commit(&B->s_full[b]);
        }
        if (j >= 1) {
          const int jp = j - 1;
          const int sp = jp % kStages;
          ok = wait_or_abort(&B->p_full, jp & 1, B, p.error_word);
          if (!ok) break;
          tc::fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk) {
            const uint32_t aoff = (kk >> 2) * kHalf + (kk & 3) * 32;
            const uint32_t boff = sp * kTileBytes + kk * 2048;
            tc::mma_f16(tmem + kColO, tc::smem_desc_sw128(sP + aoff, 16, 1024),
                        tc::smem_desc_sw128(sV + boff, kHalf, 1024), idesc_pv,
                        (jp > 0 || kk > 0) ? 1u : 0u);
          }
          tc::mma_commit(&B->pv_done);
          tc::mma_commit(&B->kv_empty[sp]);
        }
      }
      // drain: all issued MMAs complete before TMEM is released
      tc::mma_commit(&B->drain);
      mbar_wait(&B->drain, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int row = threadIdx.x;  // 0..127 == TMEM lane
    const int tok = mt * tpt + row / G;
    const int head = g * G + row % G;
    const bool valid = tok < q_len;
    const int pos = start + (valid ? tok : q_len - 1);
    // Q row -> shared memory (128-byte swizzle, two 64-dim halves)
    {
      const uint4* src = reinterpret_cast<const uint4*>(
          p.q + ((int64_t)(q0 + (valid ? tok : q_len - 1)) * p.num_q_heads + head) * kD);
      uint8_t* qs = smem + SmemLayout::q;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        uint4 v = valid ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(qs + (c >> 3) * kHalf + swz(row, c & 7)) = v;
      }
      fence_proxy_async_smem();
      asm volatile("bar.sync 1, 160;" ::: "memory");
    }
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    float m_run = -INFINITY, l_run = 0.f;
    const float sl = p.scale_log2;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int b = j & 1;
      bool w = true;
      if (lane == 0) w = wait_or_abort(&B->s_full[b], (j >> 1) & 1, B, p.error_word);
      w = __shfl_sync(0xffffffffu, w, 0);
      if (!w) { ok = false; break; }
      tc::fence_after_sync();
      float s[kBN];
      const uint32_t sc = trow + (b ? kColS1 : kColS0);
#pragma unroll
      for (int c = 0; c < 4; ++c) tc::tmem_ld32(sc + 32 * c, s + 32 * c);
      tc::tmem_wait_ld();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&B->s_empty[b]);

      const int kbase = j * kBN;
      float mt_max = -INFINITY;
      if (kbase + kBN - 1 > pos) {
#pragma unroll
        for (int i = 0; i < kBN; ++i) {
          s[i] = (kbase + i <= pos) ? s[i] * sl : -INFINITY;
          mt_max = fmaxf(mt_max, s[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < kBN; ++i) {
          s[i] *= sl;
          mt_max = fmaxf(mt_max, s[i]);
        }
      }
      const float m_new = fmaxf(m_run, mt_max);
      const bool resc = (m_new - m_run) > 8.f;  // also true on the first tile
      const float m_use = resc ? m_new : m_run;
      const float alpha = resc ? exp2f(m_run - m_use) : 1.f;
      m_run = m_use;
      float lsum = 0.f;
      uint32_t pk[kBN / 2];
#pragma unroll
      for (int i = 0; i < kBN; i += 2) {
        const float a = exp2f(s[i] - m_use);
        const float c = exp2f(s[i + 1] - m_use);
        lsum += a + c;
        pk[i / 2] = float2_to_bf16x2(a, c);
      }
      l_run = l_run * alpha + lsum;

      // P buffer and O are free once P.V of the previous tile completed
      if (j > 0) {
        if (lane == 0) w = wait_or_abort(&B->pv_done, (j - 1) & 1, B, p.error_word);
        w = __shfl_sync(0xffffffffu, w, 0);
        if (!w) { ok = false; break; }
        tc::fence_after_sync();
        if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float o[32];
            tc::tmem_ld32(trow + kColO + 32 * c, o);
            tc::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= alpha;
            tc::tmem_st32(trow + kColO + 32 * c, o);
          }
          tc::tmem_wait_st();
        }
      }
      // keys at or past seq_len in this tile's valid pages hold stale data;
      // zero those V rows (P is 0 there, but 0 * NaN would not be)
      if (kbase + kBN > L) {
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
      }
      // P row -> shared memory (K-major, 128-byte swizzle)
      uint8_t* ps = smem + SmemLayout::p;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        *reinterpret_cast<uint4*>(ps + (c >> 3) * kHalf + swz(row, c & 7)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      }
      fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&B->p_full);
    }
    // epilogue: O / l -> bf16 rows
    if (ok) {
      bool w = true;
      if (lane == 0) w = wait_or_abort(&B->pv_done, (n_tiles - 1) & 1, B, p.error_word);
      w = __shfl_sync(0xffffffffu, w, 0);
      if (w) {
        tc::fence_after_sync();
        const float inv = 1.f / l_run;
        uint4* dst = reinterpret_cast<uint4*>(p.out + ((int64_t)(q0 + tok) * p.num_q_heads + head) * kD);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float o[32];
          tc::tmem_ld32(trow + kColO + 32 * c, o);
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
  if (warp == 5) tc::tmem_dealloc(tmem, kTmemCols);
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
  const int tpt = kBM / G;
  dim3 grid((a.max_q_len + tpt - 1) / tpt, a.num_kv_heads, a.num_reqs - a.num_decodes);
  prefill_kernel<<<grid, kThreads, smem, stream>>>(mk, mv, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(CB_ERR_CUDA, "prefill kernel launch: %s", cudaGetErrorString(e));
  return CB_OK;
}

}  // namespace cb
