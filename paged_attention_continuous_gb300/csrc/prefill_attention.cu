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
// tile staged in shared memory.  The grid is flat over the pairs that exist,
// times the KV heads (blockIdx.x = pair * Hkv + head; pairs counted row by
// row, a row's latest -- heaviest -- pair first, so all heads of the
// heaviest work launch first): warp 0 finds its CTA's row by a scan of the
// rows' pair counts, so rows shorter than the longest chunk launch no idle
// CTAs.  Keys stream in tiles of 128 (eight 16-token
// pages), gathered through the block table by the TMA engine: one 2-D
// tensor-map box of 16 rows x 64 dims per page half lands directly in the
// 128-byte-swizzled canonical UMMA layout.
//
// Tensor memory (512 columns): S0 | S1 | O0 | O1, 128 fp32 columns each.  The
// softmax of tile t overwrites the first 64 columns of S_t with P_t as bf16
// pairs, and P_t.V reads its A operand straight from tensor memory, so P never
// touches shared memory.
//
// Warp roles (384 threads):
//   warps 0-3 / 4-7  softmax for query tile 0 / 1: thread i owns row i (TMEM
//              lane i).  Loads its Q row into shared memory; per KV tile
//              reads its S row (a max pass, then an exp pass that streams P
//              back into tensor memory), runs the online softmax in base 2
//              (O_t is rescaled in tensor memory only when the running max
//              grows by more than 2^8); at the end normalises O_t and stores
//              it.
//   warp 8     K producer: K tiles into a 3-stage ring (TMA; pages past the
//              sequence read as zeros); a stage is released after the last
//              Q.K^T that reads it.
//   warp 9     V producer: V tiles into a 2-stage ring, released after the
//              last P.V.  (Slots past seq_len inside the last page are real
//              pool memory: their K scores are masked by the softmax, their
//              V rows are zeroed in shared memory before the P.V that reads
//              them, as P = 0 there does not cancel a non-finite value.)
//   warps 10-11  MMA issuers, one per query tile t (warp 10 also allocates
//              tensor memory): per KV tile j, P_t.V(j-1) then Q_t.K(j), each
//              as soon as its own inputs are ready -- each softmax warpgroup
//              works while the tensor core serves the other.
// Every wait is bounded (CB_DEVERR_TIMEOUT) and nothing spins forever.
//
// Sliding-window layers ("Continuous batching architecture", Memory
// management): with window W > 0 query position p attends keys p-W+1..p.
// A CTA then streams only the KV tiles from the one holding key
// (first query of its pair) - W + 1; pages before that key read as zeros
// (they may have been recycled), and keys before each row's window are
// masked in the softmax like the causal upper triangle.  A row whose keys
// in the tiles seen so far are all masked keeps a running max of -inf and
// exponentiates against 0, so its weights stay exactly 0.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "cb_error.h"
#include "device_utils.cuh"
#include "launch_common.h"
#include "prefill_dispatch.h"
#include "tcgen05.cuh"
#include "tensor_map.h"

namespace cb {
namespace prefill {

constexpr int kBM = 128;            // query rows per tile
constexpr int kBN = 128;            // keys per KV tile
constexpr int kD = 128;             // head dim
constexpr int kPage = 16;           // tokens per block
constexpr int kStagesK = 3;         // K tile ring (K is needed first: deeper)
constexpr int kStagesV = 2;         // V tile ring
constexpr int kProducerWarps = 2;
constexpr int kMmaWarp = 8 + kProducerWarps;   // MMA issuers: warps kMmaWarp + t
constexpr int kThreads = (kMmaWarp + 2) * 32;   // softmax x8, producer x2, MMA x2
constexpr uint32_t kTileBytes = kBN * kD * 2;       // 32 KB (one Q, K or V tile)
constexpr uint32_t kHalf = kTileBytes / 2;          // dims 0-63 | dims 64-127
constexpr uint32_t kTmemCols = 512;
// tensor-memory column of S_t and O_t for query tile t
__host__ __device__ constexpr uint32_t col_s(int t) { return t ? 128u : 0u; }
__host__ __device__ constexpr uint32_t col_o(int t) { return t ? 384u : 256u; }

struct SmemLayout {
  static constexpr uint32_t q = 0;                              // Q0 | Q1
  static constexpr uint32_t k = q + 2 * kTileBytes;
  static constexpr uint32_t v = k + kStagesK * kTileBytes;
  static constexpr uint32_t bars = v + kStagesV * kTileBytes;
  static constexpr uint32_t total = bars + 256;
};

struct Bars {
  uint64_t k_full[kStagesK];   // K tile landed
  uint64_t v_full[kStagesV];   // V tile landed
  uint64_t k_empty[kStagesK];  // last Q.K^T of the K tile done
  uint64_t v_empty[kStagesV];  // last P.V of the V tile done
  uint64_t s_full[2];         // per query tile: S_t of the current KV tile ready
  uint64_t p_full[2];         // per query tile: P_t written (and O_t rescaled)
  uint64_t o_done[2];         // per query tile: last P_t.V complete
  uint64_t drain[2];          // per MMA issuer: all its MMAs complete
  uint32_t tmem_base;
  uint32_t abort;
};

struct Params {
  CUtensorMap tmap_k;  // [num_blocks * Hkv * 16 rows][128 dims] bf16, box 16 x 64, 128-B swizzle
  CUtensorMap tmap_v;
  const void* k_cache;
  const void* v_cache;
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  const int32_t* cu_seqlens_q;
  const int32_t* seq_lens;
  const int32_t* block_tables;
  int32_t row_begin;          // first prefill row
  int32_t num_rows;           // prefill rows
  int32_t num_tokens;         // rows of q / out
  int32_t num_blocks, max_blocks_per_seq, num_q_heads, num_kv_heads, group;
  float scale_log2;
  int32_t window;             // sliding window (0: full attention)
  uint32_t* error_word;
  uint64_t wait_ns;           // limit of every bounded wait
  int32_t withhold_tile;      // test hook: CTA 0 never copies its K tile with
                              // this ring index (-1: none)
};

__device__ __forceinline__ void abort_cta(Bars* B, uint32_t* error_word) {
  if (atomicExch(&B->abort, 1u) == 0u) set_error(error_word, CB_DEVERR_TIMEOUT);
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Bars* B,
                                              uint32_t* error_word, uint64_t limit_ns) {
  if (mbar_wait(bar, parity, limit_ns)) return true;
  abort_cta(B, error_word);
  return false;
}

// 2^x with the hardware approximation (ex2.approx.ftz.f32): relative error
// about 2^-22, 2^-inf = 0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^x for a pair of bf16 values (low half first) with one hardware op
// (ex2.approx.ftz.bf16x2); 2^-inf = 0.
__device__ __forceinline__ uint32_t fast_exp2_bf16x2(uint32_t x) {
  uint32_t y;
  asm("ex2.approx.ftz.bf16x2 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t chunk) {
  // byte offset of 16-byte chunk `chunk` (0..7) of 128-byte row `row` under
  // the 128-byte swizzle (chunk index XOR row mod 8)
  return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

// When this grid was launched to overlap the kernel before it (the decode
// kernel of the same call), one thread of CTA 0 waits for that kernel before
// exiting, on every path, so this grid completes only after it.
__device__ __forceinline__ void order_after_previous_grid() {
  if (blockIdx.x == 0 && threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Bars* B = reinterpret_cast<Bars*>(smem + SmemLayout::bars);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // the decode rows of the same call, when launched after this grid with
  // programmatic serialization, may start at once on the SMs it leaves idle
  // (they touch nothing this grid touches)
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the producers' tensor maps travel to the TMA unit while the rows are scanned
  if ((warp == 8 || warp == 9) && lane == 0) tc::prefetch_tensormap(warp == 8 ? &p.tmap_k : &p.tmap_v);

  const int G = p.group;
  const int tpt = kBM / G;                       // tokens per query tile
  const int g = (int)(blockIdx.x % (unsigned)p.num_kv_heads);
  // ---- which (row, pair) this CTA serves: warp 0 scans the rows' pair
  // counts (ceil(q_len / pair tokens)); CTA (0, 0) also checks that no row
  // has a negative query length or a zero one with context, and that the
  // grid covers every pair
  __shared__ int s_row, s_pair;
  if (warp == 0) {
    const int tpp = 2 * tpt;
    const int x = (int)(blockIdx.x / (unsigned)p.num_kv_heads);
    const int num_pairs = (int)(gridDim.x / (unsigned)p.num_kv_heads);
    int run = 0, row = -1, pair = 0;
    bool bad = false;
    for (int b = 0; b < p.num_rows; b += 32) {
      const int i = b + lane;
      int cnt = 0;
      if (i < p.num_rows) {
        const int rr = p.row_begin + i;
        const int ql = p.cu_seqlens_q[rr + 1] - p.cu_seqlens_q[rr];
        if (ql < 0 || (ql == 0 && p.seq_lens[rr] != 0)) bad = true;
        cnt = ql > 0 ? (ql + tpp - 1) / tpp : 0;
      }
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const bool mine = cnt > 0 && x >= run + incl - cnt && x < run + incl;
      const uint32_t hit = __ballot_sync(0xffffffffu, mine);
      if (hit) {
        const int src = __ffs(hit) - 1;
        row = __shfl_sync(0xffffffffu, i, src);
        const int first = __shfl_sync(0xffffffffu, run + incl - cnt, src);
        const int n = __shfl_sync(0xffffffffu, cnt, src);
        pair = n - 1 - (x - first);              // the row's heaviest pair first
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    bad = __any_sync(0xffffffffu, bad) || run > num_pairs;
    if (lane == 0) {
      if (bad && blockIdx.x == 0) set_error(p.error_word, CB_DEVERR_SEQ_RANGE);
      s_row = row;
      s_pair = pair;
    }
  }
  __syncthreads();
  if (s_row < 0) {                               // past the last pair
    order_after_previous_grid();
    return;
  }
  const int r = p.row_begin + s_row;
  const int mp = s_pair;
  const int q0 = p.cu_seqlens_q[r];
  const int q_len = p.cu_seqlens_q[r + 1] - q0;
  const int L = p.seq_lens[r];
  const int W = p.max_blocks_per_seq;
  if (q0 < 0 || q0 + q_len > p.num_tokens || L < q_len || (L + kPage - 1) / kPage > W) {
    if (threadIdx.x == 0 && mp == 0 && g == 0) set_error(p.error_word, CB_DEVERR_SEQ_RANGE);
    order_after_previous_grid();
    return;
  }
  const int tok0 = mp * 2 * tpt;                 // first token of query tile 0
  if (tok0 >= q_len) {                           // this pair is past the chunk
    order_after_previous_grid();
    return;
  }
  const bool has_t1 = tok0 + tpt < q_len;        // query tile 1 holds tokens
  const int start = L - q_len;
  const int last_tok = min(tok0 + 2 * tpt - 1, q_len - 1);
  const int n_tiles = (start + last_tok) / kBN + 1;
  const int npages = (L + kPage - 1) / kPage;
  // with a window, the pair's first query reads keys from key_lo on: KV
  // tiles j_lo .. n_tiles - 1 (nt of them; ring positions count from j_lo)
  const int key_lo = p.window > 0 ? max(0, start + tok0 - p.window + 1) : 0;
  const int j_lo = key_lo / kBN;
  const int lo_pg = key_lo / kPage;
  const int nt = n_tiles - j_lo;
  // Lane pg (0..7) of a producer warp looks up the block of page pg of a KV
  // tile; the first tile's ids are requested here, so the lookups overlap
  // the barrier and tensor-memory set-up below.
  auto page_in = [&](int j) {
    const int page = j * (kBN / kPage) + lane;
    return lane < kBN / kPage && j < n_tiles && page < npages && page >= lo_pg;
  };
  auto page_blk = [&](int j) {
    return __ldg(p.block_tables + (int64_t)r * W + j * (kBN / kPage) + lane);
  };
  bool in0 = false;
  int blk0 = 0;
  if (warp == 8 || warp == 9) {
    in0 = page_in(j_lo);
    if (in0) blk0 = page_blk(j_lo);
  }

  if (threadIdx.x == 0) {
    // a stage is free once every active MMA issuer (one per query tile)
    // has committed its last read of it
    const uint32_t issuers = has_t1 ? 2u : 1u;
    for (int s = 0; s < kStagesK; ++s) {
      mbar_init(&B->k_full[s], 1);
      mbar_init(&B->k_empty[s], issuers);
    }
    for (int s = 0; s < kStagesV; ++s) {
      mbar_init(&B->v_full[s], 1);
      mbar_init(&B->v_empty[s], issuers);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&B->s_full[t], 1);
      mbar_init(&B->p_full[t], 4);
      mbar_init(&B->o_done[t], 1);
    }
    mbar_init(&B->drain[0], 1);
    mbar_init(&B->drain[1], 1);
    B->abort = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(&B->tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = B->tmem_base;

  if (warp >= 8 && warp < kMmaWarp) {
    // ------------------------------------------------------------ producers
    // Warp 8 streams K tiles, warp 9 V tiles.  Lane pg (0..7) holds the
    // block of page pg of a tile (the next tile's ids are requested before
    // the current tile's copies are issued, and read only afterwards); lane
    // 0 issues the two boxes of every page.  A page outside the sequence or
    // the table uses a row past the end of the tensor map, which the TMA
    // engine reads as zeros.
    const int hv = warp - 8;  // 0: K, 1: V
    const CUtensorMap* tmap = hv ? &p.tmap_v : &p.tmap_k;
    const int nst = hv ? kStagesV : kStagesK;
    const uint32_t ring = hv ? SmemLayout::v : SmemLayout::k;
    const int oob_row = p.num_blocks * p.num_kv_heads * kPage;
    // tensor-map row of a looked-up page
    auto page_row = [&](bool in, int blk) -> int {
      int row = oob_row;
      if (in) {
        if (blk >= 0 && blk < p.num_blocks)
          row = (blk * p.num_kv_heads + g) * kPage;
        else if (hv == 0)
          set_error(p.error_word, CB_DEVERR_BLOCK_RANGE);
      }
      return row;
    };
    bool in_next = in0;
    int blk_next = blk0;
    int issued = 0;
    for (int jj = 0; jj < nt; ++jj) {
      const int row = page_row(in_next, blk_next);
      in_next = page_in(j_lo + jj + 1);    // in flight while this tile is issued
      if (in_next) blk_next = page_blk(j_lo + jj + 1);
      const int s = jj % nst;
      uint64_t* full = hv ? &B->v_full[s] : &B->k_full[s];
      if (jj >= nst) {
        uint64_t* empty = hv ? &B->v_empty[s] : &B->k_empty[s];
        const bool ok = __all_sync(0xffffffffu, mbar_wait(empty, ((jj / nst) - 1) & 1, p.wait_ns));
        if (!ok) { abort_cta(B, p.error_word); break; }
      }
      if (*reinterpret_cast<volatile uint32_t*>(&B->abort)) break;
      if (lane == 0) mbar_arrive_expect_tx(full, kTileBytes);
      // test hook: the withheld tile is announced but never copied, so the
      // bounded waits on it run out
      const bool withhold = hv == 0 && blockIdx.x == 0 && jj == p.withhold_tile;
#pragma unroll
      for (int pg = 0; pg < kBN / kPage; ++pg) {
        const int rr = __shfl_sync(0xffffffffu, row, pg);
        if (lane == 0 && !withhold) {
          uint8_t* d = smem + ring + s * kTileBytes + pg * (kPage * 128);
          tc::tma_load_2d(d, tmap, 0, rr, full);
          tc::tma_load_2d(d + kHalf, tmap, 64, rr, full);
        }
      }
      __syncwarp();
      issued = jj + 1;
    }
    // drain: every issued copy lands before the CTA may exit
    for (int j = (issued > nst ? issued - nst : 0); j < issued; ++j)
      mbar_wait(hv ? &B->v_full[j % nst] : &B->k_full[j % nst], (j / nst) & 1, p.wait_ns);
  } else if (warp >= kMmaWarp) {
    // ------------------------------------------------------------------ MMA
    // Warp kMmaWarp + t issues the MMAs of query tile t: per KV tile j,
    // P_t.V(j-1) (after the softmax wrote P_t(j-1) and V(j-1) landed), then
    // Q_t.K(j) (after K(j) landed).  S_t is free for Q_t.K(j) because
    // P_t.V(j-1) was issued before it.  With one issuer per tile, neither
    // tile's chain waits behind the other's issue.
    asm volatile("bar.sync 1, 320;" ::: "memory");  // Q0, Q1 are in shared memory
    tc::fence_after_sync();
    const int t = warp - kMmaWarp;
    if (lane == 0 && (t == 0 || has_t1)) {
      constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(kBM, kBN, 0);
      constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(kBM, kD, 1);
      // Shared-memory descriptors of the tiles' first k-step; a k-step's
      // descriptor is the base plus its byte offset >> 4 (the start-address
      // field is the low 14 bits and the tiles lie below 256 KB); stage s of
      // a ring adds s * kTileBytes >> 4.
      const uint64_t aq = tc::smem_desc_sw128(smem_addr(smem + SmemLayout::q) + t * kTileBytes, 16, 1024);
      const uint64_t dk0 = tc::smem_desc_sw128(smem_addr(smem + SmemLayout::k), 16, 1024);
      const uint64_t dv0 = tc::smem_desc_sw128(smem_addr(smem + SmemLayout::v), kHalf, 1024);
      constexpr uint32_t kTileDesc = kTileBytes >> 4;
      bool ok = true;
      for (int jj = 0; jj <= nt && ok; ++jj) {
        if (jj >= 1) {
          const int jr = jj - 1;            // ring position of the previous tile
          const int jp = j_lo + jr;         // its KV tile
          const int sp = jr % kStagesV;
          ok = wait_or_abort(&B->p_full[t], jr & 1, B, p.error_word, p.wait_ns) &&
               wait_or_abort(&B->v_full[sp], (jr / kStagesV) & 1, B, p.error_word, p.wait_ns);
          if (!ok) break;
          if ((L & (kPage - 1)) != 0 && jp == (L - 1) / kBN) {
            // rows L .. end of the last page hold pool slots past the
            // sequence: zero them (both 64-dim halves) before P.V reads them
            // (both issuers write the same zeros)
            uint8_t* vt = smem + SmemLayout::v + sp * kTileBytes;
            const int r0 = L - jp * kBN, r1 = ((L + kPage - 1) / kPage) * kPage - jp * kBN;
            for (int rw = r0; rw < r1; ++rw)
              for (int c = 0; c < 8; ++c) {
                *reinterpret_cast<uint4*>(vt + rw * 128 + c * 16) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(vt + kHalf + rw * 128 + c * 16) = make_uint4(0, 0, 0, 0);
              }
          }
          // zeroed rows (generic proxy) and P (tcgen05.st) before the MMA reads
          fence_proxy_async_smem();
          tc::fence_after_sync();
          const uint64_t bv = dv0 + sp * kTileDesc;
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            tc::mma_f16_ts(tmem + col_o(t), tmem + col_s(t) + kk * 8, bv + (kk * 2048 >> 4),
                           idesc_pv, (jr > 0 || kk > 0) ? 1u : 0u);
          tc::mma_commit(&B->v_empty[sp]);
          if (jj == nt) tc::mma_commit(&B->o_done[t]);
        }
        if (jj < nt) {
          const int s = jj % kStagesK;
          ok = wait_or_abort(&B->k_full[s], (jj / kStagesK) & 1, B, p.error_word, p.wait_ns);
          if (!ok) break;
          const uint64_t bk = dk0 + s * kTileDesc;
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
            tc::mma_f16(tmem + col_s(t), aq + off, bk + off, idesc_qk, kk > 0);
          }
          tc::mma_commit(&B->s_full[t]);
          tc::mma_commit(&B->k_empty[s]);
        }
      }
      // drain: all issued MMAs complete before tensor memory is released
      tc::mma_commit(&B->drain[t]);
      mbar_wait(&B->drain[t], 0, p.wait_ns);
    }
    __syncwarp();
  } else if (warp < 8) {
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
      asm volatile("bar.sync 1, 320;" ::: "memory");
    }
    const bool active = t == 0 || has_t1;
    const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t colS = col_s(t), colO = col_o(t);
    float m_run = -INFINITY, l_run = 0.f;
    const float sl = p.scale_log2;
    bool ok = active;
    // keys before key_row are outside this row's window
    const int key_row = p.window > 0 ? pos - p.window + 1 : -(1 << 30);
    for (int jj = 0; jj < nt && ok; ++jj) {
      // the two warpgroups take turns (softmax 0 of tile j, softmax 1 of
      // tile j, softmax 0 of tile j + 1, ...), so each runs alone on the
      // SM's exp and FMA units while the tensor core works for the other
      if (has_t1 && (t == 1 || jj >= 1)) {
        const bool tw = __all_sync(0xffffffffu, t == 0 ? mbar_wait(&B->p_full[1], (jj - 1) & 1, p.wait_ns)
                                                     : mbar_wait(&B->p_full[0], jj & 1, p.wait_ns));
        if (!tw) { abort_cta(B, p.error_word); ok = false; break; }
      }
      bool w = __all_sync(0xffffffffu, mbar_wait(&B->s_full[t], jj & 1, p.wait_ns));
      if (!w) { abort_cta(B, p.error_word); ok = false; break; }
      tc::fence_after_sync();
      const int kbase = (j_lo + jj) * kBN;
      const int lim = pos - kbase;               // key kbase+i visible iff lo <= i <= lim
      const int lo = key_row - kbase;
      const bool masked = lim < kBN - 1 || lo > 0;
      // the whole S row in registers with one TMEM wait
      float sv[kBN];
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) tc::tmem_ld32(trow + colS + 32 * c, sv + 32 * c);
      tc::tmem_wait_ld();
      if (masked) {
#pragma unroll
        for (int i = 0; i < kBN; ++i) sv[i] = (i <= lim && i >= lo) ? sv[i] : -INFINITY;
      }
      // row max in 8 chains of 3-input max
      float mx[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mx[u] = fmax3(sv[u], sv[8 + u], sv[16 + u]);
#pragma unroll
      for (int i = 24; i + 16 <= kBN; i += 16)
#pragma unroll
        for (int u = 0; u < 8; ++u) mx[u] = fmax3(mx[u], sv[i + u], sv[i + 8 + u]);
#pragma unroll
      for (int u = 0; u < 8; ++u) mx[u] = fmaxf(mx[u], sv[kBN - 8 + u]);
      const float mt_max = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                 fmaxf(mx[6], mx[7])) * sl;
      const float m_new = fmaxf(m_run, mt_max);
      const bool resc = (m_new - m_run) > 8.f;   // also true on the first tile
      const float m_use = resc ? m_new : m_run;  // weights stay <= 2^8 otherwise
      const float alpha = resc ? fast_exp2(m_run - m_use) : 1.f;
      m_run = m_use;
      // p = 2^(s*scale - m) for a pair of scores at a time: one packed FMA,
      // the pair rounded to bf16, one packed bf16 ex2 -- which is already P
      // in the bf16 layout the P.V MMA reads.  The row sum adds those bf16
      // values two pairs at a time in bf16 (one rounding, relative 2^-9),
      // then in fp32 (4 packed chains).  P is written over the S columns
      // (all read above).
      // a row with every key so far masked has m_use = -inf: subtract 0
      // instead, so its masked scores give 2^-inf = 0 rather than NaN
      const float m_sub = m_use == -INFINITY ? 0.f : m_use;
      const float2 sl2 = make_float2(sl, sl), nm2 = make_float2(-m_sub, -m_sub);
      float2 ls2[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) ls2[u] = make_float2(0.f, 0.f);
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float2 x2 = __ffma2_rn(make_float2(sv[32 * h + i], sv[32 * h + i + 1]), sl2, nm2);
          const float2 y2 = __ffma2_rn(make_float2(sv[32 * h + i + 2], sv[32 * h + i + 3]), sl2, nm2);
          const uint32_t pa = fast_exp2_bf16x2(float2_to_bf16x2(x2.x, x2.y));
          const uint32_t pb = fast_exp2_bf16x2(float2_to_bf16x2(y2.x, y2.y));
          pk[i / 2] = pa;
          pk[i / 2 + 1] = pb;
          // two P pairs added in bf16 first (one rounding), then in fp32
          uint32_t ps;
          asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(ps) : "r"(pa), "r"(pb));
          ls2[(i >> 2) & 3] = __fadd2_rn(ls2[(i >> 2) & 3], bf16x2_to_float2(ps));
        }
        tc::tmem_st16(trow + colS + 16 * h, pk);
      }
      const float lsum = ((ls2[0].x + ls2[0].y) + (ls2[1].x + ls2[1].y)) +
                         ((ls2[2].x + ls2[2].y) + (ls2[3].x + ls2[3].y));
      l_run = l_run * alpha + lsum;
      // S_t(j) ready implies P_t.V(j-1) completed (same issuing thread, in
      // order), so O_t is stable here and may be rescaled.
      if (jj >= 1 && __any_sync(0xffffffffu, resc)) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float o[32];
          tc::tmem_ld32_sync(trow + colO + 32 * c, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= alpha;
          tc::tmem_st32(trow + colO + 32 * c, o);
        }
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&B->p_full[t]);
    }
    // epilogue: O_t / l -> bf16 rows
    if (ok) {
      const bool w = __all_sync(0xffffffffu, mbar_wait(&B->o_done[t], 0, p.wait_ns));
      if (!w) abort_cta(B, p.error_word);
      if (w) {
        tc::fence_after_sync();
        const float inv = 1.f / l_run;
        uint4* dst = reinterpret_cast<uint4*>(p.out + ((int64_t)(q0 + tok) * p.num_q_heads + head) * kD);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float o[32];
          tc::tmem_ld32_sync(trow + colO + 32 * c, o);
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
  if (warp == kMmaWarp) tc::tmem_dealloc(tmem, kTmemCols);
  order_after_previous_grid();
}

}  // namespace prefill

bool prefill_supported(int group) {
  return group == 1 || group == 2 || group == 4 || group == 8 || group == 16;
}

size_t prefill_workspace_bytes(int64_t, int64_t, int64_t) { return 0; }

int64_t prefill_ctas(const cb_attention_args& a) {
  using namespace prefill;
  const int G = a.num_q_heads / a.num_kv_heads;
  if (G <= 0 || G > kBM) return 0;
  const int tpp = 2 * (kBM / G);  // tokens per CTA (a pair of query tiles)
  // every row's pairs: at most (prefill tokens) / tpp rounded up per row
  const int64_t pairs = ((int64_t)a.num_tokens - a.num_decodes + tpp - 1) / tpp +
                        (a.num_reqs - a.num_decodes);
  return pairs > 0 ? pairs * a.num_kv_heads : 0;
}

cb_status launch_prefill_bf16(const cb_attention_args& a, uint32_t* error_word, uint8_t*,
                              cudaStream_t stream, bool overlap_previous) {
  using namespace prefill;
  if (a.head_dim != kD || a.block_size != kPage || a.dtype != CB_DTYPE_BF16) return CB_ERR_UNSUPPORTED;
  const int G = a.num_q_heads / a.num_kv_heads;
  if (!prefill_supported(G)) return CB_ERR_UNSUPPORTED;
  const size_t smem = SmemLayout::total + 1024;
  static std::atomic<uint8_t> attr_set[kMaxDevices];
  cb_status st = ensure_smem_attr(reinterpret_cast<const void*>(prefill_kernel), smem, attr_set);
  if (st != CB_OK) return st;
  const int64_t rows = (int64_t)a.num_blocks * a.num_kv_heads * kPage;
  if (rows >= ((int64_t)1 << 31) - kPage) return CB_ERR_UNSUPPORTED;
  Params p{};
  st = cached_cache_map(&p.tmap_k, a.k_cache, rows, kD);
  if (st != CB_OK) return st;
  st = cached_cache_map(&p.tmap_v, a.v_cache, rows, kD);
  if (st != CB_OK) return st;
  p.k_cache = a.k_cache;
  p.v_cache = a.v_cache;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.cu_seqlens_q = a.cu_seqlens_q;
  p.seq_lens = a.seq_lens;
  p.block_tables = a.block_tables;
  p.row_begin = a.num_decodes;
  p.num_rows = a.num_reqs - a.num_decodes;
  p.num_tokens = a.num_tokens;
  p.num_blocks = a.num_blocks;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = G;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.window = a.sliding_window;
  p.error_word = error_word;
  p.wait_ns = wait_limit_ns();
  p.withhold_tile = withheld_prefill_tile();
  const int64_t ctas = prefill_ctas(a);
  if (ctas <= 0) return CB_OK;
  if (ctas >= ((int64_t)1 << 31)) return CB_ERR_UNSUPPORTED;
  dim3 grid((unsigned)ctas, 1, 1);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute lattr[1];
  lattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  lattr[0].val.programmaticStreamSerializationAllowed = overlap_previous ? 1 : 0;
  cfg.attrs = lattr;
  cfg.numAttrs = 1;
  cudaError_t le = cudaLaunchKernelEx(&cfg, prefill_kernel, p);
  if (le != cudaSuccess) return fail(CB_ERR_CUDA, "prefill kernel launch: %s", cudaGetErrorString(le));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(CB_ERR_CUDA, "prefill kernel launch: %s", cudaGetErrorString(e));
  return CB_OK;
}

}  // namespace cb
