/*
 * cb.h -- C ABI of the GB300 continuous-batching paged-attention step.
 *
 * One serving step of a continuous-batching engine with chunked prefill and
 * a paged KV cache:
 *
 *   1. cb_schedule_step  (host)  picks the batch: one token per running
 *      decode, then prefill chunks, under a token budget, a request cap and
 *      the free-block budget, and emits the step's metadata
 *      (cu_seqlens_q, seq_lens, block_tables, slot_mapping).
 *   2. cb_kv_append      (GPU)   writes the step's new K/V into the paged
 *      cache at slot_mapping.
 *   3. cb_paged_attention(GPU)   every scheduled query attends, causally over
 *      absolute positions, to its request's K/V read through its block table.
 *   4. cb_step_done      (host)  commits the step: advances each request,
 *      finishes requests and returns their blocks to the pool.
 *
 * Around the step: cb_kv_swap (GPU) moves offloaded requests' blocks to and
 * from a pinned host swap pool; cb_validate_step (host) checks a step's
 * metadata; cb_paged_decode_noalloc runs decode rows without a caller
 * workspace; the scheduler options cover the PrefillFirst policy, prefill
 * caps, offloading with soft reset, prefix caching with eviction
 * (cb_add_request_tokens) and sliding-window layers, and
 * cb_sched_hold_blocks / cb_sched_release_blocks inject memory pressure.
 *
 * Sources (page title, section):
 *   - "Continuous batching architecture" (HF Transformers docs): Request
 *     lifecycle; Chunked prefill; Scheduler (token budget max_batch_tokens,
 *     cache budget, request cap max_requests_per_batch); FIFO; Admission
 *     (all-or-nothing, safety_margin); Offloading (stalled requests and their
 *     block demand; offloading to a CPU swap pool; Soft reset); Prefix
 *     caching; Eviction; PrefillFirst; Memory management (sliding layers).
 *   - "Chunked Prefill" (Ultralytics glossary): How chunked prefill works
 *     (decode tokens first, then chunks; each chunk attends under a causal
 *     mask over absolute positions to all earlier chunks plus itself).
 *   - "vLLM serving internals" (AI Engineering from Scratch, phase 17 lesson
 *     04): PagedAttention as a virtual memory system (fixed 16-token blocks,
 *     per-sequence block tables, blocks back to the pool on finish);
 *     Iteration-level continuous batching; What the scheduler looks like.
 *
 * Conventions for every call:
 *   - Every function returns cb_status; CB_OK == 0.  On failure
 *     cb_last_error() returns a thread-local message.  No C++ exception
 *     crosses this boundary.
 *   - GPU calls are asynchronous on the given stream (a cudaStream_t passed
 *     as cb_stream_t; NULL = legacy default stream).  Argument errors are
 *     detected on the host before anything is launched.  Errors found on
 *     the device (a block id outside the pool, a slot outside the cache, a
 *     decode row whose query length is not 1, a timed-out wait) set bits in
 *     the workspace's device error word instead of faulting; read them with
 *     cb_attention_read_errors.
 *   - All device pointers are caller-owned (e.g. allocated by PyTorch) and
 *     must stay valid until the stream has executed the call.  Nothing here
 *     allocates device memory; the attention workspace is sized by
 *     cb_attention_workspace_size and owned by the caller.
 *   - Cache layout: k_cache and v_cache are [num_blocks][Hkv][block_size][D],
 *     row-major, so one (block, KV head) page of block_size x D elements is
 *     contiguous.  Token tensors are [tokens][heads][D].  block_size is 16.
 */
#ifndef CB_H_
#define CB_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* cb_stream_t; /* same type as cudaStream_t */

typedef enum cb_status {
  CB_OK = 0,
  CB_ERR_INVALID_ARG = 1,   /* bad argument; nothing was changed or launched */
  CB_ERR_NO_BLOCKS = 2,     /* no batch could be scheduled: the cache is full
                               (see cb_step.stalled_*) or the next waiting
                               request does not fit */
  CB_ERR_CUDA = 3,          /* a CUDA runtime call failed */
  CB_ERR_UNSUPPORTED = 4,   /* valid but not implemented shape/dtype */
  CB_ERR_DEVICE_CHECK = 5,  /* a kernel reported bad metadata (see
                               cb_attention_read_errors) */
  CB_ERR_STATE = 6          /* call out of order (e.g. two schedule calls
                               without cb_step_done) */
} cb_status;

typedef enum cb_dtype {
  CB_DTYPE_F32 = 0,         /* float32 storage, float32 arithmetic */
  CB_DTYPE_BF16 = 1         /* bfloat16 storage, float32 accumulation,
                               outputs rounded to nearest even */
} cb_dtype;

/* Returns the message of the last failed call on this thread ("" if none). */
const char* cb_last_error(void);

/* ABI version, (major << 16) | minor. */
int32_t cb_version(void);

/* ------------------------------------------------------------------------
 * Scheduler (host).
 * "Continuous batching architecture", sections Scheduler / FIFO / Admission /
 * Offloading; "vLLM serving internals", What the scheduler looks like.
 * ---------------------------------------------------------------------- */
typedef struct cb_config {
  int32_t block_size;             /* tokens per KV block; > 0 */
  int32_t num_blocks;             /* blocks in the pool; > 0 */
  int32_t max_batch_tokens;       /* token budget per step; > 0 */
  int32_t max_requests_per_batch; /* request cap per step (decodes count); > 0 */
  int32_t max_prefill_chunk;      /* per-request prefill chunk cap; 0 = none */
  int32_t max_blocks_per_seq;     /* width of a block_tables row; a request
                                     whose prompt_len+output_len-1 tokens need
                                     more blocks is rejected */
  float safety_margin;            /* fraction of num_blocks that must stay
                                     free after admitting a NEW request:
                                     admit iff free_after >=
                                     ceil((double)margin * num_blocks).
                                     FIFO default 0.15; 0 disables it */
  const int32_t* initial_free_list; /* optional host array of num_blocks
                                       distinct ids in [0, num_blocks): the
                                       allocation order; NULL = 0,1,2,...
                                       Copied; not retained. */
  int32_t policy;                 /* CB_POLICY_FIFO (0, default): decodes,
                                     running prefills, new prompts;
                                     CB_POLICY_PREFILL_FIRST (1): running
                                     prefills, new prompts, then decodes with
                                     what is left ("Continuous batching
                                     architecture", PrefillFirst).  Rows are
                                     always emitted decodes first. */
  int32_t max_prefill_reqs;       /* prefill rows (running + new) per step;
                                     0 = no cap */
  int32_t long_prefill_tokens;    /* prompts longer than this are "long";
                                     0 = no long-prefill cap */
  int32_t max_long_prefills;      /* long requests allowed in their prefill
                                     phase at once (vLLM post, request-
                                     parallel prefill); a long waiting
                                     request held by it is skipped, not
                                     blocking shorter ones behind it */
  int32_t offload;                /* 0: stalled requests are only reported.
                                     1: offload them ("Continuous batching
                                     architecture", Offloading / Soft
                                     reset): the fewest stalled requests,
                                     newest first, never the last active
                                     one, when a batch was scheduled; when
                                     none fits, the newest active requests,
                                     retrying within the step.  A victim
                                     goes to the CPU swap pool if its free
                                     slots hold all its blocks, else it is
                                     soft-reset (generated tokens join the
                                     prompt, blocks freed, front of the
                                     queue).  Swapped requests are resumed,
                                     oldest offload first, at the start of a
                                     later step when blocks allow. */
  int32_t swap_blocks;            /* CPU swap pool capacity in blocks (one
                                     block of every layer's K and V per
                                     slot); 0 = soft reset only */
  int32_t prefix_caching;         /* 1: share blocks of equal prompt
                                     prefixes ("Continuous batching
                                     architecture", Prefix caching,
                                     Eviction) among requests queued with
                                     cb_add_request_tokens.  A block inside
                                     the known prompt tokens is keyed, when
                                     the step that completes it is
                                     committed, by a fingerprint of the whole
                                     token prefix up to its end (128 bits,
                                     plus a check of the block's own tokens)
                                     unless another block holds that key.
                                     At admission the longest leading run of
                                     keyed blocks is reused (at most
                                     prompt_len - 1 tokens: one prompt token
                                     is always computed); reused tokens are
                                     cached and take no budget.  Blocks are
                                     reference-counted; a freed keyed block
                                     keeps its K/V and key in an
                                     "initialized" pool and can still be
                                     matched; allocation takes the free
                                     queue first and then demotes the NEWEST
                                     initialized block (its key dropped).
                                     Free capacity counts both. */
  int32_t sliding_window;         /* W > 0: every layer served by this pool
                                     is a sliding-window layer ("Continuous
                                     batching architecture", Memory
                                     management): a query at position p
                                     reads keys p-W+1..p only.  After each
                                     committed step, pages of a running
                                     request that lie wholly before
                                     num_cached - W + 1 are recycled (to the
                                     free queue's tail, batch order then
                                     table order, before finished requests
                                     release theirs) and their table entries
                                     become -1.  Only live pages are swapped.
                                     Not combinable with prefix_caching.
                                     0 = full attention. */
} cb_config;

#define CB_POLICY_FIFO 0
#define CB_POLICY_PREFILL_FIRST 1

typedef struct cb_sched cb_sched;

/* One scheduled step.  All arrays are HOST memory owned by the scheduler,
 * valid until the next cb_schedule_step or cb_sched_destroy.  Batch order:
 * decodes (admission order), then running prefills (admission order), then
 * newly admitted prompts (arrival order). */
typedef struct cb_step {
  int32_t num_reqs;              /* R */
  int32_t num_tokens;            /* T = cu_seqlens_q[R] */
  int32_t num_decodes;           /* the first num_decodes rows are decodes
                                    (exactly one query token each) */
  int32_t max_q_len;             /* max over rows of the query length */
  int32_t max_seq_len;           /* max over rows of seq_lens */
  int32_t max_blocks_per_seq;    /* row stride of block_tables */
  const int64_t* req_ids;        /* [R] */
  const int32_t* cu_seqlens_q;   /* [R+1] prefix sums of query lengths */
  const int32_t* seq_lens;       /* [R] tokens in the cache after this step's
                                    append (cached + scheduled) */
  const int32_t* block_tables;   /* [R][max_blocks_per_seq], -1 padded */
  const int32_t* slot_mapping;   /* [T] block*block_size + offset of each new
                                    token's K/V */
  int32_t num_stalled;           /* active requests that could not get the
                                    blocks they need this step */
  const int64_t* stalled_ids;    /* [num_stalled] */
  const int32_t* stalled_demand; /* [num_stalled] blocks each one needs */
  /* KV copies the caller must make BEFORE this step's kernels, in this
   * order (also when the step returns CB_ERR_NO_BLOCKS): swap-ins, swap
   * pool slot -> cache block; then swap-outs, cache block -> swap pool
   * slot (cb_kv_swap moves every layer's K and V of each pair). */
  int32_t num_swap_in;
  const int32_t* swap_in_slots;  /* [num_swap_in] */
  const int32_t* swap_in_blocks; /* [num_swap_in] */
  int32_t num_swap_out;
  const int32_t* swap_out_blocks; /* [num_swap_out] */
  const int32_t* swap_out_slots;  /* [num_swap_out] */
} cb_step;

/* Create / destroy a scheduler.  *out is NULL on failure. */
cb_status cb_sched_create(const cb_config* cfg, cb_sched** out);
void cb_sched_destroy(cb_sched* s);

/* Queue a new request (state PENDING); arrival order = call order.
 * CB_ERR_INVALID_ARG for a duplicate id, prompt_len < 1, output_len < 1 or a
 * request longer than max_blocks_per_seq blocks. */
cb_status cb_add_request(cb_sched* s, int64_t req_id, int32_t prompt_len,
                         int32_t output_len);

/* cb_add_request with the ids of the first num_tokens (<= prompt_len)
 * prompt tokens (host array, copied), which prefix caching matches on.
 * Without prefix_caching the ids are ignored. */
cb_status cb_add_request_tokens(cb_sched* s, int64_t req_id, int32_t prompt_len,
                                int32_t output_len, const int32_t* tokens,
                                int32_t num_tokens);

/* Resume a request whose first num_cached tokens already have K/V in the
 * cache (the swap-in path of "Offloading": resume without recomputing).  It
 * joins the running set after the requests already there and takes
 * ceil(num_cached / block_size) blocks from the free list.  If num_cached >=
 * prompt_len it is DECODING with num_cached - prompt_len + 1 tokens generated
 * (requires num_cached <= prompt_len + output_len - 2), else PREFILLING.
 * CB_ERR_NO_BLOCKS if the pool is too small (nothing allocated). */
cb_status cb_add_running_request(cb_sched* s, int64_t req_id,
                                 int32_t prompt_len, int32_t output_len,
                                 int32_t num_cached);

/* Schedule the next step (FIFO policy).  Returns CB_OK with a possibly empty
 * batch, or CB_ERR_NO_BLOCKS when nothing could be scheduled although
 * requests are stalled or waiting; *out is filled in both cases.  After
 * CB_OK the caller runs the step and then must call cb_step_done before the
 * next cb_schedule_step (CB_ERR_STATE otherwise). */
cb_status cb_schedule_step(cb_sched* s, cb_step* out);

/* Commit the last CB_OK step.  *num_finished / *finished_ids (host, owned by
 * the scheduler, valid until the next call) list requests that finished, in
 * batch order; their blocks went back to the tail of the free list (keyed
 * blocks to the initialized pool, shared blocks once their last user
 * finished).  Either
 * output pointer may be NULL. */
cb_status cb_step_done(cb_sched* s, int32_t* num_finished,
                       const int64_t** finished_ids);

/* slots_out[i] = slot of position start+i of request req_id (positions must
 * lie inside the request's allocated blocks). */
cb_status cb_request_slots(const cb_sched* s, int64_t req_id, int32_t start,
                           int32_t count, int32_t* slots_out);

/* Pool and queue sizes; any output pointer may be NULL. */
cb_status cb_sched_counts(const cb_sched* s, int32_t* free_blocks,
                          int32_t* num_waiting, int32_t* num_running);

/* Copies the free list into out[0..capacity): the free queue in allocation
 * order, then the initialized pool (prefix caching) oldest first; *count
 * gets its length. */
cb_status cb_sched_free_list(const cb_sched* s, int32_t* out, int32_t capacity,
                             int32_t* count);

/* Fault injection (a test hook for memory pressure; between steps only,
 * CB_ERR_STATE while a step is open).  cb_sched_hold_blocks takes up to n
 * blocks out of the allocatable pool exactly as allocation would (free
 * queue head first, then the newest initialized blocks, demoted), writes
 * their ids to out_ids and their number to *count; they stay out until
 * cb_sched_release_blocks puts them back at the free queue's tail, in the
 * given order (CB_ERR_INVALID_ARG, nothing released, if an id is not held
 * or is listed twice). */
cb_status cb_sched_hold_blocks(cb_sched* s, int32_t n, int32_t* out_ids, int32_t* count);
cb_status cb_sched_release_blocks(cb_sched* s, const int32_t* ids, int32_t n);

/* Prefix caching counters (any pointer may be NULL): prompt tokens reused
 * from cached blocks so far, keyed blocks, keyed blocks in the initialized
 * pool (free but still matchable). */
cb_status cb_sched_prefix_stats(const cb_sched* s, int64_t* hit_tokens,
                                int32_t* keyed_blocks, int32_t* pool_blocks);

/* Requests currently in the swap pool (offload order) into out[0..capacity);
 * *count gets their number; free swap slots into *free_slots (NULL ok). */
cb_status cb_sched_swapped(const cb_sched* s, int64_t* out, int32_t capacity,
                           int32_t* count, int32_t* free_slots);

/* ------------------------------------------------------------------------
 * cb_validate_step (host).  Checks a step's metadata, given as HOST arrays,
 * against what cb_kv_append and cb_paged_attention require, and names the
 * first row or token that breaks a rule (CB_ERR_INVALID_ARG, message in
 * cb_last_error()):
 *   - cu_seqlens_q[0] >= 0 and non-decreasing, cu_seqlens_q[num_reqs] <=
 *     num_tokens; rows [0, num_decodes) have one query (or are padding);
 *   - a row with no queries has seq_len 0 (padding); otherwise seq_len >=
 *     its query length and ceil(seq_len / block_size) <= max_blocks_per_seq;
 *   - every block id the row's queries read (from the first query's window
 *     with sliding_window > 0) lies in [0, num_blocks);
 *   - slot_mapping (optional, may be NULL) entries lie in [-1, num_blocks *
 *     block_size).
 * With CB_VALIDATE=1 in the environment, cb_paged_attention and
 * cb_kv_append copy their metadata back (synchronising the stream) and run
 * these checks before launching, except while the stream is being captured
 * into a CUDA graph.
 * ---------------------------------------------------------------------- */
cb_status cb_validate_step(const int32_t* cu_seqlens_q, const int32_t* seq_lens,
                           const int32_t* block_tables, const int32_t* slot_mapping,
                           int32_t num_reqs, int32_t num_decodes, int32_t num_tokens,
                           int32_t max_blocks_per_seq, int32_t num_blocks,
                           int32_t block_size, int32_t sliding_window);

/* ------------------------------------------------------------------------
 * cb_kv_append (GPU).  "vLLM serving internals", PagedAttention as a virtual
 * memory system: token t's K/V goes to block slot_mapping[t] / block_size,
 * offset slot_mapping[t] % block_size, for every KV head.
 *
 *   k_new, v_new  device [num_tokens][Hkv][D] (dtype)
 *   slot_mapping  device int32 [num_tokens]; -1 = padding, skipped
 *   k_cache, v_cache device [num_blocks][Hkv][block_size][D] (dtype)
 *   error_word    optional device uint32; a slot >= num_blocks*block_size is
 *                 skipped and sets CB_DEVERR_SLOT_RANGE there.
 * D * sizeof(dtype) must be 16 bytes times a power of two (every head size
 * the attention takes) and every pointer 16-byte aligned; at most 2^31
 * 16-byte vectors per call (CB_ERR_UNSUPPORTED otherwise).  Bit-exact copy.
 * ---------------------------------------------------------------------- */
cb_status cb_kv_append(const void* k_new, const void* v_new,
                       const int32_t* slot_mapping, int32_t num_tokens,
                       void* k_cache, void* v_cache, int32_t num_blocks,
                       int32_t num_kv_heads, int32_t head_dim,
                       int32_t block_size, cb_dtype dtype,
                       uint32_t* error_word, cb_stream_t stream);

/* ------------------------------------------------------------------------
 * cb_kv_swap (GPU).  "Continuous batching architecture", Offloading: move
 * whole KV blocks between two sets of pools in one launch -- for every pair
 * i and every pool k:  dst_pools[k][dst_ids[i]] = src_pools[k][src_ids[i]]
 * (block_bytes each).  The pools are typically every layer's K and V cache
 * on one side and the same layers' pinned-host swap pools on the other;
 * either side may be memory of the current device or pinned host memory
 * (accessed directly by the kernel through its mapped device address);
 * any other pointer is refused with CB_ERR_INVALID_ARG before a launch.  Pairs whose ids fall outside [0, src_capacity) /
 * [0, dst_capacity) are skipped and flagged (CB_DEVERR_BLOCK_RANGE in
 * error_word, optional).  src_ids/dst_ids are device arrays; the pool
 * pointer arrays are host arrays read at the call.  The caller keeps the
 * source blocks unchanged until the copy has run (stream order).
 * ---------------------------------------------------------------------- */
#define CB_SWAP_MAX_POOLS 128
typedef struct cb_swap_args {
  int32_t num_pairs;
  const int32_t* src_ids;       /* device [num_pairs] */
  const int32_t* dst_ids;       /* device [num_pairs] */
  int32_t num_pools;            /* pools moved per pair, <= CB_SWAP_MAX_POOLS */
  const void* const* src_pools; /* host [num_pools] base pointers, 16-B aligned */
  void* const* dst_pools;       /* host [num_pools] base pointers, 16-B aligned */
  int64_t src_capacity;         /* blocks in each source pool */
  int64_t dst_capacity;         /* blocks in each destination pool */
  int64_t block_bytes;          /* bytes per block (Hkv * block_size * D * elem),
                                   a multiple of 16 */
  uint32_t* error_word;         /* optional device word */
} cb_swap_args;

cb_status cb_kv_swap(const cb_swap_args* args, cb_stream_t stream);

/* ------------------------------------------------------------------------
 * cb_paged_attention (GPU).  "Chunked Prefill", How chunked prefill works:
 * query i of row r (absolute position p = seq_lens[r] - q_len + i) attends
 * to keys 0..p of its own request, read through block_tables[r]:
 *   out[t,h] = sum_{j<=p} softmax_j(scale * q[t,h].k[j,g]) v[j,g],
 *   g = h / (Hq/Hkv).
 * Rows [0, num_decodes) must have query length 1 and run the split-KV decode
 * kernel (which also merges the splits of requests whose cache it split);
 * the remaining rows run the prefill-chunk kernel.  Both go to `stream`;
 * the prefill kernel may start on SMs the decode kernel has left (the two
 * share no data), and it completes only after the decode kernel, so work
 * queued on `stream` after the call runs after both.
 * With sliding_window = W > 0 the sum runs over j = p-W+1..p instead.
 * A row with query length 0 and seq_len 0 is padding and is skipped (no
 * error bit), so a step may be padded to a fixed shape (row counts, token
 * count, max_q_len) and captured once in a CUDA graph; padded tokens carry
 * slot -1 for cb_kv_append.
 * ---------------------------------------------------------------------- */
typedef struct cb_attention_args {
  const void* q;                /* device [num_tokens][Hq][D] */
  void* out;                    /* device [num_tokens][Hq][D], same dtype */
  const void* k_cache;          /* device [num_blocks][Hkv][block_size][D] */
  const void* v_cache;          /* same layout */
  const int32_t* cu_seqlens_q;  /* device [num_reqs+1] */
  const int32_t* seq_lens;      /* device [num_reqs] */
  const int32_t* block_tables;  /* device [num_reqs][max_blocks_per_seq] */
  int32_t num_reqs;
  int32_t num_decodes;          /* rows [0, num_decodes) are decodes */
  int32_t num_tokens;
  int32_t max_q_len;            /* host bound on rows' query length */
  int32_t max_seq_len;          /* host bound on seq_lens */
  int32_t num_blocks;           /* pool size (block ids are range-checked) */
  int32_t max_blocks_per_seq;
  int32_t block_size;           /* must be 16 */
  int32_t num_q_heads;          /* Hq, a multiple of Hkv */
  int32_t num_kv_heads;         /* Hkv */
  int32_t head_dim;             /* D: 64 or 128 */
  float scale;                  /* softmax scale, usually 1/sqrt(D) */
  cb_dtype dtype;
  void* workspace;              /* device, >= cb_attention_workspace_size(),
                                   256-byte aligned, zeroed once by
                                   cb_attention_workspace_init; calls leave it
                                   ready for the next call */
  size_t workspace_bytes;
  int32_t sliding_window;       /* W > 0: sliding-window layer ("Continuous
                                   batching architecture", Memory management)
                                   -- query position p attends keys
                                   p-W+1..p only, and table entries of pages
                                   wholly before a row's window are never
                                   read (they may be -1); 0: full attention */
  int32_t after_append;         /* 1: the kernel queued just before on the
                                   stream is the cb_kv_append of this step
                                   (the append of "vLLM serving internals",
                                   PagedAttention as a virtual memory system);
                                   the decode kernel then starts while the
                                   append finishes (programmatic dependent
                                   launch), plans its work meanwhile and reads
                                   the cache only once the append is complete.
                                   0: plain stream order.  Setting it when the
                                   kernel before is not that append is
                                   undefined. */
} cb_attention_args;

/* Device error bits (cb_attention_read_errors / cb_kv_append error_word). */
#define CB_DEVERR_BLOCK_RANGE 0x1u  /* block id outside [0, num_blocks) */
#define CB_DEVERR_SLOT_RANGE 0x2u   /* slot outside the cache */
#define CB_DEVERR_DECODE_QLEN 0x4u  /* a decode row with query length != 1 */
#define CB_DEVERR_SEQ_RANGE 0x8u    /* seq_len < q_len, beyond the table, or a
                                       row's queries outside [0, num_tokens) */
#define CB_DEVERR_TIMEOUT 0x10u     /* a bounded wait ran out */
#define CB_DEVERR_PLAN 0x20u        /* decode splits did not fit the partial slots */

/* Workspace bytes for calls with up to num_reqs rows and these head sizes
 * (0 on bad args).  One workspace serves any later call with at most that
 * many rows and the same head sizes; the regions that carry state between
 * calls sit at fixed offsets.  num_kv_heads <= 64. */
size_t cb_attention_workspace_size(int32_t num_reqs, int32_t num_q_heads,
                                   int32_t num_kv_heads, int32_t head_dim);

/* Zero a freshly allocated workspace (async on stream).  Needed once; after
 * a CB_ERR_DEVICE_CHECK, call it again. */
cb_status cb_attention_workspace_init(void* workspace, size_t workspace_bytes,
                                      cb_stream_t stream);

cb_status cb_paged_attention(const cb_attention_args* args, cb_stream_t stream);

/* Synchronizes the stream and reads (and clears) the device error word of a
 * workspace.  Returns CB_ERR_DEVICE_CHECK if any bit was set. */
cb_status cb_attention_read_errors(void* workspace, size_t workspace_bytes,
                                   cb_stream_t stream, uint32_t* bits);

/* ------------------------------------------------------------------------
 * cb_debug_inject_wait_timeout (test hook; no counterpart in the pages).
 *
 * Every device wait of the attention kernels is bounded: a wait that runs
 * out records CB_DEVERR_TIMEOUT, the kernel drains what it started and
 * returns, and the workspace is left ready for the next call (the failure
 * detection of "Continuous batching architecture" carried to the device,
 * without a GPU fault).  This hook lets a test make such a wait run out:
 *   wait_ns       limit of every bounded wait of later launches (0: the
 *                 default of 1 s);
 *   decode_item   >= 0: the decode kernel announces the first page of its
 *                 work item with this index but never copies it;
 *   prefill_tile  >= 0: CTA 0 of the prefill kernel announces its K tile
 *                 with this index but never copies it;
 *                 -1 for either: nothing is withheld.
 * The call itself launches nothing; it affects launches made after it,
 * from any thread.  Not for production use.
 * ---------------------------------------------------------------------- */
cb_status cb_debug_inject_wait_timeout(uint64_t wait_ns, int32_t decode_item,
                                       int32_t prefill_tile);

/* ------------------------------------------------------------------------
 * Step executor (host + GPU).  "Continuous batching architecture", Async
 * batching: the host schedules step N+1 while the device computes step N,
 * and step N+1's inputs and step N-1's output cross the CPU-GPU link at the
 * same time.  An executor owns two sets of device buffers (q, k_new, v_new,
 * out for every layer, and the packed step metadata), a pinned staging
 * buffer per set, a workspace, and three streams (copy-in, compute,
 * copy-out); the KV caches stay the caller's.  Steps use the two sets in
 * turn.  For one step, cb_executor_submit packs the step's host metadata
 * into the set's pinned buffer and queues: the metadata and every layer's
 * q/k/v rows host -> device (after the set's previous compute); per layer
 * cb_kv_append + cb_paged_attention (after that copy and after the set's
 * previous copy-out); every layer's output rows device -> host.  It returns
 * without waiting.
 *
 *   config        caches: device [num_blocks][Hkv][block_size][D] per layer
 *                 (host arrays of num_layers pointers, copied); sizes bound
 *                 every later step (max_reqs rows, max_tokens tokens,
 *                 block tables of max_blocks_per_seq columns).
 *   q/k/v_host    host [num_layers] pointers to [T][H][D] rows of the step
 *                 (pinned memory keeps the copies asynchronous; other host
 *                 memory is copied synchronously); they must stay unchanged
 *                 until cb_executor_synchronize.
 *   out_host      host [num_layers] pointers receiving [T][Hq][D]; complete
 *                 after cb_executor_synchronize.
 * Steps that carry offload swaps are refused (CB_ERR_UNSUPPORTED): the
 * executor does not own a swap pool.  create allocates device and pinned
 * memory; submit and run_step allocate nothing.
 * ---------------------------------------------------------------------- */
typedef struct cb_executor cb_executor;

typedef struct cb_executor_config {
  int32_t num_layers;
  void* const* k_caches;        /* host [num_layers] device pointers */
  void* const* v_caches;
  int32_t num_blocks;
  int32_t block_size;           /* 16 */
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  cb_dtype dtype;
  float scale;                  /* softmax scale */
  int32_t sliding_window;       /* 0: full attention */
  int32_t max_reqs;
  int32_t max_tokens;
  int32_t max_blocks_per_seq;
} cb_executor_config;

cb_status cb_executor_create(const cb_executor_config* cfg, cb_executor** out);
void cb_executor_destroy(cb_executor* ex);

/* Queue one scheduled step (see above); an empty step is a no-op. */
cb_status cb_executor_submit(cb_executor* ex, const cb_step* step,
                             const void* const* q_host, const void* const* k_host,
                             const void* const* v_host, void* const* out_host);

/* Schedule the next step of `sched`, submit it, and commit it with
 * cb_step_done: one call per serving step.  *num_tokens / *num_reqs get the
 * step's token and row counts (0 for an empty step; either may be NULL).
 * Returns cb_schedule_step's status when that is not CB_OK (the step is
 * then neither submitted nor committed). */
cb_status cb_executor_run_step(cb_executor* ex, cb_sched* sched,
                               const void* const* q_host, const void* const* k_host,
                               const void* const* v_host, void* const* out_host,
                               int32_t* num_tokens, int32_t* num_reqs);

/* Wait until every queued copy and kernel has finished. */
cb_status cb_executor_synchronize(cb_executor* ex);

/* Steps and tokens submitted, and the compute stream's time spent on them
 * (CUDA events around each step's kernels; steps still running are not
 * counted yet).  Any output pointer may be NULL. */
cb_status cb_executor_stats(cb_executor* ex, int64_t* steps, int64_t* tokens,
                            double* compute_ms);
cb_status cb_executor_reset_stats(cb_executor* ex);

/* Synchronize, then read and clear the device error bits of the executor's
 * appends and attention calls; CB_ERR_DEVICE_CHECK if any was set. */
cb_status cb_executor_read_errors(cb_executor* ex, uint32_t* bits);

/* ------------------------------------------------------------------------
 * cb_paged_decode_noalloc (GPU).  No counterpart in the pages: an extra
 * entry point for callers that cannot allocate device memory.
 *
 * Some callers cannot call cudaMalloc at the point where they run attention:
 * code embedded in a host framework that owns the whole device-memory
 * budget and forbids side allocations while it executes (a serving-engine
 * plugin called from the framework's enqueue path, for instance), or a
 * latency-critical loop that cannot afford cudaMalloc's implicit device
 * synchronisation.  This call runs the same split-KV decode kernel as
 * cb_paged_attention but takes no workspace: its scratch (split partials,
 * split counters, work counters) lives in a fixed array of
 * CB_NOALLOC_SCRATCH_BYTES
 * inside this library, which every GPU that loads the library keeps until
 * the process exits.  It allocates nothing and calls no allocating routine.
 *
 *   args        as for cb_paged_attention, but EVERY row must be a decode
 *               (num_decodes == num_reqs == num_tokens, at most 1024 rows);
 *               args->workspace and args->workspace_bytes are ignored.
 *   error_word  optional device uint32 that receives CB_DEVERR_* bits
 *               (NULL: device-side errors are not reported).
 *   stream      the stream to run on.
 *
 * Limits: the call needs at least 2 * num_reqs * num_q_heads *
 * (head_dim + 2) * 4 bytes of split partials in CB_NOALLOC_SCRATCH_BYTES
 * (more room lets it cut the caches into more, smaller splits); larger
 * calls are rejected with CB_ERR_INVALID_ARG and a message giving the sizes.
 * Set-up: the first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current.  With CUDA's default
 * lazy module loading, the library's module -- and with it the 64 MiB
 * array -- is put on a device when the module is first needed there, at
 * the latest by that first call: a caller that cannot allocate later makes
 * the first call at set-up time, and before any stream capture.
 * Every call clears the counters it needs, then uses the array;
 * all calls in the process share it, so calls that may overlap on the GPU
 * (different streams without ordering between them) race with each other.
 * ---------------------------------------------------------------------- */
#define CB_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

cb_status cb_paged_decode_noalloc(const cb_attention_args* args, uint32_t* error_word,
                                  cb_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* CB_H_ */
