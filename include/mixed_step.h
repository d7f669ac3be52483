/*
 * mixed_step.h -- C ABI of the GB300 (sm_103a) mixed-batch attention step.
 *
 * One forward step of an attention layer over a paged KV cache, for a batch
 * that packs single-token decodes next to prefill chunks under a token budget
 * (chunked prefill with stall-free, decode-first batching).  Three calls make
 * the step:
 *
 *   ms_build_batch_metadata  host: decode-first token-budget packing and the
 *                            varlen metadata of the packed rows;
 *   ms_kv_append_rope        device: rotary embedding at absolute positions
 *                            for q and k, and the paged append of k and v;
 *   ms_mixed_step_attention  device: causal attention of every packed row
 *                            over its cached prefix plus its own new tokens.
 *
 * Sources, cited by page title and section:
 *   [zwj] "Chunked Prefill 的 Token 预算" (zwjcode.cn)
 *   [sar] "Chunked Prefill: Ending the Great Stall" (manishklach.github.io)
 *   [mer] "Splitting Prefill From Decode Inside a Step" (mercemay.com)
 *   [sfe] "Prefill head-of-line blocking" (sference.com)
 *
 * Conventions for every call:
 *   - All integers are int32 unless stated.  bf16 tensors are raw 16-bit
 *     storage (void*).  Pointers marked "device" must be device memory of the
 *     current CUDA device; "host" pointers are ordinary host memory.
 *   - The caller owns every buffer (metadata, tensors, K/V pools, workspace,
 *     stream).  The library allocates no memory and never synchronises, except
 *     in ms_read_status, which waits on the given stream.
 *   - Device calls only enqueue work on `stream`; they return MS_OK once the
 *     launches are queued.  Launch errors are returned as MS_ERR_CUDA.
 *   - Page size is 16 tokens.  Head dim D is 64 or 128.  H_q % H_kv == 0.
 *   - Return value: MS_OK (0) or a negative MS_ERR_* code; on error nothing is
 *     enqueued and no output is written.
 */
#ifndef MIXED_STEP_H_
#define MIXED_STEP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MS_API __attribute__((visibility("default")))
#else
#define MS_API
#endif

/* CUDA stream handle (cudaStream_t); NULL is the legacy default stream. */
typedef struct CUstream_st* ms_stream_t;

enum {
  MS_OK = 0,
  MS_ERR_ARG = -1,       /* bad shape, size, capacity, alignment or null pointer */
  MS_ERR_BUDGET = -2,    /* more running decodes than the token budget ([zwj] section 05) */
  MS_ERR_NO_PAGES = -3,  /* a block table cannot address the scheduled tokens ([mer]) */
  MS_ERR_CUDA = -4,      /* a CUDA runtime/driver call failed */
  MS_ERR_DEVICE = -5,    /* a device-side check failed (see ms_read_status) */
  MS_ERR_SCRATCH = -6    /* the step needs more than the library's static scratch
                            (ms_mixed_step_attention_noalloc) */
};

/* Device status bits, accumulated in a caller-owned int32 status word. */
enum {
  MS_STATUS_BAD_SLOT = 1,      /* slot_mapping entry outside the page pool */
  MS_STATUS_BAD_POSITION = 2,  /* position outside the cos/sin table */
  MS_STATUS_BAD_PAGE = 4,      /* block_tables entry outside the page pool */
  MS_STATUS_TIMEOUT = 8,       /* a bounded in-kernel wait gave up */
  MS_STATUS_BAD_META = 16,     /* inconsistent row metadata (lengths, offsets) */
  MS_STATUS_INTERNAL = 32      /* an internal invariant failed (shared-memory alignment) */
};

/* One request as the scheduler sees it.
 *   cached_len        c, tokens already in the KV cache (absolute positions
 *                     0..c-1; positions are never reset, [zwj] section 07)
 *   remaining_prompt  0 for a running decode; > 0 prompt tokens still to prefill
 *   block_table       host, num_pages physical page ids in logical order,
 *                     reserved by the caller before the request's first chunk
 *                     ([mer] "The arithmetic of chunk boundaries") */
typedef struct {
  int32_t cached_len;
  int32_t remaining_prompt;
  const int32_t* block_table;
  int32_t num_pages;
} ms_request;

/* Priority orders of one round ([mer] "Choosing the priority order"). */
enum {
  MS_POLICY_DECODE_FIRST = 0,  /* every running decode, then prompts take the leftover (stall-free) */
  MS_POLICY_PREFILL_FIRST = 1, /* prompts take the budget first, decodes whatever remains */
  MS_POLICY_FAIR_SHARE = 2     /* decodes may use decode_share_permille of the budget, prompts the
                                  rest; what one class leaves unused goes to the other */
};

/* token_budget           B_tok, the most tokens one step may hold
 *                        ([zwj] section 04: |D_t| + sum |c| <= B_tok)
 * max_chunk_per_request  ceiling on one prompt's take per round; 0 = none
 *                        ([sfe] "The fix", [mer] build_batch's chunk_size)
 * policy                 MS_POLICY_*
 * min_chunk_per_request  floor: every waiting prompt first gets up to this many
 *                        tokens (arrival order), then the leftover is handed out
 *                        in arrival order; 0 = none ([sfe] "What comes next")
 * prefill_quota          decode-first only: while prompts wait, decodes use at
 *                        most budget - min(quota, what the prompts can take) and
 *                        the rest wait a round ([zwj] section 08: a reserved
 *                        prefill quota against starvation); 0 = none
 * decode_share_permille  fair share only: the decode class's share of the
 *                        budget, 0..1000 */
typedef struct {
  int32_t token_budget;
  int32_t max_chunk_per_request;
  int32_t policy;
  int32_t min_chunk_per_request;
  int32_t prefill_quota;
  int32_t decode_share_permille;
} ms_sched_config;

/* Summary of one packed step.  bt_stride is the row stride of block_tables;
 * num_deferred counts running decodes the policy left for a later round. */
typedef struct {
  int32_t num_rows;
  int32_t num_decodes;
  int32_t num_tokens;
  int32_t bt_stride;
  int32_t unused_tokens;
  int32_t num_deferred;
} ms_batch_info;

/* ms_build_batch_metadata -- pack one round, decode first ([zwj] sections
 * 03-05 and 08, [sar] sections 03-04), and emit its varlen metadata
 * ([zwj] section 06).  Host only; pure (reqs are not modified: the caller
 * commits progress after the step, [zwj] section 08).
 *
 * Packing (decode-first, no quota): every request with remaining_prompt == 0
 * is a decode row (c, 1), in input order; more decodes than token_budget is
 * MS_ERR_BUDGET.  Then, in input order, each prompt takes min(remaining,
 * leftover, cap) tokens as a chunk row (c, take); packing stops when the
 * leftover reaches 0.  The other policies and limits of ms_sched_config change
 * how the budget is split; rows are always the scheduled decodes in input
 * order, then the chunks in input order.
 *
 * Outputs (host, caller-allocated, capacities in elements):
 *   cu_seqlens_q  [cap_rows + 1]  row token offsets, cu[0] = 0
 *   q_start_pos   [cap_rows]      c of each row
 *   context_lens  [cap_rows]      c + d, the row's length after the step
 *   positions     [cap_tokens]    absolute position c + j of each new token
 *   slot_mapping  [cap_tokens]    block_table[pos / 16] * 16 + pos % 16
 *   block_tables  [cap_bt]        rows x bt_stride page ids, padded with -1;
 *                                 bt_stride = max over rows of ceil((c+d)/16)
 *   row_req       [cap_rows]      request index of each row
 *   num_scheduled [n_req]         tokens each request got this round (0 or d)
 *   info          summary (num_rows, num_decodes, num_tokens, bt_stride, unused)
 * Errors: MS_ERR_ARG (null pointer, capacity too small, negative lengths, a
 * page id that a scheduled row reads below 0 or above INT32_MAX / 16 - 1),
 * MS_ERR_BUDGET, MS_ERR_NO_PAGES (a block table shorter than ceil((c+d)/16)). */
MS_API int ms_build_batch_metadata(const ms_request* reqs, int32_t n_req, const ms_sched_config* cfg,
                                   int32_t cap_rows, int32_t cap_tokens, int64_t cap_bt,
                                   int32_t* cu_seqlens_q, int32_t* q_start_pos, int32_t* context_lens,
                                   int32_t* positions, int32_t* slot_mapping, int32_t* block_tables,
                                   int32_t* row_req, int32_t* num_scheduled, ms_batch_info* info);

/* ms_build_batch_metadata_ragged -- the same packing and metadata as
 * ms_build_batch_metadata, with the block table in its ragged form: row s
 * holds exactly the ceil((c+d)/16) pages it reads ([zwj] section 06 gives a
 * row ceil((c+d)/B) entries), at bt_pages[bt_offsets[s] .. bt_offsets[s+1]).
 * The padded form costs rows x (longest row's pages) entries; in a step that
 * mixes a few 64K-128K-token decodes with hundreds of short ones that is over
 * ten times the pages in use, built on the host and copied to the device every
 * step.
 *   bt_offsets [cap_rows + 1]  host int32, bt_offsets[0] = 0, bt_offsets[S] = pages
 *   bt_pages   [cap_pages]     host int32 page ids, row after row
 * The other outputs, info (bt_stride is still the longest row's page count)
 * and the errors are those of ms_build_batch_metadata; MS_ERR_ARG also when
 * the pages exceed cap_pages. */
MS_API int ms_build_batch_metadata_ragged(const ms_request* reqs, int32_t n_req, const ms_sched_config* cfg,
                                          int32_t cap_rows, int32_t cap_tokens, int64_t cap_pages,
                                          int32_t* cu_seqlens_q, int32_t* q_start_pos, int32_t* context_lens,
                                          int32_t* positions, int32_t* slot_mapping, int32_t* bt_offsets,
                                          int32_t* bt_pages, int32_t* row_req, int32_t* num_scheduled,
                                          ms_batch_info* info);

/* ms_rope_table -- host: cos/sin of p * base^(-2i/D) for p < max_pos, i < D/2,
 * computed in double precision and rounded to fp32.  Output layout
 * [max_pos][D/2] row-major, caller-allocated host buffers.  The rotary phase
 * is taken at the absolute position ([zwj] section 07).
 * Errors: MS_ERR_ARG (null pointer, max_pos < 1, D odd or < 2, base <= 0). */
MS_API int ms_rope_table(int32_t max_pos, int32_t D, double base, float* cos_tab, float* sin_tab);

/* ms_kv_append_rope -- device: for every new token t at p = positions[t],
 * rotate q[t] and k[t] with the rotate-half pairing (element i with i + D/2):
 *     y_i       = x_i * cos - x_{i+D/2} * sin
 *     y_{i+D/2} = x_{i+D/2} * cos + x_i * sin
 * each as two fp32 products and one fp32 sum, rounded to nearest, never fused,
 * then rounded to bf16 (nearest even); write q_rot[t], and rotated k[t] and
 * raw v[t] into the paged pools at slot_mapping[t] ([zwj] section 06; slot -1
 * means no write).
 *   q      device bf16 [T, H_q, D];   q_rot device bf16 [T, H_q, D] (may alias q)
 *   k, v   device bf16 [T, H_kv, D]
 *   positions, slot_mapping  device int32 [T]
 *   cos_tab, sin_tab         device fp32 [max_pos, D/2] (ms_rope_table)
 *   k_cache, v_cache         device bf16 [num_pages, H_kv, 16, D]
 *   dev_status               device int32 status word or NULL.  Slot -1 is
 *                            the one "no write" value; any other negative
 *                            slot, or one past the pool, writes nothing and
 *                            sets MS_STATUS_BAD_SLOT.  A token whose position
 *                            lies outside the table writes nothing at all
 *                            (no q_rot row, no K, no V) and sets
 *                            MS_STATUS_BAD_POSITION.  Bits are recorded only
 *                            when dev_status is given.
 * All tensor pointers 16-byte aligned.  T == 0 is a no-op.
 * Errors: MS_ERR_ARG, MS_ERR_CUDA. */
MS_API int ms_kv_append_rope(const void* q, const void* k, const void* v,
                             const int32_t* positions, const int32_t* slot_mapping, int32_t T,
                             const float* cos_tab, const float* sin_tab, int32_t max_pos,
                             void* k_cache, void* v_cache, int32_t num_pages, void* q_rot,
                             int32_t H_q, int32_t H_kv, int32_t D, int32_t page_size,
                             int32_t* dev_status, ms_stream_t stream);

/* ms_attention_workspace_size -- bytes of device workspace that
 * ms_mixed_step_attention needs for steps of at most max_rows rows,
 * max_tokens new tokens and max_context_total = sum over rows of context_lens.
 * The first 256 bytes of a workspace hold its header, 64 int32 words: word 0
 * the status word, then queue counters and the step's plan (word 9: how many
 * CTAs started on chunk work) and, kept across calls, word 10: the SM clock
 * in MHz the last call measured, which the next call's SM-split cost model
 * uses.  Zero the whole workspace once before its first use. */
MS_API size_t ms_attention_workspace_size(int32_t max_rows, int32_t max_tokens, int64_t max_context_total,
                                          int32_t H_q, int32_t H_kv, int32_t D);

/* ms_mixed_step_attention -- device: for every packed token t of row s
 * (absolute position p = q_start_pos[s] + t - cu_seqlens_q[s]) and query head h
 * (KV head h / (H_q / H_kv)):
 *     out[t, h] = softmax_j(scale * q_rot[t, h] . K[j]) V[j],   j = 0..p
 * with K/V row j read from page block_tables[s * bt_stride + j / 16], slot
 * j % 16.  A chunk [c, c+d) sees the cached prefix [0, c) plus its own tokens
 * causally ([zwj] sections 02 and 07; [sar] section 05).  Rows with d == 1 run
 * the split-KV decode path; rows with d > 1 run the tensor-core chunk path; a
 * persistent queue orders the work longest-first.  A row with d == 0
 * (cu_seqlens_q[s + 1] == cu_seqlens_q[s], context_lens[s] == q_start_pos[s])
 * is a pad row and computes nothing; tokens no row covers are left unwritten
 * (the padding of a fixed-shape step, [sar] section 05).  bf16 in, fp32 accumulate,
 * bf16 out.
 *   q_rot        device bf16 [num_tokens, H_q, D]
 *   k_cache, v_cache  device bf16 [num_pages, H_kv, 16, D], num_pages pages
 *   cu_seqlens_q [num_rows + 1], q_start_pos [num_rows], context_lens [num_rows],
 *   block_tables [num_rows * bt_stride]   device int32, as built by
 *                ms_build_batch_metadata (context_lens[s] must equal
 *                q_start_pos[s] + d_s)
 *   out          device bf16 [num_tokens, H_q, D]
 *   workspace    device, ws_bytes >= ms_attention_workspace_size(...) for
 *                this step's sizes, zeroed before first use; its first int32 is
 *                the status word (read it with ms_read_status)
 * Out-of-range page ids are not read (MS_STATUS_BAD_PAGE).  A step holds at
 * most 8192 rows and 2^21 tokens.  Steps that share a workspace must not
 * overlap on the GPU.
 * Errors: MS_ERR_ARG, MS_ERR_CUDA. */
MS_API int ms_mixed_step_attention(const void* q_rot, const void* k_cache, const void* v_cache,
                                   int32_t num_pages,
                                   const int32_t* cu_seqlens_q, const int32_t* q_start_pos,
                                   const int32_t* context_lens, const int32_t* block_tables,
                                   int32_t bt_stride, int32_t num_rows, int32_t num_tokens,
                                   int64_t context_total,
                                   int32_t H_q, int32_t H_kv, int32_t D, int32_t page_size, float scale,
                                   void* out, void* workspace, size_t ws_bytes, ms_stream_t stream);

/* ms_mixed_step_attention_ragged -- ms_mixed_step_attention with the block
 * table in the ragged form of ms_build_batch_metadata_ragged: row s reads its
 * pages from bt_pages[bt_offsets[s] ..], and bt_offsets[s + 1] - bt_offsets[s]
 * must be at least ceil(context_lens[s] / 16).
 *   bt_offsets   device int32 [num_rows + 1]
 *   bt_pages     device int32 [num_bt_pages]
 * A row whose pages fall outside bt_pages, or has fewer than it needs, makes
 * the step compute nothing and sets MS_STATUS_BAD_META.  Everything else
 * (layouts, workspace, status, errors) is as ms_mixed_step_attention. */
MS_API int ms_mixed_step_attention_ragged(const void* q_rot, const void* k_cache, const void* v_cache,
                                          int32_t num_pages,
                                          const int32_t* cu_seqlens_q, const int32_t* q_start_pos,
                                          const int32_t* context_lens, const int32_t* bt_offsets,
                                          const int32_t* bt_pages, int64_t num_bt_pages,
                                          int32_t num_rows, int32_t num_tokens, int64_t context_total,
                                          int32_t H_q, int32_t H_kv, int32_t D, int32_t page_size, float scale,
                                          void* out, void* workspace, size_t ws_bytes, ms_stream_t stream);

/* ms_mixed_step -- one step of one attention layer: ms_kv_append_rope of the
 * step's num_tokens new tokens, then the attention of ms_mixed_step_attention
 * (block_tables padded with bt_stride, bt_offsets == NULL) or of
 * ms_mixed_step_attention_ragged (block_tables = bt_pages with bt_len entries,
 * bt_offsets given), in that order on `stream`, with the same arguments,
 * layouts, status words and errors as those calls.  Decodes and prompt
 * chunks share one forward pass ([sar] sections 02-04), so a step calls this
 * once per attention layer over the whole packed batch.  T of the
 * append is num_tokens.  On steps of at most 1024 rows the append and the
 * attention's prologue share one launch (two kernels per step instead of
 * three); results are bit-identical to the two separate calls.  Every
 * argument of both parts is checked before the first enqueue.
 * Errors: MS_ERR_ARG, MS_ERR_CUDA. */
MS_API int ms_mixed_step(const void* q, const void* k, const void* v, const int32_t* positions,
                         const int32_t* slot_mapping, const float* cos_tab, const float* sin_tab, int32_t max_pos,
                         void* k_cache, void* v_cache, int32_t num_pages, void* q_rot,
                         const int32_t* cu_seqlens_q, const int32_t* q_start_pos, const int32_t* context_lens,
                         const int32_t* block_tables, const int32_t* bt_offsets, int64_t bt_len, int32_t bt_stride,
                         int32_t num_rows, int32_t num_tokens, int64_t context_total,
                         int32_t H_q, int32_t H_kv, int32_t D, int32_t page_size, float scale,
                         void* out, void* workspace, size_t ws_bytes, int32_t* dev_status, ms_stream_t stream);

/* ms_mixed_step_attention_noalloc -- the same attention step as
 * ms_mixed_step_attention, for callers that cannot give the library a
 * workspace.  A serving process that reserves nearly all device memory for
 * its KV-cache pool at start-up has no room for another allocation, and host
 * code on a per-step path should not call cudaMalloc (it may synchronise the
 * device and stall other streams).  This call allocates nothing: no
 * cudaMalloc, cudaFree or allocating library routine.  It works out of a
 * scratch array the library owns, 64 MiB per device (the step's workspace
 * size, ms_attention_workspace_size(num_rows, num_tokens, context_total, H_q,
 * H_kv, D), must not exceed it -- else MS_ERR_SCRATCH and nothing is
 * enqueued).  The array is device memory that every GPU which loads this
 * library holds until the process exits.
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  All calls share the one array per device and it keeps the last
 * call's contents: each call's first kernel clears the status word and the
 * work counters before anything of the call can set them, so calls that
 * overlap on the GPU (other streams, other host threads) race and must be
 * serialised by the caller.  All argument checks come before anything is
 * enqueued: a call that returns an error has put nothing on the stream.
 *
 * Arguments are those of ms_mixed_step_attention without the workspace, plus
 * dev_status: device int32 or NULL; when given, it is overwritten on `stream`
 * with this call's device status bits (MS_STATUS_*) after the kernels.
 * The pages have no counterpart of this call: it only changes where the
 * scratch lives.
 * Errors: MS_ERR_ARG, MS_ERR_SCRATCH, MS_ERR_CUDA. */
MS_API int ms_mixed_step_attention_noalloc(const void* q_rot, const void* k_cache, const void* v_cache,
                                           int32_t num_pages,
                                           const int32_t* cu_seqlens_q, const int32_t* q_start_pos,
                                           const int32_t* context_lens, const int32_t* block_tables,
                                           int32_t bt_stride, int32_t num_rows, int32_t num_tokens,
                                           int64_t context_total, int32_t H_q, int32_t H_kv, int32_t D,
                                           int32_t page_size, float scale, void* out, int32_t* dev_status,
                                           ms_stream_t stream);

/* ms_test_attention_stall -- test hook for the bounded device waits, not for
 * production use.  It enqueues ms_mixed_step_attention exactly as that call
 * would, except that the producer warp of every CTA's chunk phase publishes no
 * work item and issues no copy, as a producer that had stopped would, and
 * every chunk-phase wait gives up after wait_limit_ns (instead of 2 s).  The
 * other roles of each CTA then wait for an item that never comes: the first
 * wait that runs out sets MS_STATUS_TIMEOUT in the workspace's status word,
 * the CTA unwinds (nothing is in flight), frees its tensor memory and
 * returns.  The chunk rows' outputs are left unwritten.  The workspace stays
 * usable: the next ms_mixed_step_attention on it computes the step normally.
 * It checks the library's own failure detection (the pages have no
 * counterpart) and faults nothing.  Arguments as ms_mixed_step_attention,
 * plus wait_limit_ns in
 * [100000, 2000000000].
 * Errors: MS_ERR_ARG, MS_ERR_CUDA. */
MS_API int ms_test_attention_stall(const void* q_rot, const void* k_cache, const void* v_cache,
                                   int32_t num_pages,
                                   const int32_t* cu_seqlens_q, const int32_t* q_start_pos,
                                   const int32_t* context_lens, const int32_t* block_tables,
                                   int32_t bt_stride, int32_t num_rows, int32_t num_tokens,
                                   int64_t context_total,
                                   int32_t H_q, int32_t H_kv, int32_t D, int32_t page_size, float scale,
                                   void* out, void* workspace, size_t ws_bytes, int64_t wait_limit_ns,
                                   ms_stream_t stream);

/* ms_test_attention_split -- test hook: ms_mixed_step_attention (bt_offsets ==
 * NULL, block_tables padded with bt_stride) or ms_mixed_step_attention_ragged
 * (bt_offsets given, block_tables = bt_pages with bt_len entries) with the
 * starting split of the SMs forced: chunk_ctas CTAs (clamped to the SM count)
 * start on chunk work, the others on decode items.  CTAs still move to the
 * other queue when their own runs dry, so the outputs equal the ordinary
 * call's; only the timing changes.  The pages have no counterpart: the hook
 * lets a test sweep the split against the cost model's choice (workspace
 * header word 9).  Errors: MS_ERR_ARG (also for chunk_ctas < 0), MS_ERR_CUDA. */
MS_API int ms_test_attention_split(const void* q_rot, const void* k_cache, const void* v_cache, int32_t num_pages,
                                   const int32_t* cu_seqlens_q, const int32_t* q_start_pos,
                                   const int32_t* context_lens, const int32_t* block_tables,
                                   const int32_t* bt_offsets, int64_t bt_len, int32_t bt_stride, int32_t num_rows,
                                   int32_t num_tokens, int64_t context_total, int32_t H_q, int32_t H_kv, int32_t D,
                                   int32_t page_size, float scale, void* out, void* workspace, size_t ws_bytes,
                                   int32_t chunk_ctas, ms_stream_t stream);

/* ---- Multi-round engine (host) ------------------------------------------
 * A page pool with full-input admission and a plan/commit round driver over
 * ms_build_batch_metadata.  A request reserves ceil((prompt_len +
 * max_new_tokens) / 16) pages when it is admitted, before its first chunk, or
 * is refused ([mer] "The arithmetic of chunk boundaries"; [zwj] section 11,
 * admission against the complete input length).  Each round is plan (pack the
 * live requests in arrival order), the caller's device step, then commit
 * ([zwj] section 08: progress is committed after the step).  The last prompt
 * chunk yields a request's first new token, each decode one more; a request
 * with max_new_tokens tokens is finished and its pages go back to the pool.
 * Pages are handed out last-in-first-out from a free list that starts as
 * num_pages-1 .. 0 (so the first request gets 0, 1, 2, ...); a finished
 * request returns its pages in block-table order.  Not thread-safe: one
 * engine per host thread. */
typedef struct ms_engine ms_engine;

typedef struct {
  int32_t num_live;        /* admitted and not finished */
  int32_t num_prefilling;  /* live requests with prompt tokens left */
  int32_t num_free_pages;
  int32_t num_pages;
  int32_t max_request_pages; /* largest block table of a live request (sizes plan's cap_bt) */
  int64_t rounds;          /* committed rounds */
} ms_engine_counts;

/* ms_engine_create -- a pool of num_pages pages and a copy of *cfg (the
 * packing of every round).  *out owns the engine until ms_engine_destroy.
 * Errors: MS_ERR_ARG (null pointer, num_pages < 0, out of host memory). */
MS_API int ms_engine_create(int32_t num_pages, const ms_sched_config* cfg, ms_engine** out);

/* ms_engine_destroy -- frees the engine (NULL is a no-op). */
MS_API int ms_engine_destroy(ms_engine* e);

/* ms_engine_add_request -- admit a prompt of prompt_len tokens, cached_len of
 * them already in the cache ([sar] section 05: only the rest is prefilled),
 * that will generate max_new_tokens tokens; *request_id gets its id (0, 1, ...
 * in admission order).  A fully cached prompt is a running decode that has
 * its first new token, so it must ask for at least two.
 * Errors: MS_ERR_ARG (prompt_len < 1, max_new_tokens < 1, cached_len outside
 * 0..prompt_len, the fully cached case with max_new_tokens < 2),
 * MS_ERR_NO_PAGES (refused: not enough free pages; nothing changes). */
MS_API int ms_engine_add_request(ms_engine* e, int32_t prompt_len, int32_t max_new_tokens, int32_t cached_len,
                                 int32_t* request_id);

/* ms_engine_request_pages -- the block table of a live request: *num_pages
 * and, when cap allows, the page ids in logical order into pages (host).
 * Errors: MS_ERR_ARG (unknown id, cap too small, null pointer). */
MS_API int ms_engine_request_pages(const ms_engine* e, int32_t request_id, int32_t* pages, int32_t cap,
                                   int32_t* num_pages);

/* ms_engine_plan -- pack the next round over the live requests and write its
 * metadata exactly as ms_build_batch_metadata does (same outputs, capacities
 * and errors), with row_request_id [cap_rows] holding each row's request id
 * instead of its index.  Planning again before commit replaces the plan. */
MS_API int ms_engine_plan(ms_engine* e, int32_t cap_rows, int32_t cap_tokens, int64_t cap_bt,
                          int32_t* cu_seqlens_q, int32_t* q_start_pos, int32_t* context_lens,
                          int32_t* positions, int32_t* slot_mapping, int32_t* block_tables,
                          int32_t* row_request_id, ms_batch_info* info);

/* ms_engine_commit -- advance every row of the last plan (a decode by one
 * token, a chunk by its length), release finished requests and write their
 * ids, in arrival order, to finished_ids [cap_finished] (host).
 * Errors: MS_ERR_ARG (no plan since the last commit, cap_finished smaller
 * than the number finishing; nothing changes). */
MS_API int ms_engine_commit(ms_engine* e, int32_t* finished_ids, int32_t cap_finished, int32_t* num_finished);

/* ms_engine_stats -- counts of the pool and the live requests. */
MS_API int ms_engine_stats(const ms_engine* e, ms_engine_counts* out);

/* ---- CUDA-graph replay with padded token buckets (device) -----------------
 * A CUDA graph records fixed shapes while chunked prefill changes the token
 * count every step; the engine captures one graph per token bucket and pads
 * each step up to the next bucket ([sar] section 05).  One graph records
 * ms_kv_append_rope + ms_mixed_step_attention at the bucket's token count,
 * max_rows rows, block-table stride max_row_pages and context bound
 * num_pages * 16.  A replay pads the step: tokens past num_tokens get slot -1
 * (no cache write) and position 0, rows past num_rows get d = 0 (pad rows).
 * The pad tokens still pass through the append (their q_rot rows are junk);
 * the attention output of real tokens equals the unpadded call's. */
typedef struct ms_step_graph ms_step_graph;

/* H_q, H_kv, D, num_pages  as for ms_mixed_step_attention
 * max_rows       rows any replayed step may hold (<= 8192)
 * max_row_pages  block-table stride of every replay (the longest row's pages)
 * max_pos        rows of the cos/sin tables
 * scale          softmax scale
 * buckets        host, num_buckets ascending token counts, one graph each */
typedef struct {
  int32_t H_q, H_kv, D;
  int32_t num_pages;
  int32_t max_rows;
  int32_t max_row_pages;
  int32_t max_pos;
  float scale;
  int32_t num_buckets;
  const int32_t* buckets;
} ms_graph_config;

/* Device buffers the graphs are recorded on (caller-owned, fixed for the
 * graph's life).  q [B, H_q, D], k and v [B, H_kv, D], q_rot and out
 * [B, H_q, D] (bf16, B = the largest bucket): the caller writes each step's
 * new tokens into rows 0..num_tokens-1 of q, k, v before ms_graph_run.
 * cos_tab/sin_tab fp32 [max_pos][D/2]; k_cache/v_cache the page pools;
 * workspace 256-byte aligned, ws_bytes >= ms_graph_workspace_size (it holds
 * the fixed metadata buffers and the attention workspace); dev_status device
 * int32 or NULL (the append's status bits). */
typedef struct {
  const void* q;
  const void* k;
  const void* v;
  const float* cos_tab;
  const float* sin_tab;
  void* k_cache;
  void* v_cache;
  void* q_rot;
  void* out;
  void* workspace;
  size_t ws_bytes;
  int32_t* dev_status;
} ms_graph_buffers;

/* ms_graph_workspace_size -- bytes of workspace for this config, 0 if the
 * config is invalid. */
MS_API size_t ms_graph_workspace_size(const ms_graph_config* cfg);

/* ms_graph_create -- clear the workspace to an all-pad step, run each bucket's
 * step once on `stream` (one-time kernel setup) and capture it into a graph.
 * Call it outside any stream capture, on a stream other than the legacy
 * default stream (NULL), which cannot be captured.  Unlike the other device
 * calls it allocates: two pinned host staging buffers (cudaHostAlloc) and the
 * instantiated graphs, all released by ms_graph_destroy.
 * Errors: MS_ERR_ARG (bad config, NULL stream, workspace too small or
 * misaligned), MS_ERR_CUDA. */
MS_API int ms_graph_create(const ms_graph_config* cfg, const ms_graph_buffers* bufs, ms_stream_t stream,
                           ms_step_graph** out);

/* ms_graph_destroy -- waits for pending metadata copies, frees the graphs and
 * the staging buffers (NULL is a no-op). */
MS_API int ms_graph_destroy(ms_step_graph* g);

/* ms_graph_bucket -- the bucket a step of num_tokens tokens runs in, or
 * MS_ERR_ARG when it exceeds the largest bucket. */
MS_API int ms_graph_bucket(const ms_step_graph* g, int32_t num_tokens);

/* ms_graph_run -- one step: pad the host metadata (as ms_build_batch_metadata
 * writes it) into the pinned staging buffer, copy it into the fixed device
 * buffers on `stream` and launch the bucket's graph.  The host waits only for
 * the copies of the replay before last (the staging buffers alternate).
 * Every replay of one graph rewrites the same device metadata buffers, so
 * the caller issues them on one stream (or orders the streams itself): a
 * replay's copies must not start while the previous replay still runs.
 * *bucket_used (may be NULL) gets the bucket.  Device errors land in the
 * status words (ms_graph_read_status).
 * Errors: MS_ERR_ARG (num_tokens above the largest bucket, num_rows >
 * max_rows, bt_stride > max_row_pages, cu_seqlens_q inconsistent with
 * num_tokens, null pointers), MS_ERR_CUDA. */
MS_API int ms_graph_run(ms_step_graph* g, const int32_t* cu_seqlens_q, const int32_t* q_start_pos,
                        const int32_t* context_lens, const int32_t* positions, const int32_t* slot_mapping,
                        const int32_t* block_tables, int32_t bt_stride, int32_t num_rows, int32_t num_tokens,
                        ms_stream_t stream, int32_t* bucket_used);

/* ms_graph_read_status -- waits for `stream`, ORs and clears the append and
 * attention status words of the graph's buffers into *host_status.  Returns
 * MS_OK, MS_ERR_DEVICE when a bit was set, or MS_ERR_ARG / MS_ERR_CUDA. */
MS_API int ms_graph_read_status(ms_step_graph* g, ms_stream_t stream, int32_t* host_status);

/* ms_read_status -- waits for `stream`, copies the int32 device status word at
 * dev_status (for attention: the workspace pointer) to *host_status and
 * clears it.  Returns MS_OK, MS_ERR_DEVICE when the word was non-zero, or
 * MS_ERR_ARG / MS_ERR_CUDA. */
MS_API int ms_read_status(int32_t* dev_status, ms_stream_t stream, int32_t* host_status);

/* ms_cost_model_rates -- host: the current device's rates behind the SM
 * split of the attention call, before any call has measured the SM clock:
 * the rated SM clock in MHz, and the HBM bandwidth in GB/s taken as the
 * nominal rate (memory clock x bus width, double data rate) times 0.80, the
 * sustained share a device-to-device copy reaches.
 * Errors: MS_ERR_ARG (NULL output), MS_ERR_CUDA. */
MS_API int ms_cost_model_rates(float* sm_mhz, float* hbm_gbs);

/* ms_num_sms -- SM count of the current device (the persistent grid size), or
 * a negative MS_ERR_* code. */
MS_API int ms_num_sms(void);

#ifdef __cplusplus
}
#endif

#endif /* MIXED_STEP_H_ */
