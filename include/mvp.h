/*
 * mvp.h -- masked varlen prefill attention for GB300 (sm_103a), C ABI.
 *
 * Two operations, as described by the vLLM pages this library restates:
 *
 *   mvp_fill_query_ranges  -- vLLM PR #50294 review ("FA4 mm_prefix range
 *       scan -> O(1) table lookup"), "Implementation breakdown" step 1 and the
 *       fill_mm_prefix_query_ranges listing: per packed query row, the closed
 *       [start, end] of the bidirectional range holding that row's absolute
 *       position, or (-1, -1).
 *   mvp_attn_fwd_varlen    -- the forward pass of variable-length MHA/GQA
 *       softmax attention under serving masks: causal with a chunked-prefill
 *       context offset (step14_4 "Causal Mask optimisation" tutorial, key j is
 *       masked iff j > start_pos + i), sliding windows (PR #50294 mask_mod and
 *       forward() wiring; PR #49815 symmetric window), the range table OR-ed in
 *       (PR #50294 mask_mod), and per-head sinks in two modes (PR #49815
 *       "_fwd_kernel sinks branch": key-0 bias or null logit).
 *
 * Conventions shared by every entry point:
 *   - Pointers are DEVICE pointers unless a parameter says otherwise.  The
 *     caller owns every buffer; the library never frees caller memory.
 *   - Work is enqueued on `stream` (a cudaStream_t, NULL = legacy default
 *     stream) and the call returns without synchronising.
 *   - Argument errors are detected on the host before anything is launched;
 *     nothing is written then.  Return values are mvp_status codes.
 *   - The library keeps one 4-byte device error word per device: a
 *     __device__ variable of the library's own module, so nothing is
 *     allocated for it; its device address is looked up on the first call on
 *     that device.  Kernels that hit a bounded-wait timeout record a code
 *     there and unwind instead of hanging (so does a prefill kernel whose
 *     workspace queue another launch took over); mvp_get_last_device_error()
 *     reads and clears it.
 *   - Per-device state (that address, the SM count, kernel attributes, a
 *     second stream and two events for mixed batches) is set up on the first
 *     attention call on a device -- make that call before any stream
 *     capture -- and kept for the life of the process; a cudaDeviceReset()
 *     invalidates it, so the library must not be used on a device after a
 *     reset.
 */
#ifndef MVP_H_
#define MVP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MVP_OK = 0,
  MVP_ERR_ARG = -1,          /* null pointer, bad size, inconsistent shape      */
  MVP_ERR_CAPACITY = -2,     /* out_capacity < num_tokens (the page asserts)    */
  MVP_ERR_UNSUPPORTED = -3,  /* head_dim / head ratio / alignment not supported */
  MVP_ERR_CUDA = -4,         /* a CUDA runtime call or launch failed            */
  MVP_ERR_DEVICE_TIMEOUT = -5, /* a kernel recorded a bounded-wait timeout (or a
                                  work queue shared by overlapping calls)    */
  MVP_ERR_DEVICE_BOUNDS = -6   /* bounds-checked build (libmvp_debug.so) only: a
                                  kernel found an index derived from the
                                  caller's offsets, range table or block table
                                  outside its buffer and skipped the access   */
} mvp_status;

typedef enum {
  MVP_SINK_NONE = 0,
  MVP_SINK_KEY0_BIAS = 1,  /* s[i,0] += sink[h] when key 0 is visible (MiMo)       */
  MVP_SINK_NULL_LOGIT = 2  /* exp(sink[h]) joins the denominator only (GPT-OSS)   */
} mvp_sink_mode;

/*
 * Range table fill.  Source: vLLM PR #50294 review, "Key source snippets",
 * fill_mm_prefix_query_ranges, and "Implementation breakdown" step 1.
 *
 * ranges          int32 [num_reqs, max_ranges, 2], row-major.  Absolute closed
 *                 (start, end) token positions of each request's
 *                 bidirectional ranges; entries with start >= end are
 *                 degenerate and skipped (use (0, 0) for padding).  Within a
 *                 request, valid ranges must not overlap; if they do, the
 *                 last listed range that holds a query position wins.
 * query_start_loc int32 [num_reqs + 1], packed query row offsets (ascending,
 *                 query_start_loc[0] == 0, query_start_loc[num_reqs] ==
 *                 num_tokens).
 * seq_lens        int32 [num_reqs], total key length of each request; the
 *                 request's first scheduled query sits at absolute position
 *                 seq_lens[b] - (query_start_loc[b+1] - query_start_loc[b]).
 * num_tokens      host int, normally query_start_loc[num_reqs] (the caller
 *                 knows it on the host, as the page's builder does); rows at
 *                 or past query_start_loc[num_reqs] (a batch padded to a
 *                 fixed capacity) are written as (-1, -1).
 * out             int32 [out_capacity, 2]: rows [0, num_tokens) are ALL
 *                 written: (start, end) of the range holding the row's
 *                 absolute position, clipped to nothing (the range itself is
 *                 stored unclipped), or (-1, -1).  Rows >= num_tokens are
 *                 not touched.
 * rows_written    int32 device scalar or NULL: set to num_tokens if at least
 *                 one row got a range, else 0 (the page's return value; 0
 *                 means the attention call may skip the range test).
 * Errors: MVP_ERR_ARG (null pointer with num_tokens > 0, negative sizes),
 *         MVP_ERR_CAPACITY (out_capacity < num_tokens), MVP_ERR_CUDA.
 * num_tokens == 0: nothing is launched except the rows_written reset.
 */
int mvp_fill_query_ranges(const int32_t* ranges, int num_reqs, int max_ranges,
                          const int32_t* query_start_loc, const int32_t* seq_lens,
                          int num_tokens, int32_t* out, int out_capacity,
                          int32_t* rows_written, void* stream);

/*
 * Bytes of caller-provided workspace that mvp_attn_fwd_varlen can use.  The
 * first 256 bytes hold the prefill kernel's work queue: its persistent CTAs
 * walk the work items with a static stride but claim the last round one at a
 * time from the queue (whichever CTA frees up first takes the next item),
 * which evens out the end of batches whose items differ in length (batches
 * of fewer than two rounds, and masks with a window shorter than max_k_len,
 * whose items are even already, keep the stride).  The rest holds partial results that let long
 * single-token (decode) rows be split across several CTAs.  num_reqs is the
 * number of requests the decode kernel covers (num_decode_reqs, or the whole
 * batch when that is -1; 0: header only).  Returns 0 for negative num_reqs
 * or non-positive sizes.
 * The workspace needs no initialisation and is left valid for the next call
 * (the queue words carry a per-launch tag, and each launch resets its
 * counter when its last CTA is done).  Two calls
 * that may run at the same time on the GPU (different streams) need separate
 * workspaces; a kernel that finds its queue taken over records a device
 * error (mvp_get_last_device_error) and stops claiming.  Workspace is
 * optional: without it (NULL, fewer than 256 bytes, or not 16-byte aligned)
 * the prefill items are walked with a static stride and every decode row is
 * handled by one CTA per KV head.
 */
size_t mvp_attn_workspace_size(int num_reqs, int num_heads_q, int head_dim, int max_k_len);

/*
 * Masked varlen attention forward.  The visible set of query row i of request
 * b (absolute position p = ctx_b + i, ctx_b = context_lens[b] or
 * k_len_b - q_len_b) for key j in [0, k_len_b):
 *   base(p,j) = (causal ? j <= p : (window_right < 0 || j <= p + window_right))
 *               && (window_left < 0 || j >= p - window_left)
 *   rng(p,j)  = table_row.start <= j <= table_row.end
 *               && (window_left < 0 || j >= p - window_left)
 *   visible   = base || rng
 * A "W-token causal window" is window_left = W - 1 (PR #50294 forward():
 * the kept distance is < 1 + window); a symmetric window |i - j| <= w is
 * causal = 0, window_left = window_right = w (PR #49815).
 * Scores s = scale * q.k with KV head h / (num_heads_q / num_heads_kv).
 * Sinks (fp32 [num_heads_q], natural-log units): KEY0_BIAS adds sink[h] to
 * s[.,0] when key 0 is visible; NULL_LOGIT adds exp(sink[h]) to the softmax
 * denominator.  out = sum_j softmax_j * v_j; lse = ln(denominator) (sink
 * included).  A row with nothing visible gets out = 0, lse = -inf (sink in
 * null-logit mode).
 *
 * q      bf16 [total_q, num_heads_q, head_dim], contiguous, 16-byte aligned.
 * k, v   bf16 [total_k, num_heads_kv, head_dim], contiguous, 16-byte aligned.
 * out    bf16 [total_q, num_heads_q, head_dim] (written for every row).
 * lse    fp32 [num_heads_q, total_q] or NULL.  NULL skips the log-sum-exp
 *                 (the prefill kernel then runs an instantiation without its
 *                 unrounded-sum add); out is the same bit for bit either way.
 * cu_seqlens_q, cu_seqlens_k  int32 [num_reqs + 1] packed offsets, within
 *                 total_q / total_k, with 0 <= q_len <= k_len per request.
 *                 The product library trusts them (reading them on the host
 *                 would synchronise); the bounds-checked build
 *                 (libmvp_debug.so) reports a request with q_len > k_len, or
 *                 a row outside total_q, as MVP_ERR_DEVICE_BOUNDS.
 * context_lens int32 [num_reqs] or NULL (NULL: k_len - q_len).
 * max_q_len, max_k_len  host upper bounds of the per-request lengths (used to
 *                 size the grid; rows beyond them are not computed).
 * num_decode_reqs -1: the batch may mix single-token (decode) requests and
 *                 longer ones anywhere; both kernels cover every request and
 *                 each skips the other's, one after the other.  k >= 0: the
 *                 caller guarantees that requests [0, k) are exactly those
 *                 with q_len == 1 (the decode-first order vLLM's scheduler
 *                 uses); then the decode kernel covers only [0, k), the
 *                 prefill kernel only [k, num_reqs), a side with no requests
 *                 is not launched, and when both are the decode kernel runs
 *                 beside the prefill kernel on a second stream of the
 *                 library's (forked from and joined back to `stream`; see
 *                 mixed_prefill_sms of mvp_attn_options).
 * head_dim       64, 128, 256 or 512.  num_heads_q % num_heads_kv == 0.
 * range_table    int32 [total_q, 2] from mvp_fill_query_ranges, or NULL.
 * range_covered  int32 device scalar (rows_written of the fill) or NULL; when
 *                it reads 0 the table is ignored.
 * workspace      device scratch of workspace_bytes (may be NULL / 0); see
 *                mvp_attn_workspace_size.
 * scale          softmax scale, finite and > 0 (MVP_ERR_ARG otherwise).
 * Errors: MVP_ERR_ARG, MVP_ERR_UNSUPPORTED (head_dim, alignment, head ratio),
 *         MVP_ERR_CUDA.  Requests with q_len == 0 produce no rows.
 */
int mvp_attn_fwd_varlen(const void* q, const void* k, const void* v, void* out, float* lse,
                        const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                        const int32_t* context_lens, int num_reqs, int total_q, int total_k,
                        int max_q_len, int max_k_len, int num_decode_reqs, int num_heads_q,
                        int num_heads_kv,
                        int head_dim, const int32_t* range_table, const int32_t* range_covered,
                        int causal, int window_left, int window_right, const float* sinks,
                        int sink_mode, float scale, void* workspace, size_t workspace_bytes,
                        void* stream);

/*
 * Variants and testing options of one attention call (mvp_attn_fwd_varlen_ext).
 *
 * variant        MVP_VARIANT_DEFAULT, or MVP_VARIANT_D512_HEAD_SPLIT (head_dim
 *                512 only, MVP_ERR_UNSUPPORTED otherwise): a 2-CTA cluster
 *                splits the head dimension of each 128-row query tile, so
 *                O of all 512 value columns stays in tensor memory and QK^T is
 *                not recomputed; the two CTAs add their partial scores through
 *                distributed shared memory every key tile.  Same results
 *                within the tolerances, but slower on GB300 than the default
 *                (which splits the value dimension over two work items, each
 *                recomputing the scores).
 * wait_limit_us  budget of one bounded device wait in microseconds; 0 means
 *                the default of one second.  Every legitimate wait lasts
 *                microseconds per key tile, but a wait can span a whole work
 *                item (its rows times its keys), so a budget below a few
 *                milliseconds risks reporting a timeout on a healthy call.
 * mixed_prefill_sms
 *                batches with both single-token (decode) rows and longer
 *                rows, given in decode-first order (num_decode_reqs >= 1
 *                and rows after them), run the decode kernel beside the
 *                prefill kernel: the prefill kernel's persistent CTAs take
 *                this many SMs (0: the library's choice, 1.2 times the
 *                prefill side's part of the two sides' estimated work, at
 *                most three quarters of the SMs, when the decode side's
 *                estimated work is at least a third of the prefill side's,
 *                else the two kernels run in turn; > 0: that many, rounded
 *                to CTA pairs and at most the SM count - 2) and the decode
 *                kernel runs on a second stream
 *                of the library's (one per device), forked from and joined
 *                back to `stream` with events, so all the call's work is
 *                still ordered before later work on `stream`, also inside a
 *                CUDA graph capture.  -1: the two kernels run one after the
 *                other on `stream`.
 * fault          MVP_FAULT_NONE for every real call.  MVP_FAULT_WITHHOLD_PROBS
 *                exists to test the timeout path: in every prefill CTA that
 *                gets work (rank 0 of each CTA pair) one softmax warp never
 *                signals that its first key tile's probabilities are ready,
 *                so the MMA issuer's wait for them runs out; the kernel
 *                records MVP_ERR_DEVICE_TIMEOUT (see
 *                mvp_get_last_device_error), unwinds, frees its tensor memory
 *                and returns, the prefill outputs of that call being
 *                undefined.  Single-token rows (the decode kernel) are not
 *                affected.
 */
typedef enum { MVP_VARIANT_DEFAULT = 0, MVP_VARIANT_D512_HEAD_SPLIT = 1 } mvp_variant;
typedef enum { MVP_FAULT_NONE = 0, MVP_FAULT_WITHHOLD_PROBS = 1 } mvp_fault;
typedef struct {
  int variant;            /* mvp_variant */
  unsigned wait_limit_us; /* 0: default (1 s) */
  int fault;              /* mvp_fault */
  int mixed_prefill_sms;  /* 0: estimate; > 0: SMs of the prefill kernel; -1: no overlap */
} mvp_attn_options;

/*
 * mvp_attn_fwd_varlen with options (NULL options: identical to
 * mvp_attn_fwd_varlen).  Errors as mvp_attn_fwd_varlen, plus MVP_ERR_ARG for
 * an unknown variant or fault and MVP_ERR_UNSUPPORTED for the D = 512 head
 * split at another head_dim.
 */
int mvp_attn_fwd_varlen_ext(const void* q, const void* k, const void* v, void* out, float* lse,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                            const int32_t* context_lens, int num_reqs, int total_q, int total_k,
                            int max_q_len, int max_k_len, int num_decode_reqs, int num_heads_q,
                            int num_heads_kv, int head_dim, const int32_t* range_table,
                            const int32_t* range_covered, int causal, int window_left, int window_right,
                            const float* sinks, int sink_mode, float scale, void* workspace,
                            size_t workspace_bytes, void* stream, const mvp_attn_options* options);

/*
 * The same attention over a paged K/V cache (the block-table layout of
 * vLLM's paged attention, which the FA4 pages run their masks on): the keys
 * and values of request b are not packed rows but seq_lens_k[b] positions
 * spread over fixed-size blocks of a shared cache.
 *
 * k_cache, v_cache  bf16 [num_blocks * block_size, num_heads_kv, head_dim]
 *                 (that is, [num_blocks, block_size, Hkv, D] contiguous),
 *                 16-byte aligned.
 * block_table     int32 [num_reqs, max_blocks_per_seq]: key j of request b
 *                 is row block_table[b][j / block_size] * block_size
 *                 + j % block_size of the caches.  Only the entries of blocks
 *                 holding the request's keys are read; ids outside
 *                 [0, num_blocks) read zeros (TMA bounds), never out of the
 *                 caches.
 * seq_lens_k      int32 [num_reqs], keys per request (k_len); the request's
 *                 queries end at its last key unless context_lens says
 *                 otherwise.
 * block_size      16, 32, 64, 128 or 256.
 * max_blocks_per_seq * block_size must cover max_k_len.
 * All other arguments, results and errors are those of mvp_attn_fwd_varlen
 * (cu_seqlens_k is replaced by seq_lens_k + block_table); packed and paged
 * calls on the same logical keys give bit-identical results.
 * Errors: MVP_ERR_ARG also for a block size outside the list, a table too
 * short for max_k_len, or NULL block_table / seq_lens_k.
 */
int mvp_attn_fwd_paged(const void* q, const void* k_cache, const void* v_cache, void* out, float* lse,
                       const int32_t* cu_seqlens_q, const int32_t* seq_lens_k, const int32_t* block_table,
                       int block_size, int max_blocks_per_seq, int num_blocks, const int32_t* context_lens,
                       int num_reqs, int total_q, int max_q_len, int max_k_len, int num_decode_reqs,
                       int num_heads_q, int num_heads_kv, int head_dim, const int32_t* range_table,
                       const int32_t* range_covered, int causal, int window_left, int window_right,
                       const float* sinks, int sink_mode, float scale, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * Scan mode: the same attention with the request-level range list of vLLM's
 * Triton path instead of the per-row table (PR #50294 review,
 * "Implementation breakdown" 2: the (num_seqs, max_ranges, 2) tensor that
 * compute_mm_prefix_range_tensor keeps for the Triton path; the metadata
 * test's old per-score scan: keep iff some valid range, start < end, holds
 * both the query position and the key).  No fill step: each query row scans
 * its request's ranges once (not once per score) and keeps the union of the
 * valid ranges holding its position, which is one interval because they all
 * contain it.  Visible = base || (that interval, clamped by window_left on
 * the past side), exactly as with the table.  With non-overlapping ranges
 * (the invariant the page's O(1) table relies on) the results are
 * bit-identical to mvp_fill_query_ranges + mvp_attn_fwd_varlen; overlapping
 * ranges follow the scan (union), where the table keeps the last range.
 *
 * ranges      int32 [num_reqs, max_ranges, 2] row-major, 8-byte aligned,
 *             closed (start, end) absolute positions; padding (0, 0).
 * max_ranges  1..4096 (0: no ranges, as a call without a table).
 * All other arguments, results and errors are those of mvp_attn_fwd_varlen
 * (no range_table / range_covered); MVP_ERR_ARG also for max_ranges outside
 * [0, 4096] or NULL ranges with max_ranges > 0.
 */
int mvp_attn_fwd_varlen_scan(const void* q, const void* k, const void* v, void* out, float* lse,
                             const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, const int32_t* context_lens,
                             int num_reqs, int total_q, int total_k, int max_q_len, int max_k_len,
                             int num_decode_reqs, int num_heads_q, int num_heads_kv, int head_dim,
                             const int32_t* ranges, int max_ranges, int causal, int window_left, int window_right,
                             const float* sinks, int sink_mode, float scale, void* workspace,
                             size_t workspace_bytes, void* stream);

/*
 * Allocation-free variant of mvp_attn_fwd_varlen.  The pages have no
 * counterpart of this call; it exists for callers that cannot allocate device
 * memory where they run attention (an engine whose free memory is already
 * committed to its KV-cache pool, a plugin inside a framework that owns the
 * allocator, a path that must not synchronise on an allocation) and so cannot
 * pass the split-KV workspace.  Arguments and results are exactly those of
 * mvp_attn_fwd_varlen without workspace/workspace_bytes: the split-KV partials
 * go to a fixed 16 MiB array in the library's own device memory
 * (mvp_static_scratch_bytes()), which every GPU that loads the library holds
 * until the process exits.  The call allocates nothing.
 *   - Long decode rows are split over as many CTAs as the array holds
 *     partials for (at most what mvp_attn_workspace_size would give), so a
 *     large decode batch runs with fewer splits than with a full workspace.
 *     The maximum: the array (less its 256-byte header) must hold one
 *     split's partials of the call's decode rows, decode_requests x
 *     num_heads_q x (head_dim + 2) x 4 bytes (decode_requests =
 *     num_decode_reqs, or num_reqs when that is -1); a larger call is
 *     rejected with MVP_ERR_CAPACITY before anything is launched.
 *   - The first call on a device looks up the array's device address (and the
 *     library's other per-device state); make that first call before any
 *     stream capture.
 *   - All calls share the array and it keeps the last call's contents; nothing
 *     in it needs to start at zero.  Calls whose kernels overlap on the GPU
 *     (unordered streams) race on it.
 */
int mvp_attn_fwd_varlen_static_ws(const void* q, const void* k, const void* v, void* out, float* lse,
                                  const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                  const int32_t* context_lens, int num_reqs, int total_q, int total_k,
                                  int max_q_len, int max_k_len, int num_decode_reqs, int num_heads_q,
                                  int num_heads_kv, int head_dim, const int32_t* range_table,
                                  const int32_t* range_covered, int causal, int window_left, int window_right,
                                  const float* sinks, int sink_mode, float scale, void* stream);

/* Size in bytes of the fixed scratch array used by mvp_attn_fwd_varlen_static_ws. */
size_t mvp_static_scratch_bytes(void);

/*
 * Step metadata for CUDA-graph replays.  Source: vLLM PR #50294 review,
 * "Implementation breakdown" step 3 (FlashAttentionMetadataBuilder): a pinned
 * host staging area and a persistent device buffer are allocated once for
 * the largest batch; each step fills the staging area on the host from the
 * query offsets and an upper bound of the sequence lengths, then copies it to
 * the device without blocking.  The optimistic bound places a decode row at
 * or past its true position, which keeps it outside every range (ranges hold
 * prompt tokens; a decoded token never lies in one).
 *
 * One "metadata block" (int32, mvp_meta_block_bytes bytes, identical layout
 * on host and device) holds, at the element offsets mvp_meta_offsets gives:
 *   [0] query_start_loc  [max_reqs + 1]   (cu_seqlens_q of the attention)
 *   [1] seq_lens_k       [max_reqs]       (exact key lengths: the paged call)
 *   [2] cu_seqlens_k     [max_reqs + 1]   (prefix sums of [1]: the packed call)
 *   [3] seq_lens_bound   [max_reqs]       (the fill's key lengths)
 *   [4] ranges           [max_reqs, max_ranges, 2]  (8-byte aligned)
 * A batch of num_reqs <= max_reqs requests and query_start_loc[num_reqs] <=
 * max_tokens rows is padded to the capacity with requests that have no rows,
 * no keys and no ranges, so every step is the same two operations (one copy
 * of the whole block, one fill of max_tokens table rows) on the same
 * pointers, whatever the batch: capture them, and an attention call on the
 * block's arrays sized for the capacity (num_reqs = max_reqs, total_q =
 * max_tokens, max_q_len / max_k_len upper bounds), in one CUDA graph and
 * replay it for every batch that fits.
 */
typedef struct mvp_meta mvp_meta;

/* Bytes of a metadata block for this capacity (0 for max_reqs outside
 * [1, 65535] or max_ranges outside [0, 4096]). */
size_t mvp_meta_block_bytes(int max_reqs, int max_ranges);

/* Element offsets of the five arrays of a block into offsets[0..4]. */
int mvp_meta_offsets(int max_reqs, int max_ranges, size_t* offsets);

/*
 * Host only (no CUDA call): writes the padded block for one batch into
 * `block` (host memory of mvp_meta_block_bytes bytes).  All inputs are HOST
 * arrays:
 *   query_start_loc [num_reqs + 1], starting at 0, non-decreasing;
 *   seq_lens_k      [num_reqs] exact key lengths, or NULL (then [1] and [2]
 *                   hold zeros and the caller supplies its own);
 *   seq_lens_bound  [num_reqs] the fill's lengths (>= the exact ones; a
 *                   prefill row needs the exact value, a decode row may take
 *                   an upper bound), or NULL to use seq_lens_k;
 *   ranges          [num_reqs, num_ranges, 2] as for mvp_fill_query_ranges,
 *                   or NULL (no ranges).
 * Errors (nothing written): MVP_ERR_ARG for NULL inputs a batch needs, a
 * query_start_loc that does not start at 0 or decreases, a key length below
 * the request's query count, keys summing past INT_MAX; MVP_ERR_CAPACITY for
 * num_reqs > max_reqs, num_ranges > max_ranges or more than max_tokens rows.
 */
int mvp_meta_pack(const int32_t* query_start_loc, const int32_t* seq_lens_k, const int32_t* seq_lens_bound,
                  const int32_t* ranges, int num_reqs, int num_ranges, int max_reqs, int max_tokens,
                  int max_ranges, int32_t* block);

/*
 * Creates a builder on the current device.  The caller owns and keeps alive
 * the device arrays: device_block (mvp_meta_block_bytes, 16-byte aligned),
 * range_table (int32 [max_tokens, 2], 8-byte aligned) and range_covered
 * (int32 scalar).  The builder allocates its pinned staging block here and
 * nothing afterwards; the staged batch starts empty.
 * Errors: MVP_ERR_ARG, MVP_ERR_UNSUPPORTED (alignment), MVP_ERR_CUDA.
 */
int mvp_meta_create(int max_reqs, int max_tokens, int max_ranges, int32_t* device_block, int32_t* range_table,
                    int32_t* range_covered, mvp_meta** out);

/* Waits for the builder's last copy and frees its staging block and event. */
int mvp_meta_destroy(mvp_meta* meta);

/*
 * Host step: waits until the last upload's copy (eager or replayed from a
 * graph) has read the staging block, then packs this batch into it
 * (mvp_meta_pack's arguments and errors).  Not a stream operation: call it
 * outside any capture.
 */
int mvp_meta_stage(mvp_meta* meta, const int32_t* query_start_loc, const int32_t* seq_lens_k,
                   const int32_t* seq_lens_bound, const int32_t* ranges, int num_reqs, int num_ranges);

/*
 * Stream step (capturable): one asynchronous copy of the staged block into
 * device_block, an event marking the staging block free, and the range-table
 * fill over the block (max_reqs requests, max_tokens rows) into range_table
 * and range_covered.  Two kernel-side operations and no allocation.
 */
int mvp_meta_upload(mvp_meta* meta, void* stream);

/*
 * Work accounting of one attention call (host only, no CUDA call).
 *
 * Source: vLLM PR #55624 report ("Support Sliding Window Attention and hybrid
 * layers in MFU/MBU estimation"), Implementation breakdown 2 and 4 and the
 * ExecutionContext snippet: each request adds num_tokens x
 * min(context_len, sliding_window) token-context products (the full context
 * without a window); attn_qk and attn_av cost 2 x heads x head_dim FLOPs per
 * product; decode requests read min(context_len, sliding_window) keys and
 * values per KV head.  The report's risks name this an upper bound never
 * reconciled with profiler counts; the exact and executed fields below are
 * what closes that gap (the executed ones are the figures a profiler's
 * tensor-instruction and DRAM counters measure for this library).
 *
 * Readings: context_len = the request's key count (seq_lens_k);
 * sliding_window = window_left + 1 (the keys a causal window keeps), none
 * when window_left < 0; requests with one query row are decode requests.
 */
typedef struct {
  /* the page's estimate */
  double est_token_context_product; /* sum num_tokens * min(context_len, window)      */
  double est_attn_qk_flops;         /* 2 Hq D x the product                            */
  double est_attn_av_flops;         /* 2 Hq D x the product                            */
  double est_decode_kv_read_bytes;  /* decode rows: 2 (K, V) Hkv D 2 bytes min(ctx, W)  */
  /* the exact mask of this library (per query row; every q head alike) */
  long long visible_prefill;        /* visible (row, key) pairs of rows with q_len > 1 */
  long long visible_decode;         /* ... of single-row (decode) requests             */
  double exact_flops;               /* 4 D Hq (visible_prefill + visible_decode)      */
  double exact_decode_kv_bytes;     /* 2 (K, V) Hkv D 2 bytes visible_decode           */
  /* what the kernels execute */
  long long prefill_items;          /* work items with at least one key tile           */
  long long prefill_tiles;          /* key tiles visited, summed over items            */
  long long prefill_mma_instructions; /* tcgen05.mma issued: tiles x (D/16 + BN/16)   */
  double prefill_mma_flops;         /* 2 M BN (D + DV) per tile (M = 128 x CTAs/MMA),
                                       plus 2 M BN 32 per tile at D = 128 (row sums
                                       carried by the PV MMA)                          */
  double prefill_compulsory_bytes;  /* q and out once, K and V of the visited tiles    */
                                    /* once (lse not included)                         */
  long long decode_keys_walked;     /* keys read per KV head (tiles start on multiples */
                                    /* of the decode tile size)                        */
  double decode_read_bytes;         /* walked K and V once + q                         */
  double decode_cta_read_bytes;     /* the same as the decode CTAs load it (a KV head  */
                                    /* is read once per CTA of its q-head group)       */
} mvp_attn_counts;

/*
 * Fills *out for an attention call with these HOST arrays: cu_seqlens_q
 * [num_reqs + 1], seq_lens_k [num_reqs], context_lens [num_reqs] or NULL,
 * range_table [total_q, 2] (as mvp_fill_query_ranges leaves it) or NULL, and
 * the call's heads, head_dim and mask scalars; variant (mvp_variant) selects
 * the prefill kernel whose executed work is counted.
 * Errors: MVP_ERR_ARG (NULL out or arrays, negative lengths, a query offset
 * array not starting at 0, bad mask scalars, unknown variant),
 * MVP_ERR_UNSUPPORTED (head_dim, or the D = 512 head split at another one).
 */
int mvp_attn_accounting(const int32_t* cu_seqlens_q, const int32_t* seq_lens_k, const int32_t* context_lens,
                        const int32_t* range_table, int num_reqs, int num_heads_q, int num_heads_kv, int head_dim,
                        int causal, int window_left, int window_right, int variant, mvp_attn_counts* out);

/* Synchronises `stream`, returns MVP_ERR_DEVICE_TIMEOUT if a kernel recorded a
 * timeout since the last call (and clears it), MVP_ERR_DEVICE_BOUNDS if a
 * kernel of the bounds-checked build (libmvp_debug.so, compiled with
 * MVP_DEBUG_BOUNDS; every entry point the same) found an index outside its
 * buffer, MVP_ERR_CUDA on a CUDA error, else MVP_OK.  Each library has its
 * own error word. */
int mvp_get_last_device_error(void* stream);

/* Static string for a status code. */
const char* mvp_status_str(int status);

/* Number of kernel launches the last successful mvp_attn_fwd_varlen /
 * mvp_attn_fwd_paged / mvp_fill_query_ranges call enqueued on this thread
 * (for launch accounting). */
int mvp_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* MVP_H_ */
