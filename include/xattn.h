/*
 * libxattn -- XAttention block-sparse attention (BSA) for chunked prefill,
 * single GPU, sm_103a.
 *
 * One chunk of prefill is three steps, each an entry point below, all issued
 * on one caller-given CUDA stream in this order:
 *
 *   xattn_estimate       block importance: stride-reshaped Q.K^T scores,
 *                        softmax statistics merged across KV tiles, and
 *                        per-(query block, KV block) attention mass
 *   xattn_select         cumulative-attention threshold per (head, query block),
 *                        GQA "any" per KV-head group, majority vote, sink and
 *                        last history block forced, block_table lookup
 *   bsa_chunk_attention  attention over the selected history pages
 *                        (non-causal) and the current chunk (causal), merged
 *                        by log-sum-exp, with the output's LSE
 *
 * and lse_merge, the stand-alone merge of two partial attention results;
 * xattn_store_kv, which writes a chunk's keys and values into the pool pages
 * its positions map to (the history of the request's next chunk).
 *
 * Sources: "XAttention BSA Policy 设计文档" (nano-vllm
 * docs/xattn_bsa_policy_design.md), sections 核心算法 1 select_blocks (Steps 1-4)
 * and 2 compute_chunked_prefill; "XAttention Offload Stream Synchronization
 * Fix" (docs/xattn_offload_stream_sync_fix.md), section 技术细节 (three-stage
 * KV chunking, stream configuration); "Atenção paginada" (transformers docs
 * paged_attention.md), Caminho Varlen / Caminho de decodificação (cu_seq_lens,
 * block_table); "Task Plan: Layerwise Offload Refactoring" (task_plan.md),
 * Phase 1.2 (per-block KV store).
 *
 * Conventions common to every entry point
 * ---------------------------------------
 * Memory:    every pointer marked DEVICE is global memory of the current
 *            device, owned by the caller; the library allocates nothing and
 *            frees nothing.  HOST pointers are read during the call only.
 * Streams:   all work is enqueued on `stream`; no call synchronises the host,
 *            touches the default stream or records events.  Data produced on
 *            another stream must be ordered by the caller (an event wait on
 *            `stream`) before the call -- the ordering bug the stream-sync
 *            page documents cannot occur inside the library.
 * Tokens:    a chunk packs B requests along the token axis (B = 1 for a plain
 *            chunked prefill).  Request r owns query tokens
 *            [cu_seqlens_q[r], cu_seqlens_q[r+1]) of q, k_cur, v_cur, o, lse,
 *            and has cu_seqlens_kh[r+1]-cu_seqlens_kh[r] history tokens stored
 *            in the paged pool.  Every length is a multiple of block_size.
 * Layouts:   q, o      bf16 [H, tokens, D]   (head h at h*q_head_stride)
 *            k_cur,v_cur bf16, element (KV head h, token t, d) at
 *                      h*kv_head_stride + t*kv_token_stride + d: [Hkv, tokens, D]
 *                      (kv_token_stride = D) or [tokens, Hkv, D]
 *                      (kv_head_stride = D, kv_token_stride = Hkv*D, e.g. the
 *                      chunk's own pages of a pool laid out in logical order)
 *            lse       fp32 [H, tokens]      (head at h*lse_head_stride)
 *            k_pool,v_pool bf16 [num_pages, block_size, Hkv, D]
 *            block_table int32 [B, bt_stride]; history token t of request r is
 *                      row t % block_size of page block_table[r][t / block_size];
 *                      -1 marks an unallocated page.
 *            GQA:      query head h reads KV head h / (H / Hkv).
 * Errors:    argument checks happen on the host before any launch and return a
 *            negative status with nothing enqueued.  Faults found by kernels
 *            (a page id outside [0, num_pages) reached through block_table or
 *            the selection) never trap: the kernel skips the page, records the
 *            first such fault in a device error word and continues; read it
 *            with xattn_device_error.  Every wait inside a kernel is bounded:
 *            one that runs out records XATTN_ETIMEOUT and the kernel returns.
 * Lifetime:  the library looks up, once per device, the device addresses of its
 *            own __device__ variables (the error word, the counters of
 *            xattn_select_noalloc) and keeps them for the life of the process.
 *            Do not use it across cudaDeviceReset or any other teardown of a
 *            device's primary context: the kept addresses would be stale.
 */
#ifndef XATTN_H
#define XATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *xattn_stream_t; /* identical to cudaStream_t */

typedef enum xattn_status {
  XATTN_OK = 0,
  XATTN_EINVAL = -1,          /* null pointer, bad size or divisibility */
  XATTN_EALIGN = -2,          /* pointer or stride not 16-byte aligned */
  XATTN_EPAGE = -3,           /* (device word) page id out of range */
  XATTN_ECUDA = -4,           /* a CUDA runtime call or launch failed */
  XATTN_EUNSUPPORTED = -5,    /* head_dim / block geometry not built */
  XATTN_EWORKSPACE = -6,      /* workspace smaller than xattn_workspace_size */
  XATTN_ETIMEOUT = -7         /* (device word) a kernel pipeline wait ran out; the
                                 kernel stopped early and its outputs are invalid */
} xattn_status;

#define XATTN_MAX_REQUESTS 64
#define XATTN_MAX_BLOCKS_PER_ROW 8192 /* history + current blocks of one request */

/* Problem description shared by every entry point (host memory).
 * Constraints (XATTN_EINVAL / XATTN_EUNSUPPORTED otherwise):
 *   1 <= num_requests <= XATTN_MAX_REQUESTS; num_heads % num_kv_heads == 0;
 *   head_dim in {64, 128}; block_size % 64 == 0; block_size % stride == 0;
 *   block_size / stride a power of two in [8, 32]; 1 <= stride <= 64;
 *   every query and history length a multiple of block_size;
 *   history blocks + query blocks of a request <= XATTN_MAX_BLOCKS_PER_ROW;
 *   history blocks of a request <= bt_stride. */
typedef struct xattn_problem {
  int32_t num_requests;           /* B */
  int32_t num_heads;              /* H, query heads */
  int32_t num_kv_heads;           /* Hkv */
  int32_t head_dim;               /* D */
  int32_t stride;                 /* S, XAttention stride ("stride reshape") */
  int32_t block_size;             /* Bk: BSA block == KV page size (tokens) */
  const int32_t *cu_seqlens_q;    /* HOST [B+1] cumulative query-chunk lengths */
  const int32_t *cu_seqlens_kh;   /* HOST [B+1] cumulative history lengths */
  const int32_t *block_table;     /* DEVICE [B, bt_stride] physical page ids */
  int32_t bt_stride;              /* row pitch of block_table (>= history blocks) */
  int32_t num_pages;              /* pages in k_pool / v_pool */
  int64_t q_head_stride;          /* elements between heads of q and o */
  int64_t kv_head_stride;         /* elements between heads of k_cur and v_cur */
  int64_t lse_head_stride;        /* elements between heads of lse */
  int64_t kv_token_stride;        /* elements between tokens of k_cur and v_cur;
                                     0 means head_dim (the [Hkv, tokens, D] layout).
                                     The two strides must describe [Hkv, tokens, D]
                                     (kv_head_stride >= tokens * kv_token_stride) or
                                     [tokens, Hkv, D] (kv_token_stride >= Hkv *
                                     kv_head_stride), both >= D, multiples of 8
                                     (XATTN_EINVAL / XATTN_EALIGN otherwise). */
} xattn_problem;

/* Bytes of scratch the caller must provide to xattn_estimate, xattn_select and
 * bsa_chunk_attention for this problem (0 on invalid problems).  The workspace
 * holds the estimation's per-(reshaped row, KV block) partial sums and
 * per-tile softmax statistics, the selection's vote counters (and the counter
 * that tells its last CTA to run the vote) and the attention's partial
 * results; its contents between calls are unspecified.  The estimation and
 * selection use the start of the buffer they are given, the attention the end
 * of it: with one buffer for a whole chunked prefill, a chunk's estimate does
 * not touch what the previous chunk's attention is still using (see
 * xattn_estimate, Ordering). */
size_t xattn_workspace_size(const xattn_problem *p);

/* Number of fp32 elements of block_sums (and bytes of the optional mask):
 * request by request, [H, Qb_r, Kb_r] with Qb_r = q_len_r / block_size and
 * Kb_r = (kh_len_r + q_len_r) / block_size (history blocks first, then the
 * current chunk's blocks), requests packed back to back. */
size_t xattn_block_sums_count(const xattn_problem *p);

/* Element offset of request r's [H, Qb_r, Kb_r] slab inside block_sums. */
size_t xattn_block_sums_offset(const xattn_problem *p, int32_t r);

/* Estimation (BSA policy page, select_blocks Steps 1-2; stream-sync page,
 * three-stage KV chunking).  For every query head h (KV head h / G), reshaped
 * row a < q_len/S and reshaped column b over [history ; current chunk]:
 *   s[a,b] = scale * sum_{i<S} q[S a + S-1-i] . k[S b + i]        (antidiagonal)
 * current-chunk column b' is visible from row a iff b' <= a; history is all
 * visible.  Per row, softmax statistics (max, sum of exp) are taken per
 * 128-column tile, merged across tiles, and
 *   block_sums[h, qb, kb] = sum over the (block/S)^2 visible cells of the
 *                           block of exp(s - m_row) / l_row.
 *   q       DEVICE bf16, layout above      k_cur  DEVICE bf16
 *   k_pool  DEVICE bf16 paged history keys
 *   scale   logit scale; the usual choice is 1 / (sqrt(D) * S)
 *   workspace, workspace_bytes   DEVICE scratch >= xattn_workspace_size(p)
 *   block_sums  DEVICE fp32 [xattn_block_sums_count(p)], written fully.
 * Ordering: when the call right before this one on `stream` is this
 * library's bsa_chunk_attention (a previous chunk's), and the workspace this
 * estimate writes does not overlap the part of its workspace that attention
 * uses (the library checks the two ranges), the estimate may start on SMs
 * that attention has released while its last CTAs still run (programmatic
 * dependent launch).  It finishes only after that attention has, so
 * everything enqueued after it sees both complete.  Its inputs must not be
 * that attention's outputs: do not pass its o or lse as q or keys here.
 * After any other kernel or stream operation the estimate starts as usual.
 * The same holds for xattn_estimate_seq and xattn_estimate_sampled. */
xattn_status xattn_estimate(const xattn_problem *p, const void *q, const void *k_cur,
                            const void *k_pool, float scale, void *workspace,
                            size_t workspace_bytes, float *block_sums,
                            xattn_stream_t stream);

/* The same estimation, reading each request's keys -- history, then the
 * current chunk -- from one buffer in logical token order instead of the pool
 * pages and k_cur.  The BSA policy page's select_blocks (Step 1) copies every
 * history K block to the GPU and transposes it to [heads, k_len, D] before
 * its GEMM; here the caller keeps the keys in that order (as a prefill holds
 * its K anyway), so the GEMM fetches the 256 keys of a score tile at one
 * stride phase as a single strided copy rather than one copy per page.
 * Results equal xattn_estimate's on the same keys bit for bit.
 *   k_seq               DEVICE bf16, element (KV head h, token t, d) at
 *                       h*k_seq_head_stride + t*k_seq_token_stride + d
 *   k_seq_head_stride, k_seq_token_stride   elements, multiples of 8, >= D;
 *                       token stride 0 means D; the layout is [Hkv, tokens, D]
 *                       or [tokens, Hkv, D] (as for k_cur)
 *   k_seq_start         HOST int64 [B]: request r's kh_r + q_r keys are tokens
 *                       [k_seq_start[r], k_seq_start[r] + kh_r + q_r) of k_seq,
 *                       its history first; each a multiple of the stride
 * The buffer must hold max_r(k_seq_start[r] + kh_r + q_r) tokens.  Other
 * arguments, outputs and errors as xattn_estimate. */
xattn_status xattn_estimate_seq(const xattn_problem *p, const void *q, const void *k_seq,
                                int64_t k_seq_head_stride, int64_t k_seq_token_stride,
                                const int64_t *k_seq_start, float scale, void *workspace,
                                size_t workspace_bytes, float *block_sums,
                                xattn_stream_t stream);

/* Estimation from a sample of each history block's keys (BSA policy page,
 * 性能分析, 优化方向 2: estimate with part of the K blocks; the chunked-prefill
 * page's Phase 1 loads samples_per_chunk tokens of each history chunk).  Of
 * every history block only its first `samples` reshaped columns
 * (samples * S tokens) are scored; each sampled cell stands for
 * (block_size / S) / samples cells of its block, so it is counted with that
 * weight in the row's softmax sum and in the block's sum.  The current chunk's
 * columns are all scored.  With the history sampled the score GEMM does about
 * samples / (block_size / S) of the history work.  A request whose sampled
 * columns, rounded up to 128, would not be fewer than its history's is
 * estimated in full.
 *   samples   (block_size / S) / 4 or / 2, and >= 4 (XATTN_EUNSUPPORTED
 *             otherwise)
 *   k_seq_start[r]   a multiple of block_size (XATTN_EINVAL otherwise)
 * Other arguments, outputs and errors as xattn_estimate_seq. */
xattn_status xattn_estimate_sampled(const xattn_problem *p, const void *q, const void *k_seq,
                                    int64_t k_seq_head_stride, int64_t k_seq_token_stride,
                                    const int64_t *k_seq_start, int32_t samples, float scale,
                                    void *workspace, size_t workspace_bytes, float *block_sums,
                                    xattn_stream_t stream);

/* Selection (BSA policy page, select_blocks Steps 3-4).
 * Per (request, head, query block) row, with integer masses
 * q_j = round_half_even(block_sums_j * 2^32), T = sum_j q_j, R = fl64(threshold*T):
 * blocks are visited by (q_j descending, j ascending) and block j is kept iff
 * the integer mass visited before it is < R (threshold >= 1 keeps every q_j > 0).
 * Then, over history blocks only: a KV-head group keeps a block if any of its
 * query heads does; a block is selected when
 *   votes * vote_den > vote_num * (Hkv * Qb_r)     (votes over KV heads x query blocks)
 * -- (1, 2) is the pages' strict majority -- and, if force_sink_last != 0,
 * history block 0 and block Kb_h-1 are always added.
 *   threshold   > 0 (0.9 and 0.95 are the pages' settings)
 *   vote_num, vote_den   0 <= vote_num <= vote_den, vote_den > 0 (XATTN_EINVAL otherwise)
 *   force_sink_last      0 or 1
 *   mask        DEVICE u8 [xattn_block_sums_count(p)] or NULL: per-head keep flags
 *   sel_idx     DEVICE int32 [B, bt_stride]: ascending logical history block ids
 *   sel_page    DEVICE int32 [B, bt_stride]: block_table[r][sel_idx]
 *   n_sel       DEVICE int32 [B]: number of valid entries per request
 * Entries past n_sel[r] are left untouched. */
xattn_status xattn_select(const xattn_problem *p, const float *block_sums, double threshold,
                          int32_t vote_num, int32_t vote_den, int32_t force_sink_last,
                          void *workspace, size_t workspace_bytes, uint8_t *mask,
                          int32_t *sel_idx, int32_t *sel_page, int32_t *n_sel,
                          xattn_stream_t stream);

/* Selection with one block set per KV head (BSA policy page, select_blocks
 * Step 4, "为什么使用 Majority Voting?": per-head selection beside the vote
 * across heads).  Threshold masks and the GQA "any" as for xattn_select; then
 * KV head k of request r keeps history block j when
 *   votes_k,j * vote_den > vote_num * Qb_r   (its own votes over its query blocks)
 * and, if force_sink_last != 0, blocks 0 and Kb_h-1.  Outputs are per
 * (request, KV head), row r*Hkv + k:
 *   sel_idx, sel_page   DEVICE int32 [B, Hkv, bt_stride]
 *   n_sel               DEVICE int32 [B, Hkv]
 * Other arguments and errors as xattn_select; feed the result to
 * bsa_chunk_attention_per_kv_head. */
xattn_status xattn_select_per_kv_head(const xattn_problem *p, const float *block_sums,
                                      double threshold, int32_t vote_num, int32_t vote_den,
                                      int32_t force_sink_last, void *workspace,
                                      size_t workspace_bytes, uint8_t *mask, int32_t *sel_idx,
                                      int32_t *sel_page, int32_t *n_sel, xattn_stream_t stream);

/* Capacity of the fixed counter array behind xattn_select_noalloc:
 * num_requests * bt_stride must not exceed it (1 MiB of int32 counters). */
#define XATTN_NOALLOC_MAX_COUNTERS 262144

/* Selection for callers that cannot allocate device memory.  The pages have
 * no counterpart: this exists for integrations where the caller has no
 * allocator to give the library scratch -- a serving process that hands all
 * free HBM to its KV-page pool and weights at start-up, or a C caller without
 * a caching allocator, for whom a cudaMalloc on the prefill path would block
 * the device or fail.  Same arguments, semantics and outputs as xattn_select
 * minus the workspace: the per-request vote counters live in a static device
 * array inside the library (XATTN_NOALLOC_MAX_COUNTERS int32, held by every
 * GPU that loads the library until the process exits).
 *  - Sizes: num_requests * bt_stride > XATTN_NOALLOC_MAX_COUNTERS returns
 *    XATTN_EWORKSPACE with nothing enqueued.
 *  - The first call on a device looks up the array's device address (once per
 *    device, with that device current); make that first call before any stream
 *    capture.
 *  - Every call clears the counters it uses on `stream`, then reuses the one
 *    array: calls that can overlap on the GPU (other streams, other host
 *    threads) race on it and must be ordered by the caller.
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
xattn_status xattn_select_noalloc(const xattn_problem *p, const float *block_sums,
                                  double threshold, int32_t vote_num, int32_t vote_den,
                                  int32_t force_sink_last, uint8_t *mask, int32_t *sel_idx,
                                  int32_t *sel_page, int32_t *n_sel, xattn_stream_t stream);

/* Sparse chunk attention (BSA policy page, compute_chunked_prefill).  For each
 * query token i of request r and head h, softmax attention with scale
 * softmax_scale over the keys of the selected history pages
 * (sel_page[r][0..n_sel[r]), all visible) and the current-chunk keys j <= i;
 * the history and causal parts are merged online by log-sum-exp, so the result
 * equals flash_attn_with_lse(history) merged with flash_attn_with_lse(causal).
 *   softmax_scale  > 0 (usually 1/sqrt(D)); XATTN_EINVAL otherwise
 *   workspace      DEVICE scratch of at least xattn_workspace_size(p) bytes,
 *                  16-byte aligned (XATTN_EWORKSPACE / XATTN_EALIGN otherwise);
 *                  the same buffer xattn_estimate / xattn_select take.  The
 *                  kernel picks its schedule on the device from n_sel: one CTA
 *                  per 256-row query unit for small launches, else the KV
 *                  tiles of all units split evenly over one persistent CTA per
 *                  SM; a unit cut between CTAs leaves normalised partial results
 *                  (fp32 O, LSE) here, merged by log-sum-exp into o / lse by the
 *                  CTA that finishes its part last.  The result does not depend
 *                  on which CTA that is (the parts are merged in a fixed order):
 *                  repeated calls give identical bits.
 *   o    DEVICE bf16 [H, tokens, D] (q_head_stride)   normalised output
 *   lse  DEVICE fp32 [H, tokens] (lse_head_stride)    natural-log LSE
 *        Either may instead be page-locked HOST memory (cudaHostAlloc,
 *        cudaMallocHost or cudaHostRegister): the kernel then writes it through
 *        its device alias over the host link, each row as it is finished, and
 *        no separate device-to-host copy is needed; the host may read it once
 *        the stream has passed the call.  Pageable host memory: XATTN_EINVAL.
 * A following xattn_estimate* call on the same stream may start before this
 * call has finished (see xattn_estimate, Ordering); every other operation
 * enqueued after it starts when it has finished. */
xattn_status bsa_chunk_attention(const xattn_problem *p, const void *q, const void *k_cur,
                                 const void *v_cur, const void *k_pool, const void *v_pool,
                                 const int32_t *sel_page, const int32_t *n_sel,
                                 float softmax_scale, void *workspace, size_t workspace_bytes,
                                 void *o, float *lse, xattn_stream_t stream);

/* bsa_chunk_attention over a selection per KV head (xattn_select_per_kv_head):
 * the query heads of KV head k of request r attend the pages in
 * sel_page[r][k][0..n_sel[r][k]) and the causal current chunk.
 *   sel_page  DEVICE int32 [B, Hkv, bt_stride];  n_sel  DEVICE int32 [B, Hkv]
 * Needs num_requests * num_kv_heads <= XATTN_MAX_REQUESTS (XATTN_EUNSUPPORTED
 * otherwise).  Other arguments, outputs and errors as bsa_chunk_attention. */
xattn_status bsa_chunk_attention_per_kv_head(const xattn_problem *p, const void *q,
                                             const void *k_cur, const void *v_cur,
                                             const void *k_pool, const void *v_pool,
                                             const int32_t *sel_page, const int32_t *n_sel,
                                             float softmax_scale, void *workspace,
                                             size_t workspace_bytes, void *o, float *lse,
                                             xattn_stream_t stream);

/* merge_attention_outputs (BSA policy page, compute_chunked_prefill): for each
 * of `rows` rows, lse = log(exp(lse1) + exp(lse2)) and
 * o = o1 * exp(lse1 - lse) + o2 * exp(lse2 - lse); two empty parts (-inf, -inf)
 * give o = 0, lse = -inf.
 *   o1, o2   DEVICE fp32 [rows, head_dim]; lse1, lse2 DEVICE fp32 [rows]
 *   o_out    DEVICE [rows, head_dim], fp32, or bf16 when o_out_bf16 != 0
 *   lse_out  DEVICE fp32 [rows]; o_out / lse_out may alias o1 / lse1. */
xattn_status lse_merge(const float *o1, const float *lse1, const float *o2,
                       const float *lse2, int64_t rows, int32_t head_dim, void *o_out,
                       int32_t o_out_bf16, float *lse_out, xattn_stream_t stream);

/* KV store of a prefill chunk ("Task Plan: Layerwise Offload Refactoring",
 * Phase 1.2, offload_layer_kv_async: a prefill's keys and values go block by
 * block into the cache blocks named by its block ids).  Chunk token t of
 * request r sits at position kh_r + t of the request, so for every KV head
 *   k_pool[page][row][kvh][:] = k_cur[kvh][q0_r + t][:]   (v likewise),
 *   page = block_table[r][(kh_r + t) / block_size], row = (kh_r + t) % block_size,
 * which makes the chunk's blocks history for the request's next chunk.
 *   k_cur, v_cur    DEVICE bf16 (kv_head_stride, kv_token_stride), as for
 *                   bsa_chunk_attention
 *   k_pool, v_pool  DEVICE bf16 [num_pages, block_size, Hkv, D], written
 * The block table row must reach the chunk's last block: (kh_r + lq_r) /
 * block_size <= bt_stride for every request, else XATTN_EINVAL (as are null
 * pointers and num_pages < 1); pointers must be 16-byte aligned (XATTN_EALIGN).
 * A table entry outside [0, num_pages) (-1: unallocated) records XATTN_EPAGE
 * in the device error word and that block is not written.  Enqueued on
 * `stream`; nothing else in the pools changes. */
xattn_status xattn_store_kv(const xattn_problem *p, const void *k_cur, const void *v_cur,
                            void *k_pool, void *v_pool, xattn_stream_t stream);

/* Host utility for streaming chunks (no method step): copies `rows` rows of
 * `width_bytes` bytes, src rows `src_pitch` bytes apart, dst rows `dst_pitch`
 * bytes apart -- e.g. the [H, chunk, D] window of a [H, L, D] tensor, one row
 * per head -- enqueued on `stream` (one 2-D copy).  to_device != 0: src is
 * HOST (pinned for an asynchronous copy), dst DEVICE; else the reverse.
 * XATTN_EINVAL on null pointers, negative sizes or a pitch below width_bytes. */
xattn_status xattn_copy_rows_async(void *dst, int64_t dst_pitch, const void *src, int64_t src_pitch,
                                   int64_t width_bytes, int64_t rows, int32_t to_device,
                                   xattn_stream_t stream);

/* Reads (and, if clear != 0, resets) the device error word of the current
 * device after synchronising `stream`.  *code is XATTN_OK or the first fault
 * status recorded by a kernel.  Diagnostic call: it blocks the host. */
xattn_status xattn_device_error(xattn_stream_t stream, int32_t *code, int32_t clear);

/* xattn_device_error(stream, code, 1) under the name of the boundary table:
 * the first fault status recorded since the last read, then reset.  Blocks
 * the host (diagnostics and tests). */
xattn_status xattn_last_device_error(xattn_stream_t stream, int32_t *host_code);

/* Static description of a status code. */
const char *xattn_status_string(xattn_status s);

#ifdef __cplusplus
}
#endif

#endif /* XATTN_H */
