// Internal definitions shared by the libxattn translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "xattn.h"

namespace xattn {

constexpr int kMaxReq = XATTN_MAX_REQUESTS;
constexpr int kTileCols = 128;  // columns of one softmax-statistics tile (score GEMM N tile)
constexpr int kAttnRows = 256;  // query rows per attention work unit (two 128-row MMA tiles)
constexpr int kAttnMaxCtas = 160;  // persistent attention CTAs at most (one per SM)
constexpr int kGemmRows = 256;  // reshaped rows per score-GEMM CTA (two 128-row MMA tiles)
constexpr int kGemmCols = 256;  // reshaped columns per score-GEMM CTA

// Per-request geometry of one chunk call (host-computed, passed by value).
struct ReqDesc {
  int32_t q0;      // first query token of the request in the packed token axis
  int32_t lq;      // query tokens (current chunk)
  int32_t kh;      // history tokens
  int32_t gemm0;   // first score-GEMM tile of the request
  int32_t bsum0;   // first CTA of the request in the block-sum grid
  int32_t sel0;    // ... in the selection grid
  int32_t att0;    // ... in the attention grid
  int32_t ks0;     // xattn_estimate_seq: first key group (token / S) of the request's keys
  int32_t head0;   // first query head of the request's heads (nonzero only when a
                   // request stands for one KV head's group: per-KV-head attention)
  int32_t kvh0;    // KV head of head0 (idem)
  int32_t hc;      // reshaped columns before the current chunk's: kh / S, or, when the
                   // request's history is sampled, its sampled columns padded to 128
  int32_t samp;    // 1: the history is estimated from a sample of each block's keys
  int64_t bpart_off;  // float offset of the request's [H, Qb, Kb, Br] block partial sums
  int64_t tstat_off;  // float2 offset of its [H, lq/S, ntiles] tile statistics
  int64_t bs_off;     // offset of its [H, Qb, Kb] block sums / mask
};

struct Geo {
  int32_t B, H, Hkv, D, S, Bk, bt_stride, num_pages;
  int64_t q_hs, kv_hs, lse_hs;
  int64_t kv_ts;          // elements between tokens of k_cur / v_cur
  int32_t kv_head_inner;  // 1 when kv_hs < kv_ts (a [tokens, Hkv, D] layout)
  int32_t H_all, Hkv_all; // heads of the q / k tensors (H, Hkv unless a request is one group)
  int32_t ns;             // sampled estimation: reshaped columns kept per history block
                          // (0: every column)
  const int32_t *block_table;
  int32_t *err;  // device error word
  ReqDesc req[kMaxReq];
};

// Request owning CTA `cta` of the grid whose per-request start is selected by F.
template <typename F>
__device__ __forceinline__ int find_req(const Geo &g, int cta, F start) {
  int r = 0;
  for (int i = 1; i < g.B; ++i)
    if (cta >= start(g.req[i])) r = i;
  return r;
}

__device__ __forceinline__ void record_error(int32_t *err, int32_t code) {
  atomicCAS(err, 0, code);
}

// Page id of logical block j of request r, or -1 (and an error record) when the
// block table entry is outside [0, num_pages).
__device__ __forceinline__ int page_of(const Geo &g, int r, int j) {
  int p = __ldg(g.block_table + (int64_t)r * g.bt_stride + j);
  if (p < 0 || p >= g.num_pages) {
    record_error(g.err, XATTN_EPAGE);
    return -1;
  }
  return p;
}

// ---------------------------------------------------------------------------
// Launch entry points implemented in the kernel translation units.
// ---------------------------------------------------------------------------
// Workspace of one call: the estimate's and selection's regions from the
// start of the buffer (offsets bpart, tstat, counts; est bytes), the
// attention's in a block of attn bytes at the end of the caller's buffer
// (offsets part_o, part_lse, att_cnt within that block).
struct WsLayout {
  size_t bpart, tstat, counts, est, part_o, part_lse, att_cnt, attn, total;
};

// Keys of every request in logical order (xattn_estimate_seq): element
// (kv head h, token t, d) at base[h * hs + t * ts + d]; request r's keys start
// at token S * req[r].ks0.
struct KeySeq {
  const __nv_bfloat16 *base;
  int64_t hs, ts;
};

// Score GEMM with its epilogue (block partial sums, tile statistics).  Keys
// come from kseq when it is given, else from the pool pages and k_cur.
// early: launch as a programmatic dependent of the kernel before it on st
// (it may start while that kernel finishes; it completes after it).
cudaError_t launch_score_gemm(const Geo &g, int ntiles, const __nv_bfloat16 *q,
                              const __nv_bfloat16 *kcur, const __nv_bfloat16 *kpool,
                              const KeySeq *kseq, float scale, float *bpart, float2 *tstat,
                              bool early, cudaStream_t st);
cudaError_t launch_block_sum(const Geo &g, int nctas, const float *bpart, const float2 *tstat,
                             float *block_sums, cudaStream_t st);
// Threshold selection of every (request, KV head, query block), then the GQA
// vote of every request (run by the CTA that finishes last; counts must hold
// rows * bt_stride + 1 zeroed int32: the vote counters and the finishing
// counter, with rows = B, or B * Hkv when per_kv: one selection per KV head).
cudaError_t launch_select(const Geo &g, int nctas, int max_kb, const float *block_sums,
                          double threshold, uint8_t *mask, int32_t *counts, int vote_num,
                          int vote_den, int force_sink_last, int per_kv, int32_t *sel_idx,
                          int32_t *sel_page, int32_t *n_sel, cudaStream_t st);
cudaError_t launch_attention(const Geo &g, int nctas, const __nv_bfloat16 *q,
                             const __nv_bfloat16 *kcur, const __nv_bfloat16 *vcur,
                             const __nv_bfloat16 *kpool, const __nv_bfloat16 *vpool,
                             const int32_t *sel_page, const int32_t *n_sel, float scale,
                             __nv_bfloat16 *o, float *lse, float *part_o, float *part_lse,
                             int32_t *unit_cnt, cudaStream_t st);
cudaError_t launch_store_kv(const Geo &g, int max_blocks, const __nv_bfloat16 *kc,
                            const __nv_bfloat16 *vc, __nv_bfloat16 *kp, __nv_bfloat16 *vp,
                            cudaStream_t st);
cudaError_t launch_lse_merge(const float *o1, const float *l1, const float *o2, const float *l2,
                             int64_t rows, int D, void *o_out, int bf16_out, float *l_out,
                             cudaStream_t st);

}  // namespace xattn
