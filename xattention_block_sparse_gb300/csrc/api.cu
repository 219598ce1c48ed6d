// C ABI of libxattn: argument validation, per-request geometry, workspace
// layout and kernel launches.  See include/xattn.h for the contract.
#include <math.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <unordered_map>

#include "common.cuh"

namespace xattn {

// Device error word: the first fault a kernel finds (XATTN_EPAGE, ...).
__device__ int32_t g_err_word = 0;

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Plan {
  Geo geo;
  int gemm_tiles = 0, bsum_ctas = 0, sel_ctas = 0, att_ctas = 0;
  int max_kb = 0;
  size_t bs_count = 0;
  WsLayout ws{};
};

inline bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

// Validates the problem and fills the plan (host only; no CUDA calls).
xattn_status make_plan(const xattn_problem *p, Plan &pl) {
  if (!p) return XATTN_EINVAL;
  const int B = p->num_requests, H = p->num_heads, Hkv = p->num_kv_heads, D = p->head_dim,
            S = p->stride, Bk = p->block_size;
  if (B < 1 || B > kMaxReq || H < 1 || Hkv < 1 || H % Hkv != 0) return XATTN_EINVAL;
  if (D != 64 && D != 128) return XATTN_EUNSUPPORTED;
  if (S < 1 || S > 64 || Bk < 64 || Bk % 64 != 0 || Bk % S != 0) return XATTN_EUNSUPPORTED;
  const int br = Bk / S;
  if (!pow2(br) || br < 8 || br > 32) return XATTN_EUNSUPPORTED;
  if (!p->cu_seqlens_q || !p->cu_seqlens_kh) return XATTN_EINVAL;
  if (p->cu_seqlens_q[0] != 0) return XATTN_EINVAL;

  Geo &g = pl.geo;
  memset(&g, 0, sizeof(g));
  g.B = B;
  g.H = H;
  g.Hkv = Hkv;
  g.D = D;
  g.S = S;
  g.Bk = Bk;
  g.bt_stride = p->bt_stride;
  g.num_pages = p->num_pages;
  g.q_hs = p->q_head_stride;
  g.kv_hs = p->kv_head_stride;
  g.kv_ts = p->kv_token_stride > 0 ? p->kv_token_stride : D;
  g.kv_head_inner = g.kv_hs < g.kv_ts ? 1 : 0;
  g.lse_hs = p->lse_head_stride;
  g.H_all = H;
  g.Hkv_all = Hkv;
  g.block_table = p->block_table;

  int64_t gemm = 0, bsum = 0, sel = 0, att = 0;
  size_t bpart = 0, tstat = 0, bs = 0;
  bool any_hist = false;
  for (int r = 0; r < B; ++r) {
    const int64_t q0 = p->cu_seqlens_q[r], q1 = p->cu_seqlens_q[r + 1];
    const int64_t kh = (int64_t)p->cu_seqlens_kh[r + 1] - p->cu_seqlens_kh[r];
    const int64_t lq = q1 - q0;
    if (lq < 0 || kh < 0 || lq % Bk || kh % Bk) return XATTN_EINVAL;
    if (q1 > (int64_t)1 << 30 || kh > (int64_t)1 << 30) return XATTN_EINVAL;
    const int64_t kbh = kh / Bk, qb = lq / Bk;
    if (kbh + qb > XATTN_MAX_BLOCKS_PER_ROW) return XATTN_EUNSUPPORTED;
    if (kbh > 0) {
      any_hist = true;
      if (kbh > p->bt_stride) return XATTN_EINVAL;
    }
    ReqDesc &d = g.req[r];
    d.q0 = (int32_t)q0;
    d.lq = (int32_t)lq;
    d.kh = (int32_t)kh;
    d.gemm0 = (int32_t)gemm;
    d.bsum0 = (int32_t)bsum;
    d.sel0 = (int32_t)sel;
    d.att0 = (int32_t)att;
    d.hc = (int32_t)(kh / S);
    d.samp = 0;
    d.bpart_off = (int64_t)bpart;
    d.tstat_off = (int64_t)tstat;
    d.bs_off = (int64_t)bs;
    const int64_t rq = lq / S, ncol = (kh + lq) / S;
    const int64_t ntile = (ncol + kTileCols - 1) / kTileCols;
    if (lq > 0) {
      // score-GEMM tiles right of the causal diagonal are never visited
      int64_t per_head = 0;
      for (int64_t m0 = 0; m0 < rq; m0 += kGemmRows) {
        const int64_t last = (m0 + kGemmRows < rq ? m0 + kGemmRows : rq) - 1;
        const int64_t vis = (kh / S + last + 1 < ncol) ? kh / S + last + 1 : ncol;
        per_head += (vis + kGemmCols - 1) / kGemmCols;
      }
      gemm += (int64_t)H * per_head;
      bsum += (int64_t)H * qb;
      sel += (int64_t)Hkv * qb;
      att += (int64_t)H * ((lq + kAttnRows - 1) / kAttnRows);
    }
    bpart += (size_t)H * rq * (ncol / (Bk / S));  // one float per (reshaped row, KV block)
    tstat += (size_t)H * rq * ntile;
    bs += (size_t)H * qb * (kbh + qb);
    if (kbh + qb > pl.max_kb) pl.max_kb = (int)(kbh + qb);
  }
  if (gemm > INT32_MAX || bsum > INT32_MAX || att > INT32_MAX)
    return XATTN_EUNSUPPORTED;
  if (any_hist && (!p->block_table || p->num_pages < 1)) return XATTN_EINVAL;
  if (p->bt_stride < 0) return XATTN_EINVAL;
  const int64_t tot_q = p->cu_seqlens_q[B];
  if (p->q_head_stride < tot_q * D || p->lse_head_stride < tot_q) return XATTN_EINVAL;
  // k_cur / v_cur: heads apart by kv_head_stride, tokens by kv_token_stride,
  // either head-major [Hkv, tokens, D] or token-major [tokens, Hkv, D]
  if (p->kv_token_stride < 0) return XATTN_EINVAL;
  if (g.kv_ts < D || p->kv_head_stride < D) return XATTN_EINVAL;
  if (!(p->kv_head_stride >= tot_q * g.kv_ts || g.kv_ts >= (int64_t)Hkv * p->kv_head_stride))
    return XATTN_EINVAL;
  if (p->q_head_stride % 8 || p->kv_head_stride % 8 || g.kv_ts % 8) return XATTN_EALIGN;

  pl.gemm_tiles = (int)gemm;
  pl.bsum_ctas = (int)bsum;
  pl.sel_ctas = (int)sel;
  pl.att_ctas = (int)att;
  pl.bs_count = bs;
  WsLayout &w = pl.ws;
  w.bpart = 0;
  w.tstat = align_up(w.bpart + bpart * sizeof(float));
  w.counts = align_up(w.tstat + tstat * sizeof(float2));
  // attention partial results: two slots of kAttnRows rows per persistent CTA
  const size_t part_rows = (size_t)kAttnMaxCtas * 2 * kAttnRows;
  // vote counters of every (request, KV head) -- one row per request for the
  // vote across KV heads, one per KV head for the selection per KV head --
  // then the select kernel's finishing counter
  w.est = align_up(w.counts + ((size_t)B * Hkv * (size_t)(p->bt_stride > 0 ? p->bt_stride : 1) +
                               1) * sizeof(int32_t));
  // the attention's regions, relative to their block, which sits at the END of
  // the caller's buffer (run_attention): a chunk's estimate (the start of the
  // buffer) can then run beside the previous chunk's attention
  w.part_o = 0;
  w.part_lse = align_up(w.part_o + part_rows * D * sizeof(float));
  w.att_cnt = align_up(w.part_lse + part_rows * sizeof(float));
  w.attn = align_up(w.att_cnt + (size_t)att * 2 * sizeof(int32_t));  // two per attention unit
  w.total = w.est + w.attn + kAlign;  // + the slack that aligns the attention block
  return XATTN_OK;
}

inline bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; }

// Vote ratio num/den in [0, 1]; force flag 0 or 1.
inline bool vote_ok(int32_t num, int32_t den, int32_t force) {
  return den > 0 && num >= 0 && num <= den && (force == 0 || force == 1);
}

// Device address of the error word for the current device (cached per device).
std::atomic<int32_t *> g_err_addr[64];

xattn_status err_word(int32_t **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return XATTN_ECUDA;
  if (dev < 64) {
    int32_t *c = g_err_addr[dev].load(std::memory_order_acquire);
    if (c) {
      *out = c;
      return XATTN_OK;
    }
  }
  void *ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_err_word) != cudaSuccess) return XATTN_ECUDA;
  if (dev < 64) g_err_addr[dev].store(static_cast<int32_t *>(ptr), std::memory_order_release);
  *out = static_cast<int32_t *>(ptr);
  return XATTN_OK;
}

inline xattn_status cu(cudaError_t e) { return e == cudaSuccess ? XATTN_OK : XATTN_ECUDA; }

// The device range [lo, hi) of workspace that the last attention launched on
// a stream may still be using when the next kernel on that stream starts
// early (the attention lets its programmatic dependents start before it ends).
struct Range {
  uintptr_t lo, hi;
};
std::mutex g_attn_mu;
std::unordered_map<cudaStream_t, Range> g_attn_ws;

void note_attention(cudaStream_t st, const char *lo, const char *hi) {
  std::lock_guard<std::mutex> lk(g_attn_mu);
  g_attn_ws[st] = Range{reinterpret_cast<uintptr_t>(lo), reinterpret_cast<uintptr_t>(hi)};
}

// Whether a kernel writing [lo, hi) may start before the last attention on st
// has finished: no attention recorded, or its range is disjoint.
bool clear_of_attention(cudaStream_t st, const char *lo, const char *hi) {
  std::lock_guard<std::mutex> lk(g_attn_mu);
  auto it = g_attn_ws.find(st);
  if (it == g_attn_ws.end()) return true;
  const uintptr_t a = reinterpret_cast<uintptr_t>(lo), b = reinterpret_cast<uintptr_t>(hi);
  return b <= it->second.lo || a >= it->second.hi;
}

}  // namespace
}  // namespace xattn

// Vote counters of xattn_select_noalloc: a fixed array the library owns, for
// callers that cannot hand it any scratch.  Shared by every call on a device.
// (one more than the documented limit: the select kernel's finishing counter)
static __device__ __align__(256) int32_t xattn_noalloc_counters[XATTN_NOALLOC_MAX_COUNTERS + 1];

namespace xattn {
namespace {

// Device address of xattn_noalloc_counters for the current device, looked up
// once per device (the host-side symbol is not a device address).
std::atomic<int32_t *> g_noalloc_addr[64];

xattn_status noalloc_counters(int32_t **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return XATTN_ECUDA;
  if (dev < 64) {
    int32_t *c = g_noalloc_addr[dev].load(std::memory_order_acquire);
    if (c) {
      *out = c;
      return XATTN_OK;
    }
  }
  int32_t *ptr = nullptr;
  if (cudaGetSymbolAddress((void **)&ptr, xattn_noalloc_counters) != cudaSuccess || !ptr)
    return XATTN_ECUDA;
  if (dev < 64) g_noalloc_addr[dev].store(ptr, std::memory_order_release);
  *out = ptr;
  return XATTN_OK;
}

}  // namespace
}  // namespace xattn

using namespace xattn;

// Launches the estimation (score GEMM, then block sums) for a validated plan.
static xattn_status run_estimate(Plan &pl, const void *q, const void *k_cur, const void *k_pool,
                                 const KeySeq *kseq, float scale, void *workspace,
                                 size_t workspace_bytes, float *block_sums, cudaStream_t st) {
  xattn_status s;
  if (!isfinite(scale)) return XATTN_EINVAL;
  if (!aligned16(q) || !aligned16(workspace) || !aligned16(block_sums)) return XATTN_EALIGN;
  if (workspace_bytes < pl.ws.total) return XATTN_EWORKSPACE;
  if ((s = err_word(&pl.geo.err)) != XATTN_OK) return s;
  char *ws = static_cast<char *>(workspace);
  float *bpart = reinterpret_cast<float *>(ws + pl.ws.bpart);
  float2 *tstat = reinterpret_cast<float2 *>(ws + pl.ws.tstat);
  // the score GEMM writes [bpart, counts); it may overlap a previous attention
  // that is still finishing only if that attention's regions lie elsewhere
  const bool early = clear_of_attention(st, ws + pl.ws.bpart, ws + pl.ws.counts);
  s = cu(launch_score_gemm(pl.geo, pl.gemm_tiles, static_cast<const __nv_bfloat16 *>(q),
                           static_cast<const __nv_bfloat16 *>(k_cur),
                           static_cast<const __nv_bfloat16 *>(k_pool), kseq, scale, bpart, tstat,
                           early, st));
  if (s != XATTN_OK) return s;
  return cu(launch_block_sum(pl.geo, pl.bsum_ctas, bpart, tstat, block_sums, st));
}

// Checks shared by the selection entry points; counters come from the caller.
static xattn_status check_select(const xattn_problem *p, const float *block_sums,
                                 double threshold, int32_t vote_num, int32_t vote_den,
                                 int32_t force_sink_last, const int32_t *sel_idx,
                                 const int32_t *sel_page, const int32_t *n_sel) {
  if (!block_sums || !sel_idx || !sel_page || !n_sel) return XATTN_EINVAL;
  if (!(threshold > 0.0) || !isfinite(threshold)) return XATTN_EINVAL;
  if (!vote_ok(vote_num, vote_den, force_sink_last)) return XATTN_EINVAL;
  if (p->bt_stride < 1) return XATTN_EINVAL;
  if (reinterpret_cast<uintptr_t>(block_sums) & 3) return XATTN_EALIGN;
  return XATTN_OK;
}

// Clears `rows` counter rows of bt_stride (plus the finishing counter) on the
// stream and launches the selection.
static xattn_status run_select(Plan &pl, const xattn_problem *p, const float *block_sums,
                               double threshold, int32_t vote_num, int32_t vote_den,
                               int32_t force_sink_last, int32_t *counts, int per_kv,
                               uint8_t *mask, int32_t *sel_idx, int32_t *sel_page,
                               int32_t *n_sel, cudaStream_t st) {
  xattn_status s;
  if ((s = err_word(&pl.geo.err)) != XATTN_OK) return s;
  const size_t rows = (size_t)pl.geo.B * (per_kv ? (size_t)pl.geo.Hkv : 1);
  bool any_hist = false;
  for (int r = 0; r < pl.geo.B; ++r) any_hist = any_hist || pl.geo.req[r].kh > 0;
  if (!any_hist && !mask)  // no history block to select and no mask asked for:
    return cu(cudaMemsetAsync(n_sel, 0, rows * sizeof(int32_t), st));  // every list is empty
  s = cu(cudaMemsetAsync(counts, 0, (rows * (size_t)p->bt_stride + 1) * sizeof(int32_t), st));
  if (s != XATTN_OK) return s;
  return cu(launch_select(pl.geo, pl.sel_ctas, pl.max_kb, block_sums, threshold, mask, counts,
                          vote_num, vote_den, force_sink_last, per_kv, sel_idx, sel_page, n_sel,
                          st));
}

// Launches the attention of a validated plan; per_kv: the selection holds one
// page list per (request, KV head), and each request's KV-head groups run as
// requests of their own (G query heads, one KV head).
// The address kernels write an output through: device (or managed) memory as
// given; page-locked host memory (cudaHostAlloc, cudaMallocHost, or
// cudaHostRegister'd) through its device alias, so the kernel's stores cross
// the host link as they are made; anything else (pageable host memory) is
// refused.
static xattn_status output_address(void *ptr, void **dev) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
    cudaGetLastError();  // leave no error behind for the caller's next check
    return XATTN_EINVAL;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
    *dev = ptr;
    return XATTN_OK;
  }
  if (a.type == cudaMemoryTypeHost && a.devicePointer) {
    *dev = a.devicePointer;
    return XATTN_OK;
  }
  return XATTN_EINVAL;
}

static xattn_status run_attention(Plan &pl, const xattn_problem *p, const void *q,
                                  const void *k_cur, const void *v_cur, const void *k_pool,
                                  const void *v_pool, const int32_t *sel_page,
                                  const int32_t *n_sel, float softmax_scale, void *workspace,
                                  size_t workspace_bytes, void *o, float *lse, int per_kv,
                                  cudaStream_t st) {
  xattn_status s;
  if (!q || !k_cur || !v_cur || !sel_page || !n_sel || !o || !lse || !workspace)
    return XATTN_EINVAL;
  if ((!k_pool || !v_pool) && pl.geo.num_pages > 0) return XATTN_EINVAL;
  if (p->bt_stride < 1) return XATTN_EINVAL;
  if (!isfinite(softmax_scale) || !(softmax_scale > 0.f)) return XATTN_EINVAL;
  if (!aligned16(q) || !aligned16(k_cur) || !aligned16(v_cur) || !aligned16(o) ||
      (k_pool && !aligned16(k_pool)) || (v_pool && !aligned16(v_pool)) || !aligned16(workspace))
    return XATTN_EALIGN;
  if (workspace_bytes < pl.ws.total) return XATTN_EWORKSPACE;
  if ((s = err_word(&pl.geo.err)) != XATTN_OK) return s;
  void *o_dev = nullptr, *lse_dev = nullptr;
  if ((s = output_address(o, &o_dev)) != XATTN_OK) return s;
  if ((s = output_address(lse, &lse_dev)) != XATTN_OK) return s;
  Geo g = pl.geo;
  if (per_kv) {
    // request r, KV head k -> request r * Hkv + k with the G query heads of
    // the group; its selection row is r * Hkv + k of sel_page / n_sel
    const int B = g.B, Hkv = g.Hkv, G = g.H / g.Hkv;
    if ((int64_t)B * Hkv > kMaxReq) return XATTN_EUNSUPPORTED;
    int att = 0;
    for (int r = B - 1; r >= 0; --r)
      for (int k = Hkv - 1; k >= 0; --k) g.req[r * Hkv + k] = pl.geo.req[r];
    for (int v = 0; v < B * Hkv; ++v) {
      ReqDesc &d = g.req[v];
      d.head0 = (v % Hkv) * G;
      d.kvh0 = v % Hkv;
      d.att0 = att;
      att += G * ((d.lq + kAttnRows - 1) / kAttnRows);
    }
    g.B = B * Hkv;
    g.H = G;
    g.Hkv = 1;
  }
  // the attention's regions at the end of the buffer (see make_plan), the block
  // 256-byte aligned in memory (its partial rows take 32-byte stores)
  char *ws = reinterpret_cast<char *>(
      (reinterpret_cast<uintptr_t>(workspace) + workspace_bytes - pl.ws.attn) &
      ~(uintptr_t)(kAlign - 1));
  note_attention(st, ws, static_cast<char *>(workspace) + workspace_bytes);
  return cu(launch_attention(g, pl.att_ctas, static_cast<const __nv_bfloat16 *>(q),
                             static_cast<const __nv_bfloat16 *>(k_cur),
                             static_cast<const __nv_bfloat16 *>(v_cur),
                             static_cast<const __nv_bfloat16 *>(k_pool),
                             static_cast<const __nv_bfloat16 *>(v_pool), sel_page, n_sel,
                             softmax_scale, static_cast<__nv_bfloat16 *>(o_dev),
                             static_cast<float *>(lse_dev),
                             reinterpret_cast<float *>(ws + pl.ws.part_o),
                             reinterpret_cast<float *>(ws + pl.ws.part_lse),
                             reinterpret_cast<int32_t *>(ws + pl.ws.att_cnt), st));
}

// The estimation over keys in token order, every history column scored
// (samples == 0) or the first `samples` reshaped columns of each history block.
static xattn_status estimate_keys(const xattn_problem *p, const void *q, const void *k_seq,
                                  int64_t k_seq_head_stride, int64_t k_seq_token_stride,
                                  const int64_t *k_seq_start, int32_t samples, float scale,
                                  void *workspace, size_t workspace_bytes, float *block_sums,
                                  xattn_stream_t stream) {
  Plan pl;
  xattn_status s = make_plan(p, pl);
  if (s != XATTN_OK) return s;
  if (!q || !k_seq || !k_seq_start || !workspace || !block_sums) return XATTN_EINVAL;
  const int D = p->head_dim, S = p->stride, Hkv = p->num_kv_heads, Bk = p->block_size;
  const int br = Bk / S;
  const int64_t hs = k_seq_head_stride, ts = k_seq_token_stride > 0 ? k_seq_token_stride : D;
  if (k_seq_token_stride < 0 || hs < D || ts < D) return XATTN_EINVAL;
  if (!aligned16(k_seq) || hs % 8 || ts % 8) return XATTN_EALIGN;
  if (samples != 0 && !(samples >= 4 && (samples * 4 == br || samples * 2 == br)))
    return XATTN_EUNSUPPORTED;
  int64_t end = 0;
  for (int r = 0; r < p->num_requests; ++r) {
    const int64_t st0 = k_seq_start[r];
    const ReqDesc &d = pl.geo.req[r];
    if (st0 < 0 || st0 % (samples ? Bk : S)) return XATTN_EINVAL;
    if (st0 / S + (int64_t)(d.kh + d.lq) / S > INT32_MAX) return XATTN_EINVAL;
    pl.geo.req[r].ks0 = (int32_t)(st0 / S);
    if (st0 + d.kh + d.lq > end) end = st0 + d.kh + d.lq;
  }
  // the two views of the keys must not overlap: head-major or token-major
  if (Hkv > 1 && !(hs >= end * ts || ts >= (int64_t)Hkv * hs)) return XATTN_EINVAL;
  if (samples) {
    // a request samples its history when that leaves fewer columns: the
    // sampled columns, padded to a statistics tile, before the chunk's; the
    // score tiles are counted again on that layout
    Geo &g = pl.geo;
    g.ns = samples;
    int64_t gemm = 0;
    for (int r = 0; r < g.B; ++r) {
      ReqDesc &d = g.req[r];
      const int kbh = d.kh / Bk, rq = d.lq / S, ch = d.kh / S;
      const int hc = (kbh * samples + kTileCols - 1) / kTileCols * kTileCols;
      d.samp = hc < ch ? 1 : 0;
      d.hc = d.samp ? hc : ch;
      d.gemm0 = (int32_t)gemm;
      int64_t per_head = 0;
      for (int m0 = 0; m0 < rq; m0 += kGemmRows) {
        const int last = (m0 + kGemmRows < rq ? m0 + kGemmRows : rq);
        const int vis = d.hc + last;
        per_head += (vis + kGemmCols - 1) / kGemmCols;
      }
      if (d.lq > 0) gemm += (int64_t)g.H * per_head;
    }
    pl.gemm_tiles = (int)gemm;
  }
  const KeySeq ks{static_cast<const __nv_bfloat16 *>(k_seq), hs, ts};
  return run_estimate(pl, q, nullptr, nullptr, &ks, scale, workspace, workspace_bytes,
                      block_sums, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" {

size_t xattn_workspace_size(const xattn_problem *p) {
  Plan pl;
  if (make_plan(p, pl) != XATTN_OK) return 0;
  return pl.ws.total;
}

size_t xattn_block_sums_count(const xattn_problem *p) {
  Plan pl;
  if (make_plan(p, pl) != XATTN_OK) return 0;
  return pl.bs_count;
}

size_t xattn_block_sums_offset(const xattn_problem *p, int32_t r) {
  Plan pl;
  if (make_plan(p, pl) != XATTN_OK || r < 0 || r >= p->num_requests) return 0;
  return (size_t)pl.geo.req[r].bs_off;
}

xattn_status xattn_estimate(const xattn_problem *p, const void *q, const void *k_cur,
                            const void *k_pool, float scale, void *workspace,
                            size_t workspace_bytes, float *block_sums, xattn_stream_t stream) {
  Plan pl;
  xattn_status s = make_plan(p, pl);
  if (s != XATTN_OK) return s;
  if (!q || !k_cur || !workspace || !block_sums) return XATTN_EINVAL;
  if (!k_pool && pl.geo.num_pages > 0) return XATTN_EINVAL;
  if (!aligned16(k_cur) || (k_pool && !aligned16(k_pool))) return XATTN_EALIGN;
  return run_estimate(pl, q, k_cur, k_pool, nullptr, scale, workspace, workspace_bytes,
                      block_sums, reinterpret_cast<cudaStream_t>(stream));
}

xattn_status xattn_estimate_seq(const xattn_problem *p, const void *q, const void *k_seq,
                                int64_t k_seq_head_stride, int64_t k_seq_token_stride,
                                const int64_t *k_seq_start, float scale, void *workspace,
                                size_t workspace_bytes, float *block_sums,
                                xattn_stream_t stream) {
  return estimate_keys(p, q, k_seq, k_seq_head_stride, k_seq_token_stride, k_seq_start, 0, scale,
                       workspace, workspace_bytes, block_sums, stream);
}

xattn_status xattn_estimate_sampled(const xattn_problem *p, const void *q, const void *k_seq,
                                    int64_t k_seq_head_stride, int64_t k_seq_token_stride,
                                    const int64_t *k_seq_start, int32_t samples, float scale,
                                    void *workspace, size_t workspace_bytes, float *block_sums,
                                    xattn_stream_t stream) {
  if (samples <= 0) return XATTN_EINVAL;
  return estimate_keys(p, q, k_seq, k_seq_head_stride, k_seq_token_stride, k_seq_start, samples,
                       scale, workspace, workspace_bytes, block_sums, stream);
}

xattn_status xattn_select(const xattn_problem *p, const float *block_sums, double threshold,
                          int32_t vote_num, int32_t vote_den, int32_t force_sink_last,
                          void *workspace, size_t workspace_bytes, uint8_t *mask,
                          int32_t *sel_idx, int32_t *sel_page, int32_t *n_sel,
                          xattn_stream_t stream) {
  Plan pl;
  xattn_status s = make_plan(p, pl);
  if (s != XATTN_OK) return s;
  if (!workspace) return XATTN_EINVAL;
  if ((s = check_select(p, block_sums, threshold, vote_num, vote_den, force_sink_last, sel_idx,
                        sel_page, n_sel)) != XATTN_OK)
    return s;
  if (!aligned16(workspace)) return XATTN_EALIGN;
  if (workspace_bytes < pl.ws.total) return XATTN_EWORKSPACE;
  int32_t *counts = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + pl.ws.counts);
  return run_select(pl, p, block_sums, threshold, vote_num, vote_den, force_sink_last, counts, 0,
                    mask, sel_idx, sel_page, n_sel, reinterpret_cast<cudaStream_t>(stream));
}

xattn_status xattn_select_per_kv_head(const xattn_problem *p, const float *block_sums,
                                      double threshold, int32_t vote_num, int32_t vote_den,
                                      int32_t force_sink_last, void *workspace,
                                      size_t workspace_bytes, uint8_t *mask, int32_t *sel_idx,
                                      int32_t *sel_page, int32_t *n_sel, xattn_stream_t stream) {
  Plan pl;
  xattn_status s = make_plan(p, pl);
  if (s != XATTN_OK) return s;
  if (!workspace) return XATTN_EINVAL;
  if ((s = check_select(p, block_sums, threshold, vote_num, vote_den, force_sink_last, sel_idx,
                        sel_page, n_sel)) != XATTN_OK)
    return s;
  if (!aligned16(workspace)) return XATTN_EALIGN;
  if (workspace_bytes < pl.ws.total) return XATTN_EWORKSPACE;
  int32_t *counts = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + pl.ws.counts);
  return run_select(pl, p, block_sums, threshold, vote_num, vote_den, force_sink_last, counts, 1,
                    mask, sel_idx, sel_page, n_sel, reinterpret_cast<cudaStream_t>(stream));
}

xattn_status xattn_select_noalloc(const xattn_problem *p, const float *block_sums,
                                  double threshold, int32_t vote_num, int32_t vote_den,
                                  int32_t force_sink_last, uint8_t *mask, int32_t *sel_idx,
                                  int32_t *sel_page, int32_t *n_sel, xattn_stream_t stream) {
  Plan pl;
  xattn_status s = make_plan(p, pl);
  if (s != XATTN_OK) return s;
  if ((s = check_select(p, block_sums, threshold, vote_num, vote_den, force_sink_last, sel_idx,
                        sel_page, n_sel)) != XATTN_OK)
    return s;
  const size_t n_counters = (size_t)pl.geo.B * (size_t)p->bt_stride;
  if (n_counters > (size_t)XATTN_NOALLOC_MAX_COUNTERS) return XATTN_EWORKSPACE;
  int32_t *counts = nullptr;
  if ((s = noalloc_counters(&counts)) != XATTN_OK) return s;
  // the array keeps the previous call's votes: run_select clears the part
  // this call uses
  return run_select(pl, p, block_sums, threshold, vote_num, vote_den, force_sink_last, counts, 0,
                    mask, sel_idx, sel_page, n_sel, reinterpret_cast<cudaStream_t>(stream));
}

xattn_status bsa_chunk_attention(const xattn_problem *p, const void *q, const void *k_cur,
                                 const void *v_cur, const void *k_pool, const void *v_pool,
                                 const int32_t *sel_page, const int32_t *n_sel,
                                 float softmax_scale, void *workspace, size_t workspace_bytes,
                                 void *o, float *lse, xattn_stream_t stream) {
  Plan pl;
  xattn_status s = make_plan(p, pl);
  if (s != XATTN_OK) return s;
  return run_attention(pl, p, q, k_cur, v_cur, k_pool, v_pool, sel_page, n_sel, softmax_scale,
                       workspace, workspace_bytes, o, lse, 0,
                       reinterpret_cast<cudaStream_t>(stream));
}

xattn_status bsa_chunk_attention_per_kv_head(const xattn_problem *p, const void *q,
                                             const void *k_cur, const void *v_cur,
                                             const void *k_pool, const void *v_pool,
                                             const int32_t *sel_page, const int32_t *n_sel,
                                             float softmax_scale, void *workspace,
                                             size_t workspace_bytes, void *o, float *lse,
                                             xattn_stream_t stream) {
  Plan pl;
  xattn_status s = make_plan(p, pl);
  if (s != XATTN_OK) return s;
  return run_attention(pl, p, q, k_cur, v_cur, k_pool, v_pool, sel_page, n_sel, softmax_scale,
                       workspace, workspace_bytes, o, lse, 1,
                       reinterpret_cast<cudaStream_t>(stream));
}

xattn_status lse_merge(const float *o1, const float *lse1, const float *o2, const float *lse2,
                       int64_t rows, int32_t head_dim, void *o_out, int32_t o_out_bf16,
                       float *lse_out, xattn_stream_t stream) {
  if (rows < 0 || head_dim < 4 || head_dim % 4 != 0) return XATTN_EINVAL;
  if (rows == 0) return XATTN_OK;
  if (!o1 || !lse1 || !o2 || !lse2 || !o_out || !lse_out) return XATTN_EINVAL;
  if (!aligned16(o1) || !aligned16(o2) || !aligned16(o_out)) return XATTN_EALIGN;
  if (o_out_bf16 && head_dim % 8 != 0) return XATTN_EALIGN;
  return cu(launch_lse_merge(o1, lse1, o2, lse2, rows, head_dim, o_out, o_out_bf16 ? 1 : 0,
                             lse_out, reinterpret_cast<cudaStream_t>(stream)));
}

xattn_status xattn_store_kv(const xattn_problem *p, const void *k_cur, const void *v_cur,
                            void *k_pool, void *v_pool, xattn_stream_t stream) {
  Plan pl;
  xattn_status s = make_plan(p, pl);
  if (s != XATTN_OK) return s;
  if (!k_cur || !v_cur || !k_pool || !v_pool || !p->block_table || p->num_pages < 1)
    return XATTN_EINVAL;
  if (!aligned16(k_cur) || !aligned16(v_cur) || !aligned16(k_pool) || !aligned16(v_pool))
    return XATTN_EALIGN;
  int max_blocks = 0;
  for (int r = 0; r < p->num_requests; ++r) {
    const ReqDesc &d = pl.geo.req[r];
    if ((int64_t)(d.kh + d.lq) / p->block_size > p->bt_stride) return XATTN_EINVAL;
    if (d.lq / p->block_size > max_blocks) max_blocks = d.lq / p->block_size;
  }
  if ((s = err_word(&pl.geo.err)) != XATTN_OK) return s;
  return cu(launch_store_kv(pl.geo, max_blocks, static_cast<const __nv_bfloat16 *>(k_cur),
                            static_cast<const __nv_bfloat16 *>(v_cur),
                            static_cast<__nv_bfloat16 *>(k_pool),
                            static_cast<__nv_bfloat16 *>(v_pool),
                            reinterpret_cast<cudaStream_t>(stream)));
}

xattn_status xattn_device_error(xattn_stream_t stream, int32_t *code, int32_t clear) {
  if (!code) return XATTN_EINVAL;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return XATTN_ECUDA;
  int32_t v = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_word, sizeof(v)) != cudaSuccess) return XATTN_ECUDA;
  if (clear) {
    const int32_t z = 0;
    if (cudaMemcpyToSymbol(g_err_word, &z, sizeof(z)) != cudaSuccess) return XATTN_ECUDA;
  }
  *code = v;
  return XATTN_OK;
}

xattn_status xattn_copy_rows_async(void *dst, int64_t dst_pitch, const void *src, int64_t src_pitch,
                                   int64_t width_bytes, int64_t rows, int32_t to_device,
                                   xattn_stream_t stream) {
  if (width_bytes < 0 || rows < 0 || dst_pitch < width_bytes || src_pitch < width_bytes)
    return XATTN_EINVAL;
  if (width_bytes == 0 || rows == 0) return XATTN_OK;
  if (!dst || !src) return XATTN_EINVAL;
  return cu(cudaMemcpy2DAsync(dst, (size_t)dst_pitch, src, (size_t)src_pitch, (size_t)width_bytes,
                              (size_t)rows,
                              to_device ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToHost,
                              reinterpret_cast<cudaStream_t>(stream)));
}

xattn_status xattn_last_device_error(xattn_stream_t stream, int32_t *host_code) {
  return xattn_device_error(stream, host_code, 1);
}

const char *xattn_status_string(xattn_status s) {
  switch (s) {
    case XATTN_OK: return "ok";
    case XATTN_EINVAL: return "invalid argument";
    case XATTN_EALIGN: return "pointer or stride not 16-byte aligned";
    case XATTN_EPAGE: return "page id outside the pool";
    case XATTN_ECUDA: return "CUDA runtime error";
    case XATTN_EUNSUPPORTED: return "unsupported geometry";
    case XATTN_EWORKSPACE: return "workspace too small";
    case XATTN_ETIMEOUT: return "kernel pipeline wait timed out";
  }
  return "unknown status";
}

}  // extern "C"
