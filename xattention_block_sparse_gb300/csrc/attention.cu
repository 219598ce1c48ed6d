// Block-sparse chunk attention of XAttention BSA ("XAttention BSA Policy 设计文档",
// compute_chunked_prefill): softmax attention of the current query chunk over
// the selected history pages (non-causal) and the current chunk (causal),
// merged online by log-sum-exp in one pass -- the result equals
// flash_attn_with_lse(history) merged with flash_attn_with_lse(current, causal)
// by merge_attention_outputs.
//
// Work decomposition (stream-K).  A work unit is 256 query rows -- tiles A
// and B of 128 rows -- of one (request, head); its work items are the KV tiles
// it attends (selected history pages, then the current chunk up to the unit's
// last row).  The items of all units, in (request, head, row tile, KV tile)
// order, are split into one equal contiguous range per persistent CTA (one
// CTA per SM), so every SM gets the same number of KV tiles.  A CTA walks its
// range as segments (a unit, or the piece of one that falls in its range).
// A unit cut between CTAs leaves normalised partial results (fp32 O, LSE);
// the last CTA to finish a part (a per-unit counter) merges them by
// log-sum-exp into the final O and LSE.
//
// tcgen05 pipeline of one CTA (two query tiles A and B share every K/V tile):
//   warp 0        TMA producer: Q_A, Q_B of each segment (as soon as the
//                 previous segment's last S MMA on that tile has completed),
//                 then K(t), V(t) for each KV tile t (one page of up to 128
//                 keys) through a 5-slot ring of 128B-swizzled tiles.
//   warps 1, 2    MMA issuers of tiles A and B, taking turns so the pipe
//                 sees S_A(0), S_B(0), PV_A(t), S_A(t+1), PV_B(t), S_B(t+1), ...:
//                 S_x = Q_x K^T into TMEM (128 lanes x NK fp32 columns),
//                 O_x += P_x V into a TMEM accumulator with P_x read from TMEM.
//                 While the softmax of one tile runs, the pipe works for the
//                 other; each issuer waits on its barriers during the other's turn.
//   warps 4..7    softmax of tile A, warps 8..11 softmax of tile B: thread i
//                 owns query row i (TMEM lane i).  It loads its S row, masks
//                 the causal diagonal tile, keeps a running max (rescaling O in
//                 TMEM only when the max grows by more than 2^8), writes P as
//                 bf16 back into the TMEM columns its S row came from, and at
//                 the end of a segment normalises O and writes it (256-bit
//                 stores, one full 32-byte sector per thread and instruction).
// Each thread's tcgen05 ops complete in issue order: S_x(t) being ready
// implies PV_x(t-1) has finished, so O_x may be rescaled and S_x's columns
// reused for P_x(t) without further waits.
// Every mbarrier wait is bounded; a timeout records XATTN_ETIMEOUT and the CTA
// unwinds (draining its TMA loads and MMAs, then freeing TMEM).  No CTA waits
// for another: the merge of a split unit is done by whichever CTA finishes its
// part last.
#include <stdlib.h>
#include <string.h>

#include "tc_common.cuh"

namespace xattn {
namespace {
using namespace tc;

constexpr int BM = 128;       // rows per query tile (MMA M)
constexpr int ROWS = 2 * BM;  // query rows per work unit
static_assert(ROWS == kAttnRows, "partial-output slots assume kAttnRows rows per unit");
constexpr int NSLOT = 5;      // K/V ring slots
constexpr int kMaxWaves = 8;  // waves of whole units before the stream-K part
constexpr int kStreamK = 0, kWholeUnits = 1, kWaves = 2;
constexpr int THREADS = 384;
constexpr int TMEM_COLS = 512;  // S_A | S_B | O_A | O_B, 128 columns each

template <int D, int NK>
struct Layout {
  static constexpr int HALVES = D / 64;  // 64-element (128 B) column blocks
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int KV_BYTES = NK * D * 2;
  static constexpr int OFF_Q = 0;                       // Q_A, Q_B
  static constexpr int OFF_KV = OFF_Q + 2 * Q_BYTES;    // ring
  static constexpr int OFF_BAR = OFF_KV + NSLOT * KV_BYTES;
  static constexpr int BYTES = OFF_BAR + 2048;
  static constexpr int SMEM_ALLOC = BYTES + 1024;  // slack to align the base to 1024
};

struct Bars {
  uint64_t q_full[2], q_empty[2];
  uint64_t full[NSLOT];
  uint64_t empty[NSLOT];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t pv_done[2];
  uint64_t drain;
  uint64_t grp[2];                 // barrier of one softmax warpgroup (4 warp arrivals)
  uint64_t tok[2];                 // MMA issuer turn tokens (tile A's, tile B's)
  uint32_t tmem_base;
  int abort;
  int last[2];                     // this CTA merges the unit (per query tile)
  int64_t total;                   // work items (KV tiles over all units)
  int64_t req_pos0[kMaxReq + 1];   // first work item of each request
  int32_t req_hist[kMaxReq];       // history KV tiles of the request (selected pages)
  int32_t req_per_head[kMaxReq];   // work items per head of the request
  int32_t req_unit0[kMaxReq];      // first unit id of the request
  int32_t max_unit;                // largest unit (KV tiles)
  int32_t nunits;                  // units of the launch
  int32_t mode;                    // schedule: kStreamK, kWholeUnits or kWaves
  int32_t nw;                      // kWaves: waves of whole units before stream-K
  int32_t nrg;                     // this CTA's ranges of work items
  int64_t rg_beg[kMaxWaves + 1];   // the ranges: its units of each wave (whole),
  int64_t rg_end[kMaxWaves + 1];   //   then its stream-K range (the last one)
  int64_t p_waves;                 // kWaves: first item after the waves' units
  int64_t sk_q;                    // total = sk_q * Gsk + sk_r: floor(c total / Gsk)
  int32_t sk_r;                    //   without a 64-bit division
  int32_t csk;                     // stream-K CTA index, -1 if this CTA has no range
};

struct TMaps {
  CUtensorMap q, kc, vc, kp, vp;
};

struct Unit {
  int n_a, n_b, n_tiles;  // tiles of query tile A, of B, and of the unit
  bool has_b;
};

template <int NK>
__device__ __forceinline__ Unit unit_geom(const ReqDesc &R, int n_hist, int mt) {
  Unit u;
  const int m0 = mt * ROWS;
  u.has_b = m0 + BM < R.lq;
  u.n_a = n_hist + (min(m0 + BM, R.lq) - 1) / NK + 1;
  u.n_b = u.has_b ? n_hist + (min(m0 + ROWS, R.lq) - 1) / NK + 1 : 0;
  u.n_tiles = u.has_b ? u.n_b : u.n_a;
  return u;
}

// Work-item tables of the launch, from the selection counts on the device
// (every CTA computes the same tables: no host round trip).
template <int NK>
__device__ __noinline__ void build_tables(const Geo &g, const int32_t *n_sel, Bars &bar) {
  int64_t pos = 0;
  int32_t unit = 0;
  const int sub = g.Bk / NK;
  bar.max_unit = 0;
  for (int r = 0; r < g.B; ++r) {
    const ReqDesc &R = g.req[r];
    const int kbh = R.kh / g.Bk;
    int nh = n_sel[r];
    nh = nh < 0 ? 0 : (nh > kbh ? kbh : nh);
    const int n_hist = nh * sub;
    int per_head = 0, nmt = 0;
    for (int mt = 0; mt * ROWS < R.lq; ++mt, ++nmt) {
      const int n = unit_geom<NK>(R, n_hist, mt).n_tiles;
      per_head += n;
      bar.max_unit = max(bar.max_unit, n);
    }
    bar.req_pos0[r] = pos;
    bar.req_hist[r] = n_hist;
    bar.req_per_head[r] = per_head;
    bar.req_unit0[r] = unit;
    pos += (int64_t)per_head * g.H;
    unit += nmt * g.H;
  }
  bar.req_pos0[g.B] = pos;
  bar.total = pos;
  bar.nunits = unit;
}

// First work item of unit u (units in item order: request, head, row tile);
// the total for u = nunits.
template <int NK>
__device__ __noinline__ int64_t unit_start(const Geo &g, const Bars &bar, int u) {
  if (u >= bar.nunits) return bar.total;
  int r = 0;
  while (r + 1 < g.B && u >= bar.req_unit0[r + 1]) ++r;
  const ReqDesc &R = g.req[r];
  const int nmt = (R.lq + ROWS - 1) / ROWS;
  const int l = u - bar.req_unit0[r];
  const int h = l / nmt, mt = l % nmt;
  int64_t pos = bar.req_pos0[r] + (int64_t)h * bar.req_per_head[r];
  for (int m = 0; m < mt; ++m) pos += unit_geom<NK>(R, bar.req_hist[r], m).n_tiles;
  return pos;
}

// First stream-K item of CTA c of the G stream-K CTAs.  kStreamK: the items
// split evenly.  kWaves: CTA c first runs units c, c + G, ..., c + (nw-1) G
// whole, then the items after the waves' nw G units are split so that every
// CTA's parts add up to the same total:
//   B_c = P(nw G) + floor(c T / G) - sum_w (P(w G + c) - P(w G)),
// P(u) the first item of unit u (needs nw * the longest unit <= T / G, so
// that no CTA's share is negative).
__device__ __forceinline__ int64_t share_floor(const Bars &bar, int c, int G) {
  return bar.sk_q * c + (bar.sk_r * c) / G;  // floor(c total / G); sk_r * c < G * (G + 1)
}

template <int NK>
__device__ __noinline__ int64_t cta_begin_waves(const Geo &g, const Bars &bar, int c, int G) {
  if (c >= G) return bar.total;
  int64_t b = bar.p_waves + share_floor(bar, c, G);
  for (int w = 0; w < bar.nw; ++w)
    b -= unit_start<NK>(g, bar, w * G + c) - unit_start<NK>(g, bar, w * G);
  return b;
}

template <int NK>
__device__ __forceinline__ int64_t cta_begin(const Geo &g, const Bars &bar, int c, int G) {
  return bar.mode != kWaves ? share_floor(bar, c, G) : cta_begin_waves<NK>(g, bar, c, G);
}

// The stream-K CTA whose range holds item `pos` (the last c with B_c <= pos;
// ranges may be empty).
template <int NK>
__device__ __noinline__ int cta_of(const Geo &g, const Bars &bar, int G, int64_t pos) {
  if (bar.mode != kWaves) {  // even split: the proportional guess (float, off by at
    // most one), then exact integer steps
    int c = (int)((float)pos * ((float)G / (float)bar.total));
    c = c < 0 ? 0 : (c > G - 1 ? G - 1 : c);
    while (c + 1 < G && share_floor(bar, c + 1, G) <= pos) ++c;
    while (c > 0 && share_floor(bar, c, G) > pos) --c;
    return c;
  }
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if (cta_begin<NK>(g, bar, mid, G) <= pos)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// The work of CTA blockIdx.x.  Three schedules, chosen from the tables alone
// (every CTA takes the same decision):
//  * whole units: CTA c takes unit c of the units ordered by their distance
//    from their request's last row tile (the larger units first, across
//    requests: one request per KV head when each KV head has its own
//    selection), then by request and head, the hardware handing
//    out CTAs as SMs free up -- no unit is split, no merge; used when the
//    launch is small (under kWholeUnitsTiles items per SM) and no unit
//    dwarfs a fair share, where stream-K's segment changes and merges cost
//    more than the imbalance they remove (at the 32K workload's chunks of 83
//    and 136 items per SM, one CTA per unit measured 188 against 202 us and
//    300 against 290 us);
//  * waves (when the caller allows it: keys and values larger than L2): the
//    stream-K CTAs first run nw waves of whole units -- CTA c units c, c + G,
//    ... -- then stream-K ranges of the remaining units sized so that all
//    CTAs carry the same total.  A wave's units are consecutive -- the query
//    heads of a few KV heads -- and start at their first KV page together, so
//    each page comes from DRAM once and from L2 to the other CTAs reading it,
//    where stream-K CTAs at unrelated positions would each fetch their own;
//  * stream-K: the last Gsk CTAs of the grid split the items evenly.
constexpr int kWholeUnitsTiles = 110;
template <int NK>
__device__ __noinline__ void schedule(const Geo &g, Bars &bar, int Gsk, int waves_ok) {
  const int64_t total = bar.total;
  const int grid = gridDim.x, c = blockIdx.x;
  const int64_t share = (total + Gsk - 1) / Gsk;
  const bool whole = share < kWholeUnitsTiles && 4 * (int64_t)bar.max_unit <= 5 * share;
  int nw = 0;
  if (!whole && waves_ok) {
    nw = min(bar.nunits / Gsk, kMaxWaves);
    while (nw > 0 && (int64_t)nw * bar.max_unit * Gsk > total) --nw;
  }
  bar.mode = whole ? kWholeUnits : (nw > 0 ? kWaves : kStreamK);
  bar.nw = nw;
  bar.sk_q = total / Gsk;
  bar.sk_r = (int32_t)(total - bar.sk_q * Gsk);
  bar.nrg = 0;
  bar.csk = -1;
  if (bar.mode == kWholeUnits) {
    // rank c: units by their distance d from their request's last row tile
    // (the larger units first, across requests), then request, then head
    if (c >= bar.nunits) return;  // past the last unit
    int l = c, d = 0, r = -1;
    while (r < 0) {
      int level = 0;
      for (int q = 0; q < g.B; ++q) level += (g.req[q].lq + ROWS - 1) / ROWS > d ? g.H : 0;
      if (l < level) {
        for (int q = 0; r < 0; ++q) {
          if ((g.req[q].lq + ROWS - 1) / ROWS <= d) continue;
          if (l < g.H) r = q; else l -= g.H;
        }
      } else {
        l -= level;
        ++d;
      }
    }
    const ReqDesc &R = g.req[r];
    const int nmt = (R.lq + ROWS - 1) / ROWS;
    const int mt = nmt - 1 - d, h = l;
    int64_t pos = bar.req_pos0[r] + (int64_t)h * bar.req_per_head[r];
    for (int m = 0; m < mt; ++m) pos += unit_geom<NK>(R, bar.req_hist[r], m).n_tiles;
    bar.rg_beg[0] = pos;
    bar.rg_end[0] = pos + unit_geom<NK>(R, bar.req_hist[r], mt).n_tiles;
    bar.nrg = 1;
  } else if (c >= grid - Gsk) {
    const int cs = c - (grid - Gsk);
    bar.csk = cs;
    bar.p_waves = unit_start<NK>(g, bar, nw * Gsk);
    for (int w = 0; w < nw; ++w) {
      bar.rg_beg[w] = unit_start<NK>(g, bar, w * Gsk + cs);
      bar.rg_end[w] = unit_start<NK>(g, bar, w * Gsk + cs + 1);
    }
    bar.rg_beg[nw] = cta_begin<NK>(g, bar, cs, Gsk);
    bar.rg_end[nw] = cta_begin<NK>(g, bar, cs + 1, Gsk);
    bar.nrg = nw + 1;
  }
}

// One contiguous piece of a unit handled by this CTA: tiles [t0, t1).
struct Seg {
  int r, h, mt, t0, t1, kvh, m0, n_hist, uid;
  int hq;          // query head of the tensors (h within the request's heads)
  int64_t ustart;  // work item of the unit's tile 0
  Unit u;
  bool partial;
  int slot;  // partial-output slot (0: first segment of the CTA's stream-K range, 1: last)
};

template <int NK>
__device__ __noinline__ Seg make_seg(const Geo &g, const Bars &bar, int64_t pos, int64_t end,
                                        int slot) {
  Seg s;
  s.r = 0;
  while (s.r + 1 < g.B && pos >= bar.req_pos0[s.r + 1]) ++s.r;
  int64_t rem = pos - bar.req_pos0[s.r];
  const int ph = bar.req_per_head[s.r];
  s.h = (int)(rem / ph);
  rem -= (int64_t)s.h * ph;
  const ReqDesc &R = g.req[s.r];
  s.n_hist = bar.req_hist[s.r];
  s.mt = 0;
  for (;;) {
    const int n = unit_geom<NK>(R, s.n_hist, s.mt).n_tiles;
    if (rem < n) break;
    rem -= n;
    ++s.mt;
  }
  s.t0 = (int)rem;
  s.ustart = pos - s.t0;
  s.u = unit_geom<NK>(R, s.n_hist, s.mt);
  s.t1 = (int)min((int64_t)s.u.n_tiles, (int64_t)s.t0 + (end - pos));
  s.kvh = R.kvh0 + s.h / (g.H / g.Hkv);
  s.hq = R.head0 + s.h;
  s.m0 = s.mt * ROWS;
  s.uid = bar.req_unit0[s.r] + s.h * ((R.lq + ROWS - 1) / ROWS) + s.mt;
  s.partial = !(s.t0 == 0 && s.t1 == s.u.n_tiles);
  s.slot = slot;
  return s;
}

// 32 consecutive values of an output row: fp32 (partials), or bf16 with
// 256-bit stores when rows are 32-byte aligned, else 128-bit stores.
__device__ __forceinline__ void store_f32x32(float *dst, const float (&v)[32]) {
#pragma unroll
  for (int j = 0; j < 32; j += 8)
    asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + j),
                 "f"(v[j]), "f"(v[j + 1]), "f"(v[j + 2]), "f"(v[j + 3]), "f"(v[j + 4]),
                 "f"(v[j + 5]), "f"(v[j + 6]), "f"(v[j + 7])
                 : "memory");
}
__device__ __forceinline__ void store_bf16x32(__nv_bfloat16 *dst, const float (&v)[32], bool v8) {
  uint32_t w[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) w[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
  if (v8) {
#pragma unroll
    for (int j = 0; j < 16; j += 8)
      asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + 2 * j),
                   "r"(w[j]), "r"(w[j + 1]), "r"(w[j + 2]), "r"(w[j + 3]), "r"(w[j + 4]),
                   "r"(w[j + 5]), "r"(w[j + 6]), "r"(w[j + 7])
                   : "memory");
  } else {
#pragma unroll
    for (int j = 0; j < 16; j += 4)
      *reinterpret_cast<uint4 *>(dst + 2 * j) = make_uint4(w[j], w[j + 1], w[j + 2], w[j + 3]);
  }
}

// Merge of a split unit's parts by the CTA whose part completed it: every
// part, this CTA's included, read from global memory in CTA order (the same
// arithmetic whichever CTA merges, so results are reproducible), weighted by
// e^(lse_part - lse) into the final bf16 row and its LSE.  Out of line: cold
// code, with registers of its own.
template <int D, int NK>
__device__ __noinline__ void merge_parts(const Geo &g, const Bars &bar, const Seg &sg, int x,
                                         int row, int G, const float *__restrict__ part_o,
                                         const float *__restrict__ part_lse,
                                         __nv_bfloat16 *orow, float *lrow, bool o_v8) {
  // Parts: the CTAs c0..c1 whose ranges meet the unit's items; the unit is
  // c0's last segment (slot 1) unless it starts c0's range, and the first
  // segment (slot 0) of every later CTA.
  const int64_t uend = sg.ustart + sg.u.n_tiles;
  const int c0 = cta_of<NK>(g, bar, G, sg.ustart), c1 = cta_of<NK>(g, bar, G, uend - 1);
  auto part_row = [&](int c) -> int64_t {  // -1: CTA without items
    const int64_t bc = cta_begin<NK>(g, bar, c, G);
    if (bc == cta_begin<NK>(g, bar, c + 1, G)) return -1;
    const int slot = (c == c0 && bc < sg.ustart) ? 1 : 0;
    return ((int64_t)c * 2 + slot) * ROWS + x * BM + row;
  };
  // every part, this CTA's included, from global memory in CTA order: the
  // same arithmetic whichever CTA merges, so results are reproducible
  // (rows past the request, wr == false, are whole warps: lq is a multiple of 64)
  // weights first, in CTA order
  constexpr int MP = 6;  // parts whose weights are kept in registers
  const bool few = c1 - c0 < MP;
  int64_t pr[MP];
  float lp[MP];
#pragma unroll
  for (int q = 0; q < MP; ++q) {
    pr[q] = few && c0 + q <= c1 ? part_row(c0 + q) : -1;
    lp[q] = pr[q] >= 0 ? __ldcg(part_lse + pr[q]) : -INFINITY;
  }
  float M = -INFINITY;
  if (few) {
#pragma unroll
    for (int q = 0; q < MP; ++q) M = fmaxf(M, lp[q]);
  } else {
    for (int c = c0; c <= c1; ++c) {
      const int64_t r_ = part_row(c);
      if (r_ >= 0) M = fmaxf(M, __ldcg(part_lse + r_));
    }
  }
  float den = 0.f;
  if (few) {
#pragma unroll
    for (int q = 0; q < MP; ++q) den += lp[q] != -INFINITY ? __expf(lp[q] - M) : 0.f;
  } else {
    for (int c = c0; c <= c1; ++c) {
      const int64_t r_ = part_row(c);
      const float l_ = r_ >= 0 ? __ldcg(part_lse + r_) : -INFINITY;
      den += l_ != -INFINITY ? __expf(l_ - M) : 0.f;
    }
  }
  const float rden = den > 0.f ? 1.f / den : 0.f;
  // the parts that hold keys of this row (a part without any wrote no O)
  int nv = 0;
  int64_t ra = 0, rb = 0;
  float wa = 0.f, wb = 0.f;
#pragma unroll
  for (int q = 0; q < MP; ++q) {
    if (lp[q] != -INFINITY) {
      const float wq = __expf(lp[q] - M) * rden;
      if (nv == 0) {
        ra = pr[q];
        wa = wq;
      } else if (nv == 1) {
        rb = pr[q];
        wb = wq;
      }
      ++nv;
    }
  }
  if (__all_sync(0xffffffffu, few && nv <= 2)) {
    // one or two parts (the usual split).  The warp merges its 32 rows one at a
    // time with its lanes across the columns (lane l: columns 4l..4l+3), so a
    // part row is one coalesced 512-byte read; eight rows are in flight at
    // once.  Row r's parts and weights come from lane r.
    const int lane = threadIdx.x & 31;
    for (int r0 = 0; r0 < 32; r0 += 8) {
      float4 va[8], vb[8];
      float wa_r[8], wb_r[8];
      int nv_r[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int r = r0 + u;
        nv_r[u] = __shfl_sync(0xffffffffu, nv, r);
        wa_r[u] = __shfl_sync(0xffffffffu, wa, r);
        wb_r[u] = __shfl_sync(0xffffffffu, wb, r);
        const int64_t ra_r = __shfl_sync(0xffffffffu, ra, r);
        const int64_t rb_r = __shfl_sync(0xffffffffu, rb, r);
        va[u] = nv_r[u] > 0 ? __ldcg(reinterpret_cast<const float4 *>(part_o + ra_r * D) + lane)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        vb[u] = nv_r[u] > 1 ? __ldcg(reinterpret_cast<const float4 *>(part_o + rb_r * D) + lane)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        float4 acc;
        acc.x = fmaf(wa_r[u], va[u].x, 0.f);
        acc.y = fmaf(wa_r[u], va[u].y, 0.f);
        acc.z = fmaf(wa_r[u], va[u].z, 0.f);
        acc.w = fmaf(wa_r[u], va[u].w, 0.f);
        if (nv_r[u] > 1) {
          acc.x = fmaf(wb_r[u], vb[u].x, acc.x);
          acc.y = fmaf(wb_r[u], vb[u].y, acc.y);
          acc.z = fmaf(wb_r[u], vb[u].z, acc.z);
          acc.w = fmaf(wb_r[u], vb[u].w, acc.w);
        }
        __nv_bfloat16 *dst = orow + (int64_t)(r0 + u - lane) * D + 4 * lane;
        *reinterpret_cast<uint2 *>(dst) = make_uint2(pack_bf16x2(acc.x, acc.y),
                                                     pack_bf16x2(acc.z, acc.w));
      }
    }
  } else {
    // more parts: the same arithmetic, one part at a time
    for (int cb = 0; cb < D / 32; ++cb) {
      float acc[32];
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) acc[jj] = 0.f;
      for (int c = c0; c <= c1; ++c) {
        const int64_t r_ = part_row(c);
        if (r_ < 0) continue;
        const float l_ = __ldcg(part_lse + r_);
        if (l_ == -INFINITY) continue;
        const float w_ = __expf(l_ - M) * rden;
        const float4 *src = reinterpret_cast<const float4 *>(part_o + r_ * D) + cb * 8;
        float4 v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = __ldcg(src + e);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          acc[4 * e + 0] = fmaf(w_, v[e].x, acc[4 * e + 0]);
          acc[4 * e + 1] = fmaf(w_, v[e].y, acc[4 * e + 1]);
          acc[4 * e + 2] = fmaf(w_, v[e].z, acc[4 * e + 2]);
          acc[4 * e + 3] = fmaf(w_, v[e].w, acc[4 * e + 3]);
        }
      }
      store_bf16x32(orow + cb * 32, acc, o_v8);
    }
  }
  *lrow = den > 0.f ? M + __logf(den) : -INFINITY;
}

// The first stream-K CTA of a split unit's parts; row 0 of the query tile
// also sets bar.last[x] when the unit has exactly two parts and the other
// one is already counted in (this part then completes it).
template <int NK>
__device__ __noinline__ int direct_check(const Geo &g, Bars &bar, const Seg &sg, int x, int row,
                                         int G, int32_t *unit_cnt) {
  const int64_t uend = sg.ustart + sg.u.n_tiles;
  const int c0 = cta_of<NK>(g, bar, G, sg.ustart), c1 = cta_of<NK>(g, bar, G, uend - 1);
  if (row == 0) {
    int d = 0;
    if (c1 - c0 == 1) {
      int cntv;
      asm volatile("ld.acquire.gpu.global.b32 %0, [%1];"
                   : "=r"(cntv)
                   : "l"(unit_cnt + 2 * sg.uid + x)
                   : "memory");
      d = cntv + (sg.t1 - sg.t0) == sg.u.n_tiles;
    }
    bar.last[x] = d;
  }
  return c0;
}

// Merge of a split unit by its part that ends this CTA's work, when the one
// other part (another CTA's) is already counted in: this part's rows come
// straight from the O accumulator in TMEM (normalised) instead of a round
// trip through the partial-result slots.  The rows go through this query
// tile's Q buffer in shared memory (free: the CTA loads no further Q), 64
// columns at a time, so that each warp then merges its 32 rows with its lanes
// across the columns (coalesced reads of the other part, as in merge_parts).
// The arithmetic is that of merge_parts: weights e^(lse_part - M) / den in
// CTA order, fmaf(w0, v0, 0) then fmaf(w1, v1, .) over the parts holding keys.
template <int D, int NK>
__device__ __noinline__ void merge_direct(const Bars &bar, const Geo &g, const Seg &sg, int x,
                                          int row, int G, uint32_t o_taddr, bool has_o,
                                          float inv, float lse_own, int64_t own_c, int c0,
                                          const float *__restrict__ part_o,
                                          const float *__restrict__ part_lse,
                                          uint8_t *stage, __nv_bfloat16 *orow, float *lrow) {
  const int lane = threadIdx.x & 31;
  const int oc = own_c == c0 ? c0 + 1 : c0;  // the other part's CTA
  const int64_t boc = cta_begin<NK>(g, bar, oc, G);
  const int slot = (oc == c0 && boc < sg.ustart) ? 1 : 0;
  const int64_t orw = ((int64_t)oc * 2 + slot) * ROWS + x * BM + row;  // its row, this thread
  const float lse_oth = __ldcg(part_lse + orw);
  // parts in CTA order
  const bool own_first = own_c == c0;
  const float l0 = own_first ? lse_own : lse_oth, l1 = own_first ? lse_oth : lse_own;
  const float M = fmaxf(fmaxf(-INFINITY, l0), l1);
  float den = 0.f;
  den += l0 != -INFINITY ? __expf(l0 - M) : 0.f;
  den += l1 != -INFINITY ? __expf(l1 - M) : 0.f;
  const float rden = den > 0.f ? 1.f / den : 0.f;
  const float w0 = l0 != -INFINITY ? __expf(l0 - M) * rden : 0.f;
  const float w1 = l1 != -INFINITY ? __expf(l1 - M) * rden : 0.f;
  // per row: which of (part 0, part 1) hold keys; the own one is read from stage
  const int flags = (l0 != -INFINITY ? 1 : 0) | (l1 != -INFINITY ? 2 : 0);
  float4 *st4 = reinterpret_cast<float4 *>(stage);  // [BM rows][16 chunks of 4 fp32]
  const int wrow0 = row - lane;                     // first row of this warp
#pragma unroll 1
  for (int pass = 0; pass < D / 64; ++pass) {
    // this thread's row, 64 columns, normalised, chunk j at (j ^ (row & 15))
    if (has_o) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t ov[32];
        tmem_ld32(o_taddr + pass * 64 + h * 32, ov);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int j = h * 8 + q;
          st4[row * 16 + (j ^ (row & 15))] =
              make_float4(__uint_as_float(ov[4 * q]) * inv, __uint_as_float(ov[4 * q + 1]) * inv,
                          __uint_as_float(ov[4 * q + 2]) * inv, __uint_as_float(ov[4 * q + 3]) * inv);
        }
      }
    }
    __syncwarp();
    // the warp's 32 rows, two per step (16 lanes a row), the other part's loads first
    const int j = lane & 15;
    float4 vo[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int rl = 2 * i + (lane >> 4);  // row within the warp
      const int64_t orw_r = __shfl_sync(0xffffffffu, orw, rl);
      const int fl = __shfl_sync(0xffffffffu, flags, rl);
      const bool oth_ok = own_first ? (fl & 2) : (fl & 1);
      vo[i] = oth_ok ? __ldcg(reinterpret_cast<const float4 *>(part_o + orw_r * D + pass * 64) + j)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int rl = 2 * i + (lane >> 4);
      const int r = wrow0 + rl;  // row within the query tile
      const int fl = __shfl_sync(0xffffffffu, flags, rl);
      const float a0 = __shfl_sync(0xffffffffu, w0, rl), a1 = __shfl_sync(0xffffffffu, w1, rl);
      const float4 vs = (own_first ? (fl & 1) : (fl & 2)) ? st4[r * 16 + (j ^ (r & 15))]
                                                           : make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 v0 = own_first ? vs : vo[i], v1 = own_first ? vo[i] : vs;
      float4 acc;
      // the first part holding keys starts the sum (as merge_parts)
      const bool h0 = fl & 1, h1 = (fl & 2) != 0;
      const float4 f = h0 ? v0 : v1;
      const float wf = h0 ? a0 : a1;
      acc.x = fmaf(wf, f.x, 0.f);
      acc.y = fmaf(wf, f.y, 0.f);
      acc.z = fmaf(wf, f.z, 0.f);
      acc.w = fmaf(wf, f.w, 0.f);
      if (h0 && h1) {
        acc.x = fmaf(a1, v1.x, acc.x);
        acc.y = fmaf(a1, v1.y, acc.y);
        acc.z = fmaf(a1, v1.z, acc.z);
        acc.w = fmaf(a1, v1.w, acc.w);
      }
      __nv_bfloat16 *dst = orow + (int64_t)(rl - lane) * D + pass * 64 + 4 * j;
      *reinterpret_cast<uint2 *>(dst) =
          make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
    }
    __syncwarp();  // the stage rows are rewritten by the next pass
  }
  *lrow = den > 0.f ? M + __logf(den) : -INFINITY;
}

// End of a segment for query tile x (its softmax warpgroup): O normalised and
// written -- final (bf16) when the segment is the whole unit, else a partial
// result (fp32 O, LSE) in this CTA's slot, counted in, and merged by the part
// that completes the unit.  Out of line, so that the tile loop's registers
// are its own.  False when a bounded wait gave up.
template <int D, int NK>
__device__ __noinline__ bool segment_end(const Geo &g, Bars &bar, const Seg &sg, int x, int row,
                                         int G, int csk, int nx, int cnt, float m_run,
                                         float l_run, bool last_seg, uint32_t lane_addr,
                                         uint32_t o_col, uint8_t *smem,
                                         __nv_bfloat16 *__restrict__ o, float *__restrict__ lse,
                                         int o_v8, float *__restrict__ part_o,
                                         float *__restrict__ part_lse,
                                         int32_t *__restrict__ unit_cnt, int &gb) {
  using LY = Layout<D, NK>;
  volatile int *abort = &bar.abort;
  const int lane = threadIdx.x & 31;
  const ReqDesc &R = g.req[sg.r];
  const int qrow = sg.m0 + x * BM + row;  // chunk-local query index
  // warpgroup barrier on an mbarrier: bounded, so a peer that gave up on a
  // timeout cannot leave the others waiting forever
  auto group_sync = [&]() -> bool {
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar.grp[x]);
    return mbar_wait(&bar.grp[x], gb++ & 1, abort, g.err);
  };
  const bool wr = qrow < R.lq;
  const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
  const float lse_v = l_run > 0.f ? (m_run + __log2f(l_run)) * 0.6931471805599453f : -INFINITY;
  const int64_t prow = ((int64_t)csk * 2 + sg.slot) * ROWS + x * BM + row;
  __nv_bfloat16 *orow = o + (int64_t)sg.hq * g.q_hs + (int64_t)(R.q0 + qrow) * D;
  float *lrow = lse + (int64_t)sg.hq * g.lse_hs + R.q0 + qrow;
  if (sg.partial && last_seg) {
    // the unit's other part, when it is a single CTA's and already counted
    // in, is merged right here (merge_direct)
    const int c0 = direct_check<NK>(g, bar, sg, x, row, G, unit_cnt);
    if (nx > 0) {
      if (!mbar_wait(&bar.pv_done[x], (cnt - 1) & 1, abort, g.err)) return false;
      tc_fence_after();
    }
    if (!group_sync()) return false;
    if (*reinterpret_cast<volatile int *>(&bar.last[x])) {  // uniform in the group
      __threadfence();
      if (wr)
        merge_direct<D, NK>(bar, g, sg, x, row, G, lane_addr + o_col, nx > 0, inv, lse_v, csk,
                            c0, part_o, part_lse, smem + LY::OFF_Q + x * LY::Q_BYTES, orow,
                            lrow);
      return true;
    }
  }
  if (nx > 0) {
    if (!mbar_wait(&bar.pv_done[x], (cnt - 1) & 1, abort, g.err)) return false;
    tc_fence_after();
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t ov[32];
      tmem_ld32(lane_addr + o_col + c * 32, ov);
      tmem_ld_wait();
      if (!wr) continue;
      float v[32];
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) v[jj] = __uint_as_float(ov[jj]) * inv;
      if (sg.partial)
        store_f32x32(part_o + prow * D + c * 32, v);
      else
        store_bf16x32(orow + c * 32, v, o_v8 != 0);
    }
  }
  if (wr) {
    if (sg.partial)
      part_lse[prow] = lse_v;  // -inf marks an empty part (no tile of this query tile)
    else
      *lrow = lse_v;
  }
  if (!sg.partial) return true;
  // ---- split unit: count this part's items in; the part that completes
  // the unit's count merges them all.
  __threadfence();  // this thread's part is visible GPU-wide
  if (!group_sync()) return false;
  if (row == 0) {
    const int mine = sg.t1 - sg.t0;
    __threadfence();
    const int before = atomicAdd(unit_cnt + 2 * sg.uid + x, mine);
    __threadfence();
    bar.last[x] = before + mine == sg.u.n_tiles;
  }
  if (!group_sync()) return false;
  if (!*reinterpret_cast<volatile int *>(&bar.last[x])) return true;  // uniform in the group
  __threadfence();
  if (wr)
    merge_parts<D, NK>(g, bar, sg, x, row, G, part_o, part_lse, orow, lrow, o_v8 != 0);
  return true;
}

template <int D, int NK>
__global__ void __launch_bounds__(THREADS, 1)
    attn_tc_kernel(const __grid_constant__ Geo g, const __grid_constant__ TMaps tm,
                   const int32_t *__restrict__ sel_page, const int32_t *__restrict__ n_sel,
                   float scale_log2, __nv_bfloat16 *__restrict__ o, float *__restrict__ lse,
                   int o_v8, float *__restrict__ part_o, float *__restrict__ part_lse,
                   int32_t *__restrict__ unit_cnt, int Gsk, int waves_ok) {
  using LY = Layout<D, NK>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars &bar = *reinterpret_cast<Bars *>(smem + LY::OFF_BAR);
  volatile int *abort = &bar.abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sub = g.Bk / NK;
  const int G = Gsk;  // stream-K CTAs
  // a kernel launched after this one as a programmatic dependent (the next
  // chunk's score GEMM, which reads nothing this kernel writes) may take SMs
  // as they free up here
  asm volatile("griddepcontrol.launch_dependents;");

  if (tid == 0) {
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bar.q_full[x], 1);
      mbar_init(&bar.q_empty[x], 1);
      mbar_init(&bar.s_full[x], 1);
      mbar_init(&bar.p_full[x], 4);  // one arrival per softmax warp
      mbar_init(&bar.pv_done[x], 1);
      mbar_init(&bar.grp[x], 4);
      mbar_init(&bar.tok[x], 1);
    }
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(&bar.full[s], 1);
      mbar_init(&bar.empty[s], 2);  // released by both MMA issuers
    }
    mbar_init(&bar.drain, 2);
    bar.abort = 0;
    build_tables<NK>(g, n_sel, bar);
    schedule<NK>(g, bar, Gsk, waves_ok);
    fence_mbar_init();
  }
  __syncthreads();
  const int csk = bar.csk;  // partial results only arise under stream-K
  const int nrg = bar.nrg;  // ranges: whole units, then (last) the stream-K range
  int rg0 = 0;              // the first range that holds work
  while (rg0 < nrg && bar.rg_beg[rg0] >= bar.rg_end[rg0]) ++rg0;
  if (rg0 == nrg) return;   // a CTA without work (uniform: before any TMEM use)
  if (warp == 1) {
    tmem_alloc(&bar.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // The whole warp runs the loop; lane 0 issues.  Page ids are read 32 tiles
    // ahead (one per lane) so no global load sits on the issue path.
    if (lane == 0) {
      tma_prefetch_desc(&tm.q);
      tma_prefetch_desc(&tm.kc);
      tma_prefetch_desc(&tm.vc);
      tma_prefetch_desc(&tm.kp);
      tma_prefetch_desc(&tm.vp);
    }
    int i = 0;             // K/V loads issued so far (ring position)
    int qn[2] = {0, 0};    // Q_A / Q_B loads issued so far
    bool ok = true;
    int k = 0;
    // the CTA's ranges in order (units of the waves, then the stream-K range);
    // only the stream-K range's first and last segments can be partial
    int rg = rg0;
    for (int64_t pos = bar.rg_beg[rg0]; ok && rg < nrg; ++k) {
      const int64_t re = bar.rg_end[rg];
      const Seg sg = make_seg<NK>(g, bar, pos, re, rg == nrg - 1 && pos == bar.rg_beg[rg] ? 0 : 1);
      pos += sg.t1 - sg.t0;
      if (pos >= re) {
        do ++rg; while (rg < nrg && bar.rg_beg[rg] >= bar.rg_end[rg]);
        if (rg < nrg) pos = bar.rg_beg[rg];
      }
      const ReqDesc &R = g.req[sg.r];
      const int32_t *pages = sel_page + (int64_t)sg.r * g.bt_stride;
      for (int x = 0; x < (sg.u.has_b ? 2 : 1); ++x) {
        int okq = 1;  // Q_x of the previous segment no longer read by an S MMA
        if (lane == 0 && qn[x] > 0) okq = mbar_wait(&bar.q_empty[x], (qn[x] - 1) & 1, abort, g.err);
        if (!__shfl_sync(0xffffffffu, okq, 0)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_expect_tx(&bar.q_full[x], LY::Q_BYTES);
          for (int hf = 0; hf < LY::HALVES; ++hf)
            tma_load_3d(smem + LY::OFF_Q + x * LY::Q_BYTES + hf * (BM * 128), &tm.q,
                        &bar.q_full[x], hf * 64, R.q0 + sg.m0 + x * BM, sg.hq);
        }
        ++qn[x];
      }
      if (!ok) break;
      int pg = 0;
      for (int t = sg.t0; t < sg.t1; ++t) {
        if (((t - sg.t0) & 31) == 0) {  // next 32 tiles' page ids, one per lane
          const int tt = t + lane;
          pg = tt < sg.n_hist ? __ldg(pages + tt / sub) : 0;
        }
        const int p_t = __shfl_sync(0xffffffffu, pg, (t - sg.t0) & 31);
        for (int kv = 0; kv < 2; ++kv, ++i) {
          const int s = i % NSLOT;
          int oks = 1;  // lane 0 waits, the warp follows its verdict
          if (lane == 0 && i >= NSLOT)
            oks = mbar_wait(&bar.empty[s], ((i / NSLOT) - 1) & 1, abort, g.err);
          if (!__shfl_sync(0xffffffffu, oks, 0)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            uint8_t *dst = smem + LY::OFF_KV + s * LY::KV_BYTES;
            mbar_expect_tx(&bar.full[s], LY::KV_BYTES);
            if (t < sg.n_hist) {
              const int p = (p_t < 0 || p_t >= g.num_pages) ? 0 : p_t;  // masked by the softmax
              const int tok = (t % sub) * NK;
              for (int hf = 0; hf < LY::HALVES; ++hf)
                tma_load_4d(dst + hf * (NK * 128), kv ? &tm.vp : &tm.kp, &bar.full[s], hf * 64,
                            sg.kvh, tok, p);
            } else {
              const int j0 = (t - sg.n_hist) * NK;
              for (int hf = 0; hf < LY::HALVES; ++hf) {
                if (g.kv_head_inner)  // k_cur / v_cur laid out [tokens, Hkv, D]
                  tma_load_3d(dst + hf * (NK * 128), kv ? &tm.vc : &tm.kc, &bar.full[s],
                              hf * 64, sg.kvh, R.q0 + j0);
                else
                  tma_load_3d(dst + hf * (NK * 128), kv ? &tm.vc : &tm.kc, &bar.full[s],
                              hf * 64, R.q0 + j0, sg.kvh);
              }
            }
          }
        }
        if (!ok) break;
      }
    }
    // drain: every load issued must land before shared memory is released
    // (only the last Q of each tile and the last NSLOT K/V can be in flight)
    if (lane == 0) {
      for (int x = 0; x < 2; ++x)
        if (qn[x] > 0)
          for (uint32_t n = 0; n < kSpinLimit && !mbar_try_wait(&bar.q_full[x], (qn[x] - 1) & 1);
               ++n) {
          }
      for (int j = max(0, i - NSLOT); j < i; ++j) {
        const uint32_t par = (j / NSLOT) & 1;
        for (uint32_t n = 0; n < kSpinLimit && !mbar_try_wait(&bar.full[j % NSLOT], par); ++n) {
        }
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // Warp 1 issues every MMA of query tile A, warp 2 those of tile B, taking
    // turns (two token mbarriers) so the tensor pipe still sees the single
    // ping-pong order S_A(0), S_B(0), [PV_A(t), S_A(t+1)], [PV_B(t), S_B(t+1)],
    // ...: the softmax of one tile runs while the pipe works for the other.
    // The pipe queues very few MMAs; each issuer does its barrier waits and
    // bookkeeping while the other one's turn keeps the pipe fed.  A K/V slot
    // is released when both issuers have let it go (two arrivals): a commit
    // after the MMAs that read it, or, for a tile its query tile does not
    // attend, a plain arrival once the tile has landed.
    if (lane == 0) {
      const int x = warp - 1;
      constexpr uint32_t idS = idesc_bf16(BM, NK, 0, 0);
      constexpr uint32_t idPV = idesc_bf16(BM, D, 0, 1);
      const uint32_t sQ = smem_addr(smem + LY::OFF_Q);
      const uint32_t sKV = smem_addr(smem + LY::OFF_KV);
      // Descriptors are built once; a k-step only adds its byte offset / 16 to
      // the start-address field (all operands lie below 256 KB of shared memory).
      const uint64_t dQ = sdesc_sw128(sQ, 16, 1024) + (uint64_t)((x * LY::Q_BYTES) >> 4);
      const uint64_t dK0 = sdesc_sw128(sKV, 16, 1024);
      const uint64_t dV0 = sdesc_sw128(sKV, NK * 128, 1024);
      const uint32_t tS = tmem + x * 128, tO = tmem + 256 + x * 128;
      auto slot_wait = [&](int i) {
        return mbar_wait(&bar.full[i % NSLOT], (i / NSLOT) & 1, abort, g.err);
      };
      auto issue_S = [&](int i) {  // i: load index of the K tile
        // K-step k of head_dim: byte offset (k / 4) * half + (k % 4) * 32 in
        // both operands (one PTX block of D / 16 MMAs)
        const uint64_t b0 = dK0 + (uint64_t)(((i % NSLOT) * LY::KV_BYTES) >> 4);
        static_assert(BM == 128, "query tile of 128 rows");
        if constexpr (D == 128 && NK == 128)
          mma_ss_d128_nk128(tS, dQ, b0, idS, 0u);
        else if constexpr (D == 128)
          mma_ss_d128_nk64(tS, dQ, b0, idS, 0u);
        else
          mma_ss_d64(tS, dQ, b0, idS, 0u);
        mma_commit(&bar.s_full[x]);
      };
      auto issue_PV = [&](int i, bool first) {  // i: load index of the V tile
        const uint64_t b0 = dV0 + (uint64_t)(((i % NSLOT) * LY::KV_BYTES) >> 4);
        // A = P in TMEM (16 keys = 8 columns per step); B = V, MN-major
        // (d contiguous): the two 64-wide d blocks are NK*128 bytes apart,
        // 8-key groups 1024 apart; one PTX block of NK / 16 MMAs
        if constexpr (NK == 128)
          mma_ts_nk128(tO, tS, b0, idPV, first ? 0u : 1u);
        else
          mma_ts_nk64(tO, tS, b0, idPV, first ? 0u : 1u);
        mma_commit(&bar.pv_done[x]);
      };
      int turn = 0;  // turns taken: A's turn n follows B's turn n-1, B's turn n follows A's turn n
      auto take_turn = [&]() {
        const bool got = (x == 0 && turn == 0) ||
                         mbar_wait(&bar.tok[x], (x == 0 ? turn - 1 : turn) & 1, abort, g.err);
        ++turn;
        return got;
      };
      auto pass_turn = [&]() { mbar_arrive(&bar.tok[1 - x]); };
      int ib = 0;   // load index of the segment's first K tile
      int cnt = 0;  // tiles the softmax of this query tile has handed over so far
      int qm = 0;   // Q loads of this tile consumed
      int k = 0;
      bool ok = true;
      // the CTA's ranges in order (units of the waves, then the stream-K range);
      // only the stream-K range's first and last segments can be partial
      int rg = rg0;
      for (int64_t pos = bar.rg_beg[rg0]; ok && rg < nrg; ++k) {
        const int64_t re = bar.rg_end[rg];
        const Seg sg = make_seg<NK>(g, bar, pos, re, rg == nrg - 1 && pos == bar.rg_beg[rg] ? 0 : 1);
        pos += sg.t1 - sg.t0;
        if (pos >= re) {
          do ++rg; while (rg < nrg && bar.rg_beg[rg] >= bar.rg_end[rg]);
          if (rg < nrg) pos = bar.rg_beg[rg];
        }
        const int nt = sg.t1 - sg.t0;
        const int n_x = x ? (sg.u.has_b ? sg.u.n_b : 0) : sg.u.n_a;
        const int nx = max(0, min(n_x, sg.t1) - sg.t0);
        const bool has_q = x == 0 || sg.u.has_b;  // Q_x loaded for this segment
        // turn 0 of the segment: S_x(0)
        if (has_q && !mbar_wait(&bar.q_full[x], qm++ & 1, abort, g.err)) break;
        if (nx > 0 && !slot_wait(ib)) break;
        if (!take_turn()) break;
        tc_fence_after();
        if (nx > 0) issue_S(ib);
        if (has_q && nx <= 1) mma_commit(&bar.q_empty[x]);  // Q_x released after its last S
        if (nx > 0) mma_commit(&bar.empty[ib % NSLOT]);
        pass_turn();
        for (int j = 0; j < nt; ++j) {
          const int iK = ib + 2 * j, iV = iK + 1;
          if (j < nx) {
            // waits first, then the turn: PV_x(j) and S_x(j+1) back to back
            if (!slot_wait(iV) || !mbar_wait(&bar.p_full[x], (cnt + j) & 1, abort, g.err) ||
                (j + 1 < nx && !slot_wait(iK + 2)) || !take_turn()) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_PV(iV, j == 0);  // the softmax has turned S_x(j) into P_x(j)
            mma_commit(&bar.empty[iV % NSLOT]);
            if (j + 1 < nx) {
              issue_S(iK + 2);  // after PV_x(j): S_x(j+1) overwrites P_x(j)'s columns
              if (j + 2 == nx) mma_commit(&bar.q_empty[x]);
              mma_commit(&bar.empty[(iK + 2) % NSLOT]);
            }
            pass_turn();
          } else {
            // a tile beyond this query tile's last one: an empty turn, and K, V
            // released once landed (their slots' previous phases are then complete)
            if (!take_turn()) {
              ok = false;
              break;
            }
            pass_turn();
            if (!slot_wait(iK) || !slot_wait(iV)) {
              ok = false;
              break;
            }
            mbar_arrive(&bar.empty[iK % NSLOT]);
            mbar_arrive(&bar.empty[iV % NSLOT]);
          }
        }
        ib += 2 * nt;
        cnt += nx;
      }
      // every MMA issued (by both issuers) has completed before TMEM is freed
      mma_commit(&bar.drain);
      for (uint32_t n = 0; n < kSpinLimit && !mbar_try_wait(&bar.drain, 0); ++n) {
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int x = (warp - 4) >> 2;       // query tile: 0 = A, 1 = B
    const int row = tid - 128 - x * BM;  // row within the tile == TMEM lane
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const uint32_t s_col = x * 128, o_col = 256 + x * 128;
    int cnt = 0;  // tiles handed over so far
    int gb = 0;   // uses of this warpgroup's barrier
    // warpgroup barrier on an mbarrier: bounded, so a peer that gave up on a
    // timeout cannot leave the others waiting forever
    auto group_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.grp[x]);
      return mbar_wait(&bar.grp[x], gb++ & 1, abort, g.err);
    };
    int k = 0;
    bool ok = true;
    // the CTA's ranges in order (units of the waves, then the stream-K range);
    // only the stream-K range's first and last segments can be partial
    int rg = rg0;
    for (int64_t pos = bar.rg_beg[rg0]; ok && rg < nrg; ++k) {
      const int64_t re = bar.rg_end[rg];
      const Seg sg = make_seg<NK>(g, bar, pos, re, rg == nrg - 1 && pos == bar.rg_beg[rg] ? 0 : 1);
      pos += sg.t1 - sg.t0;
      if (pos >= re) {
        do ++rg; while (rg < nrg && bar.rg_beg[rg] >= bar.rg_end[rg]);
        if (rg < nrg) pos = bar.rg_beg[rg];
      }
      const bool last_seg = rg >= nrg;  // no segment of this CTA follows
      const int n_x = x ? (sg.u.has_b ? sg.u.n_b : 0) : sg.u.n_a;
      const int nx = max(0, min(n_x, sg.t1) - sg.t0);
      const int qrow = sg.m0 + x * BM + row;  // chunk-local query index
      const int32_t *pages = sel_page + (int64_t)sg.r * g.bt_stride;
      float m_run = -INFINITY, l_run = 0.f;
      int pg = 0;
      for (int j = 0; j < nx; ++j) {
        const int t = sg.t0 + j;
        if ((j & 31) == 0) {  // next 32 tiles' page ids, one per lane
          const int tt = t + lane;
          pg = tt < sg.n_hist ? __ldg(pages + tt / sub) : 0;
        }
        const int p_cur = __shfl_sync(0xffffffffu, pg, j & 31);
        if (!mbar_wait(&bar.s_full[x], (cnt + j) & 1, abort, g.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[NK];
#pragma unroll
        for (int c = 0; c < NK / 32; ++c)
          tmem_ld32(lane_addr + s_col + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
        tmem_ld_wait();
        if (t < sg.n_hist) {
          if (p_cur < 0 || p_cur >= g.num_pages) {  // invalid page: skip its keys
#pragma unroll
            for (int jj = 0; jj < NK; ++jj) sr[jj] = __float_as_uint(-INFINITY);
            if (row == 0 && (t % sub) == 0) record_error(g.err, XATTN_EPAGE);
          }
        } else {
          const int lim = qrow - (t - sg.n_hist) * NK + 1;  // keys [0, lim) are visible
          if (lim < NK) {
#pragma unroll
            for (int jj = 0; jj < NK; ++jj)
              if (jj >= lim) sr[jj] = __float_as_uint(-INFINITY);
          }
        }
        // softmax_scale > 0, so the row max of the scaled logits is the scaled
        // max; eight independent max chains keep the reduction short
        float m8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          m8[e] = fmax3(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1]), -INFINITY);
#pragma unroll
        for (int jj = 16; jj < NK; jj += 16)
#pragma unroll
          for (int e = 0; e < 8; ++e)
            m8[e] = fmax3(m8[e], __uint_as_float(sr[jj + 2 * e]), __uint_as_float(sr[jj + 2 * e + 1]));
        const float mt =
            fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7])) *
            scale_log2;
        const float mnew = fmaxf(m_run, mt);
        const bool need = mnew > m_run + 8.f;
        const float alpha = need ? ex2(m_run - mnew) : 1.f;
        const float m_use = need ? mnew : m_run;
        const float nb = m_use == -INFINITY ? 0.f : -m_use;
        const uint64_t sc2 = f2(scale_log2, scale_log2), nb2 = f2(nb, nb);
        uint64_t sum2[4] = {0ull, 0ull, 0ull, 0ull};
        // P row -> the S row's TMEM columns (two bf16 per column), the A operand
        // of P V, 64 keys at a time; PV_x of the previous tile finished before
        // this S did
#pragma unroll
        for (int hb = 0; hb < NK / 64; ++hb) {
          uint32_t pk[32];
#pragma unroll
          for (int jj = 0; jj < 64; jj += 2) {
            const uint64_t xx = ffma2(
                f2(__uint_as_float(sr[hb * 64 + jj]), __uint_as_float(sr[hb * 64 + jj + 1])), sc2,
                nb2);
            float x0, x1;
            unf2(xx, x0, x1);
            const uint64_t pp = f2(ex2(x0), ex2(x1));
            sum2[(jj >> 1) & 3] = fadd2(sum2[(jj >> 1) & 3], pp);
            float p0, p1;
            unf2(pp, p0, p1);
            pk[jj >> 1] = pack_bf16x2(p0, p1);
          }
          tmem_st32(lane_addr + s_col + hb * 32, pk);
        }
        float s0, s1, s2, s3;
        unf2(fadd2(sum2[0], sum2[1]), s0, s1);
        unf2(fadd2(sum2[2], sum2[3]), s2, s3);
        l_run = l_run * alpha + ((s0 + s1) + (s2 + s3));
        m_run = m_use;
        if (j > 0 && __any_sync(0xffffffffu, need)) {  // O_x is stable: the previous PV is done
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(lane_addr + o_col + c * 32, ov);
            tmem_ld_wait();
#pragma unroll
            for (int jj = 0; jj < 32; ++jj)
              ov[jj] = __float_as_uint(__uint_as_float(ov[jj]) * alpha);
            tmem_st32(lane_addr + o_col + c * 32, ov);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.p_full[x]);
      }
      if (!ok) break;
      cnt += nx;
      // segment end: O written (or merged); tile x exists (rows below lq)
      // iff x == 0 or has_b
      if (x == 1 && !sg.u.has_b) continue;
      if (!segment_end<D, NK>(g, bar, sg, x, row, G, csk, nx, cnt, m_run, l_run, last_seg,
                              lane_addr, o_col, smem, o, lse, o_v8, part_o, part_lse, unit_cnt,
                              gb))
        break;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

// Whether large launches may run waves of whole units before stream-K.  They
// pay where the keys and values a launch reads (at most every history and
// chunk token of every request and KV head) are more than twice L2: stream-K
// CTAs at unrelated positions then each stream their own pages from DRAM.
// Below that, stream-K alone measured faster (the pages stay in L2 anyway).
// XATTN_ATTN_SCHEDULE = "waves" or "streamk" overrides the choice (tests and
// tuning).
inline int waves_allowed(const Geo &g) {
  const char *env = getenv("XATTN_ATTN_SCHEDULE");
  if (env && strcmp(env, "waves") == 0) return 1;
  if (env && strcmp(env, "streamk") == 0) return 0;
  int dev = 0, l2 = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
    return 0;
  int64_t kv_bytes = 0;
  for (int r = 0; r < g.B; ++r)
    kv_bytes += (int64_t)g.Hkv * (g.req[r].kh + g.req[r].lq) * g.D * 2 * 2;
  return kv_bytes > 2 * (int64_t)l2 ? 1 : 0;
}

template <int D, int NK>
cudaError_t launch_tc(const Geo &g, int grid, const __nv_bfloat16 *q, const __nv_bfloat16 *kcur,
                      const __nv_bfloat16 *vcur, const __nv_bfloat16 *kpool,
                      const __nv_bfloat16 *vpool, const int32_t *sel_page, const int32_t *n_sel,
                      float scale, __nv_bfloat16 *o, float *lse, float *part_o, float *part_lse,
                      int32_t *unit_cnt, int nunits, cudaStream_t st) {
  TMaps tm;
  const int64_t tot_q = (int64_t)g.req[g.B - 1].q0 + g.req[g.B - 1].lq;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)tot_q, (cuuint64_t)g.H_all};
    const cuuint64_t str[2] = {(cuuint64_t)D * 2, (cuuint64_t)g.q_hs * 2};
    const cuuint32_t box[3] = {64, BM, 1};
    if (!encode_bf16(&tm.q, q, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  if (g.kv_head_inner) {  // k_cur / v_cur as (d, head, token): [tokens, Hkv, D]
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)g.Hkv_all, (cuuint64_t)tot_q};
    const cuuint64_t str[2] = {(cuuint64_t)g.kv_hs * 2, (cuuint64_t)g.kv_ts * 2};
    const cuuint32_t box[3] = {64, 1, NK};
    if (!encode_bf16(&tm.kc, kcur, 3, dims, str, box)) return cudaErrorInvalidValue;
    if (!encode_bf16(&tm.vc, vcur, 3, dims, str, box)) return cudaErrorInvalidValue;
  } else {  // (d, token, head): [Hkv, tokens, D]
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)tot_q, (cuuint64_t)g.Hkv_all};
    const cuuint64_t str[2] = {(cuuint64_t)g.kv_ts * 2, (cuuint64_t)g.kv_hs * 2};
    const cuuint32_t box[3] = {64, NK, 1};
    if (!encode_bf16(&tm.kc, kcur, 3, dims, str, box)) return cudaErrorInvalidValue;
    if (!encode_bf16(&tm.vc, vcur, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  if (g.num_pages > 0 && kpool && vpool) {
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)g.Hkv_all, (cuuint64_t)g.Bk,
                                (cuuint64_t)g.num_pages};
    const cuuint64_t str[3] = {(cuuint64_t)D * 2, (cuuint64_t)g.Hkv_all * D * 2,
                               (cuuint64_t)g.Bk * g.Hkv_all * D * 2};
    const cuuint32_t box[4] = {64, 1, NK, 1};
    if (!encode_bf16(&tm.kp, kpool, 4, dims, str, box)) return cudaErrorInvalidValue;
    if (!encode_bf16(&tm.vp, vpool, 4, dims, str, box)) return cudaErrorInvalidValue;
  } else {
    tm.kp = tm.kc;
    tm.vp = tm.vc;
  }
  using LY = Layout<D, NK>;
  static_assert(sizeof(Bars) <= 2048, "barrier block");
  static_assert(LY::SMEM_ALLOC <= 232448, "dynamic shared memory of one CTA");
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D, NK>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, LY::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  // per-unit part counters start at zero
  e = cudaMemsetAsync(unit_cnt, 0, (size_t)nunits * 2 * sizeof(int32_t), st);
  if (e != cudaSuccess) return e;
  const int o_v8 = (reinterpret_cast<uintptr_t>(o) % 32 == 0) && ((g.q_hs * 2) % 32 == 0);
  // one CTA per unit (the whole-units schedule), at least Gsk (stream-K): the
  // kernel decides on the device which it runs
  const int Gsk = grid;
  const int ctas = nunits > Gsk ? nunits : Gsk;
  attn_tc_kernel<D, NK><<<ctas, THREADS, LY::SMEM_ALLOC, st>>>(
      g, tm, sel_page, n_sel, scale * 1.4426950408889634f, o, lse, o_v8, part_o, part_lse,
      unit_cnt, Gsk, waves_allowed(g));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const Geo &g, int nctas, const __nv_bfloat16 *q,
                             const __nv_bfloat16 *kcur, const __nv_bfloat16 *vcur,
                             const __nv_bfloat16 *kpool, const __nv_bfloat16 *vpool,
                             const int32_t *sel_page, const int32_t *n_sel, float scale,
                             __nv_bfloat16 *o, float *lse, float *part_o, float *part_lse,
                             int32_t *unit_cnt, cudaStream_t st) {
  if (nctas == 0) return cudaSuccess;  // no query rows
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidValue;
  const int grid = sms < kAttnMaxCtas ? sms : kAttnMaxCtas;
  const bool wide = g.Bk % 128 == 0;  // KV tile: 128 keys, else 64
  if (g.D == 128)
    return wide ? launch_tc<128, 128>(g, grid, q, kcur, vcur, kpool, vpool, sel_page, n_sel,
                                      scale, o, lse, part_o, part_lse, unit_cnt, nctas, st)
                : launch_tc<128, 64>(g, grid, q, kcur, vcur, kpool, vpool, sel_page, n_sel,
                                     scale, o, lse, part_o, part_lse, unit_cnt, nctas, st);
  if (g.D == 64)
    return wide ? launch_tc<64, 128>(g, grid, q, kcur, vcur, kpool, vpool, sel_page, n_sel,
                                     scale, o, lse, part_o, part_lse, unit_cnt, nctas, st)
                : launch_tc<64, 64>(g, grid, q, kcur, vcur, kpool, vpool, sel_page, n_sel,
                                    scale, o, lse, part_o, part_lse, unit_cnt, nctas, st);
  return cudaErrorInvalidValue;
}

}  // namespace xattn
