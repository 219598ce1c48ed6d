// Estimation score GEMM of XAttention BSA ("XAttention BSA Policy 设计文档",
// select_blocks Step 1 flat_group_gemm_fuse_reshape; "XAttention Offload
// Stream Synchronization Fix", 技术细节 Stage 1 softmax_compute_partial_stats).
//
// For one (request, head) the reshaped scores are a plain GEMM with K = S*D:
//   s[a, b] = scale * sum_{i<S} q[S a + S-1-i] . k[S b + i]
// where reshaped column b runs over [history ; current chunk].
//
//   score_gemm_kernel persistent CTAs over 256 x 256 output tiles (two 128-row
//                     MMA tiles; both accumulators fill the 512 TMEM columns).
//                     The stride reversal costs nothing: TMA views (d, phase,
//                     group, ...) of q and of the keys pick phase S-1-i of q for
//                     the k-step that uses phase i of k.  Two key sources:
//                     * pages (xattn_estimate): a tile's 256 reshaped columns
//                       are 256/Br boxes of Br rows, each one history page -- a
//                       5-D view (d, KV head, phase, group, page) of the pool,
//                       addressed through the block table -- or Br columns of
//                       the current chunk; the boxes land back to back, which is
//                       the layout of one 256-row box;
//                     * a logical-order key sequence (xattn_estimate_seq): the
//                       request's history and current keys in token order, so
//                       the tile's 256 columns at phase i are one strided box of
//                       256 rows -- one TMA instruction per k-step instead of
//                       256/Br (the box count per SM is what bounds the paged
//                       form).
//                     A launch's last wave, when it would fill at most half of
//                     the SMs, runs its tiles as 256 x 128 halves instead.
//     warp 0       TMA producer over an NST-stage ring (runs ahead into the
//                  next tile while the epilogue drains TMEM); paged form: lane
//                  q issues key box q of each k-step
//     warp 1       MMA issuer: per k-step 4 x tcgen05.mma (K = 16) per M tile
//     warps 4..11  epilogue, one thread per row, per 128-column statistics
//                  tile: the tile max m_t over the visible cells, and for each
//                  Br-column KV block of the tile the partial sum
//                  sum exp(s - m_t) over its visible cells; their total is the
//                  tile's sum l_t.  The block partials ([H][Qb][Kb][Br]: a
//                  query block's rows contiguous per KV block, so a warp's
//                  store of one block is two or four full segments) and
//                  (m_t, l_t) go to the workspace; the fp32 score matrix itself
//                  is never written.  block_sum_kernel (estimate.cu) merges
//                  the tile statistics per row and rescales the partials:
//                  sum over the block of exp(s - m)/l = sum_t-part * e^(m_t - m)/l,
//                  exactly the two-pass normalise-then-sum of the pages, with
//                  pass 2 folded into pass 1 per tile.  Tiles right of the
//                  causal diagonal are never scheduled.
#include <string.h>

#include "tc_common.cuh"

namespace xattn {
namespace {
using namespace tc;

constexpr int TM = 128;           // rows per MMA tile
constexpr int ROWS = kGemmRows;   // 256 rows per output tile
constexpr int COLS = kGemmCols;   // 256 columns per output tile
constexpr int KSTEP = 64;         // bf16 elements of K per stage (one 128-byte swizzle row)
constexpr int NST = 3;
constexpr int THREADS = 384;
constexpr int A_BYTES = ROWS * KSTEP * 2;  // 32 KB
constexpr int B_BYTES = COLS * KSTEP * 2;  // 32 KB
constexpr int STAGE = A_BYTES + B_BYTES;
constexpr int OFF_BAR = NST * STAGE;
constexpr int SMEM_ALLOC = OFF_BAR + 1024 + 1024;

struct Bars {
  uint64_t full[NST];
  uint64_t empty[NST];
  uint64_t acc_full;
  uint64_t acc_empty;
  uint32_t tmem_base;
  int abort;
};

struct Maps {
  CUtensorMap q;         // queries (d, phase, group, head)
  CUtensorMap kp, kc;    // paged form: pool keys (5-D), current-chunk keys (4-D)
  CUtensorMap ks, ksh;   // sequence form: logical-order keys, 256- and 128-row boxes
  CUtensorMap kh, khh;   // sampled history: the first ns groups of every block (5-D),
                         // 256 and 128 rows a box
  int kc_head_inner;     // the current-chunk key view is (d, head, phase, group)
  int ks_head_inner;     // the key-sequence view is (d, head, phase, group)
};

struct Tile {
  int r, h, m0, n0;  // n0: first reshaped column of the work item
  int w;             // its columns: COLS, or 128 for half of a tile of the last wave
};

// Tile t of the score GEMM: requests in order, then head, then row tile, then
// column tile; only tiles holding visible cells exist.
__device__ __forceinline__ Tile decode_tile(const Geo &g, int t) {
  const int r = find_req(g, t, [](const ReqDesc &d) { return d.gemm0; });
  const ReqDesc &R = g.req[r];
  const int S = g.S;
  const int rq = R.lq / S, ch = R.hc, ncol = R.hc + rq;  // ch: columns before the chunk's
  int per_head = 0;
  for (int m0 = 0; m0 < rq; m0 += ROWS) {
    const int vis = min(ch + min(m0 + ROWS, rq), ncol);
    per_head += (vis + COLS - 1) / COLS;
  }
  int local = t - R.gemm0;
  Tile tl;
  tl.r = r;
  tl.h = local / per_head;
  local -= tl.h * per_head;
  for (int m0 = 0; m0 < rq; m0 += ROWS) {
    const int vis = min(ch + min(m0 + ROWS, rq), ncol);
    const int n = (vis + COLS - 1) / COLS;
    if (local < n) {
      tl.m0 = m0;
      tl.n0 = local * COLS;
      return tl;
    }
    local -= n;
  }
  tl.m0 = tl.n0 = 0;  // unreachable for valid t
  return tl;
}

// Work item w of the launch: tiles 0..nfull-1 whole, then the remaining tiles
// as two 128-column halves each (the launch's last wave, so that it spreads
// over as many SMs as it can fill).
__device__ __forceinline__ Tile decode_work(const Geo &g, int w, int nfull) {
  if (w < nfull) {
    Tile tl = decode_tile(g, w);
    tl.w = COLS;
    return tl;
  }
  const int hh = w - nfull;
  Tile tl = decode_tile(g, nfull + hh / 2);
  tl.n0 += (hh & 1) * (COLS / 2);
  tl.w = COLS / 2;
  return tl;
}

// SEQ: keys from the logical-order key sequence (one box per k-step), else
// from the pool pages and the current chunk (one box per page per k-step).
// NS > 0 (with SEQ): requests marked samp keep the first NS reshaped columns
// of each history block ("XAttention BSA Policy 设计文档", 性能分析,
// 优化方向 2): their GEMM columns are the sampled history columns, padded to a
// statistics tile, then the chunk's; each sampled cell carries the weight
// BR / NS in the tile sums and block partials.
template <int BR, bool SEQ, int NS>
__global__ void __launch_bounds__(THREADS, 1)
    score_gemm_kernel(const __grid_constant__ Geo g, const __grid_constant__ Maps mp, int nwork,
                      int nfull, float scale, float *__restrict__ bpart,
                      float2 *__restrict__ tstat) {
  constexpr int NB = kTileCols / BR;  // KV blocks per statistics tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars &bar = *reinterpret_cast<Bars *>(smem + OFF_BAR);
  volatile int *abort = &bar.abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = g.S, D = g.D;
  const int ksteps = S * D / KSTEP;
  const int tile0 = (int)blockIdx.x, tstep = (int)gridDim.x;

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&bar.full[s], 1);
      mbar_init(&bar.empty[s], 1);
    }
    mbar_init(&bar.acc_full, 1);
    mbar_init(&bar.acc_empty, 8);  // one arrival per epilogue warp
    bar.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bar.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    constexpr int SUB_BYTES = BR * KSTEP * 2;   // Br rows of 128 B (a multiple of 1024)
    static_assert(COLS / BR <= 32 && SUB_BYTES % 1024 == 0, "key boxes");
    if (lane == 0) {
      tma_prefetch_desc(&mp.q);
      if (SEQ) {
        tma_prefetch_desc(&mp.ks);
        tma_prefetch_desc(&mp.ksh);
      } else {
        tma_prefetch_desc(&mp.kp);
        tma_prefetch_desc(&mp.kc);
      }
    }
    int it = 0;  // k-steps issued so far (ring position)
    bool ok = true;
    for (int t = tile0; ok && t < nwork; t += tstep) {
      const Tile tl = decode_work(g, t, nfull);
      const ReqDesc &R = g.req[tl.r];
      const int kvh = tl.h / (g.H / g.Hkv);
      const int nsub = tl.w / BR;  // paged form: key boxes per k-step
      const int ch = R.kh / S, ncol = (R.kh + R.lq) / S;
      // paged form, this lane's key box: reshaped columns [b, b + Br) are one
      // history page (its block-table entry) or Br groups of the current chunk
      bool hist = false;
      int src = R.q0 / S;  // columns past the last one: any in-bounds box (masked)
      if (!SEQ && lane < nsub) {
        const int b = tl.n0 + lane * BR;
        if (b < ch) {
          hist = true;
          src = page_of(g, tl.r, b / BR);  // -1 (and a recorded error) if out of the pool
          if (src < 0) src = 0;
        } else if (b < ncol) {
          src = R.q0 / S + (b - ch);
        }
      }
      for (int ks = 0; ks < ksteps; ++ks, ++it) {
        const int s = it % NST;
        int oks = 1;  // lane 0 waits, the warp follows its verdict
        if (lane == 0 && it >= NST)
          oks = mbar_wait(&bar.empty[s], ((it / NST) - 1) & 1, abort, g.err);
        if (!__shfl_sync(0xffffffffu, oks, 0)) {
          ok = false;
          break;
        }
        const int kk = ks * KSTEP;
        const int i = kk / D, dc = kk % D;
        uint8_t *sA = smem + s * STAGE;
        if (lane == 0) {
          mbar_expect_tx(&bar.full[s], A_BYTES + tl.w * KSTEP * 2);
          // q rows S*a + S-1-i of this tile
          tma_load_4d(sA, &mp.q, &bar.full[s], dc, S - 1 - i, R.q0 / S + tl.m0, tl.h);
          bool loaded = false;
          if constexpr (NS > 0) {
            if (R.samp) {
              // sampled history rows (blocks of NS groups), then chunk rows
              uint8_t *dst = sA + A_BYTES;
              int hrows = 0;
              if (tl.n0 < R.hc) {
                hrows = min(tl.w, R.hc - tl.n0);  // a whole box or half of one
                const CUtensorMap *hm = hrows == COLS ? &mp.kh : &mp.khh;
                const int blk = R.ks0 / BR + tl.n0 / NS;
                if (mp.ks_head_inner)
                  tma_load_5d(dst, hm, &bar.full[s], dc, kvh, i, 0, blk);
                else
                  tma_load_5d(dst, hm, &bar.full[s], dc, i, 0, blk, kvh);
              }
              if (hrows < tl.w) {
                const CUtensorMap *cm = tl.w - hrows == COLS ? &mp.ks : &mp.ksh;
                const int grp = R.ks0 + R.kh / S + max(tl.n0 - R.hc, 0);
                if (mp.ks_head_inner)
                  tma_load_4d(dst + hrows * 128, cm, &bar.full[s], dc, kvh, i, grp);
                else
                  tma_load_4d(dst + hrows * 128, cm, &bar.full[s], dc, i, grp, kvh);
              }
              loaded = true;
            }
          }
          if (SEQ && !loaded) {  // key rows S*b + i, b over the tile's columns: one box
            const CUtensorMap *km = tl.w == COLS ? &mp.ks : &mp.ksh;
            const int grp = R.ks0 + tl.n0;
            if (mp.ks_head_inner)
              tma_load_4d(sA + A_BYTES, km, &bar.full[s], dc, kvh, i, grp);
            else
              tma_load_4d(sA + A_BYTES, km, &bar.full[s], dc, i, grp, kvh);
          }
        }
        if (!SEQ) {
          __syncwarp();
          if (lane < nsub) {  // key rows S*b + i
            uint8_t *dst = sA + A_BYTES + lane * SUB_BYTES;
            if (hist)
              tma_load_5d(dst, &mp.kp, &bar.full[s], dc, kvh, i, 0, src);
            else if (mp.kc_head_inner)
              tma_load_4d(dst, &mp.kc, &bar.full[s], dc, kvh, i, src);
            else
              tma_load_4d(dst, &mp.kc, &bar.full[s], dc, i, src, kvh);
          }
        }
      }
    }
    if (lane == 0) {
      for (int k = max(0, it - NST); k < it; ++k) {
        const uint32_t par = (k / NST) & 1;
        for (uint32_t n = 0; n < kSpinLimit && !mbar_try_wait(&bar.full[k % NST], par); ++n) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_w = idesc_bf16(TM, COLS, 0, 0), idesc_h = idesc_bf16(TM, COLS / 2, 0, 0);
      // descriptors are built once and advanced by byte offset / 16
      const uint64_t d0 = sdesc_sw128(smem_addr(smem), 16, 1024);
      int it = 0, n = 0;
      bool ok = true;
      for (int t = tile0; ok && t < nwork; t += tstep, ++n) {
        const Tile tl = decode_work(g, t, nfull);
        const uint32_t idesc = tl.w == COLS ? idesc_w : idesc_h;
        const int rq = g.req[tl.r].lq / S;
        const bool two_m = tl.m0 + TM < rq;
        // the epilogue has drained the previous tile's accumulators
        if (n > 0 && !mbar_wait(&bar.acc_empty, (n - 1) & 1, abort, g.err)) break;
        tc_fence_after();
        for (int ks = 0; ks < ksteps; ++ks, ++it) {
          const int s = it % NST;
          if (!mbar_wait(&bar.full[s], (it / NST) & 1, abort, g.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t a0 = d0 + (uint64_t)((s * STAGE) >> 4);
          const uint64_t b0 = a0 + (uint64_t)(A_BYTES >> 4);
          for (int x = 0; x < (two_m ? 2 : 1); ++x) {
#pragma unroll
            for (int kq = 0; kq < KSTEP / 16; ++kq)
              mma_f16_ss(tmem + x * COLS, a0 + (uint64_t)((x * (TM * 128) + kq * 32) >> 4),
                         b0 + (uint64_t)((kq * 32) >> 4), idesc, (ks > 0 || kq > 0) ? 1u : 0u);
          }
          mma_commit(&bar.empty[s]);
        }
        mma_commit(&bar.acc_full);
      }
      // every MMA issued has completed before TMEM is freed: the epilogue waited
      // for each tile's acc_full, and no MMA follows the last commit
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int x = (warp - 4) >> 2;
    const int row = tid - 128 - x * TM;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + x * COLS;
    int n = 0;
    for (int t = tile0; t < nwork; t += tstep, ++n) {
      const Tile tl = decode_work(g, t, nfull);
      const ReqDesc &R = g.req[tl.r];
      const int rq = R.lq / S, ch = NS > 0 ? R.hc : R.kh / S;
      const int ncol = NS > 0 ? R.hc + rq : (R.kh + R.lq) / S;
      const int nj = tl.w / kTileCols;  // statistics tiles of the work item
      const int ntile = (ncol + kTileCols - 1) / kTileCols;
      const bool two_m = tl.m0 + TM < rq;
      const int a = tl.m0 + x * TM + row;
      if (!mbar_wait(&bar.acc_full, n & 1, abort, g.err)) break;
      tc_fence_after();
      if (x == 0 || two_m) {
        const bool row_ok = a < rq;
        const int Qb = rq / BR, Kbh = R.kh / g.Bk;
        const int Kb = NS > 0 ? Kbh + Qb : ncol / BR;
        // block partials are stored [H][Qb][Kb][Br]
        float *pbase = bpart + R.bpart_off +
                       ((int64_t)(tl.h * Qb + (row_ok ? a : 0) / BR) * Kb) * BR +
                       (row_ok ? a : 0) % BR;
#pragma unroll 1
        for (int j = 0; j < nj; ++j) {
          const int c0 = tl.n0 + j * kTileCols;  // first column of this statistics tile
          uint32_t v[kTileCols];
#pragma unroll
          for (int c = 0; c < kTileCols / 32; ++c)
            tmem_ld32(lane_addr + j * kTileCols + c * 32,
                      *reinterpret_cast<uint32_t(*)[32]>(&v[c * 32]));
          tmem_ld_wait();
          if (j == nj - 1) {
            // all of this tile's accumulators are in registers: release TMEM
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.acc_empty);
          }
          if constexpr (NS > 0) {
            if (R.samp && c0 < ch) {
              // sampled history columns [c0, c0 + nv), alike for every row;
              // a tile of padding only gets empty statistics
              if (!row_ok) continue;
              const int64_t ti = R.tstat_off + ((int64_t)tl.h * rq + a) * ntile + c0 / kTileCols;
              const int nv = min(kTileCols, Kbh * NS - c0);
              if (nv <= 0) {
                tstat[ti] = make_float2(-INFINITY, 0.f);
                continue;
              }
              constexpr int NBH = kTileCols / NS;
              float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
              for (int c = 0; c < kTileCols; ++c) {
                const float f = __uint_as_float(v[c]) * scale;
                v[c] = __float_as_uint(c < nv ? f : -INFINITY);
                mx[c & 3] = fmaxf(mx[c & 3], __uint_as_float(v[c]));
              }
              const float m = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
              const float ml2 = m * 1.4426950408889634f;
              float pb[NBH];
#pragma unroll
              for (int q = 0; q < NBH; ++q) pb[q] = 0.f;
#pragma unroll
              for (int c = 0; c < kTileCols; ++c)
                pb[c / NS] += ex2(fmaf(__uint_as_float(v[c]), 1.4426950408889634f, -ml2));
              constexpr float wgt = (float)(BR / NS);  // cells each sampled cell stands for
              float l = 0.f;
#pragma unroll
              for (int q = 0; q < NBH; ++q) {
                pb[q] *= wgt;
                l += pb[q];
                const int kb = c0 / NS + q;
                if (kb < Kbh) pbase[(int64_t)kb * BR] = pb[q];
              }
              tstat[ti] = make_float2(m, l);
              continue;
            }
          }
          if (!row_ok || c0 >= ncol || c0 > ch + a) continue;
          // visible columns of the row in this tile: [c0, c0 + nv)
          const int nv = min(min(kTileCols, ncol - c0), ch + a + 1 - c0);
          float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int c = 0; c < kTileCols; ++c) {
            const float f = __uint_as_float(v[c]) * scale;
            v[c] = __float_as_uint(c < nv ? f : -INFINITY);
            mx[c & 3] = fmaxf(mx[c & 3], __uint_as_float(v[c]));
          }
          const float m = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
          const float ml2 = m * 1.4426950408889634f;
          float pb[NB];
#pragma unroll
          for (int q = 0; q < NB; ++q) pb[q] = 0.f;
#pragma unroll
          for (int c = 0; c < kTileCols; ++c)
            pb[c / BR] += ex2(fmaf(__uint_as_float(v[c]), 1.4426950408889634f, -ml2));
          float l = 0.f;
#pragma unroll
          for (int q = 0; q < NB; ++q) {
            l += pb[q];
            // (with a sampled history the chunk's blocks follow its padded columns)
            const int kb = (NS > 0 && c0 >= ch ? Kbh + (c0 - ch) / BR : c0 / BR) + q;
            if (kb < Kb) pbase[(int64_t)kb * BR] = pb[q];
          }
          tstat[R.tstat_off + ((int64_t)tl.h * rq + a) * ntile + c0 / kTileCols] =
              make_float2(m, l);
        }
      } else {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.acc_empty);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
  // this CTA's work is done: the block-sum launch after this one (a
  // programmatic dependent, which waits for this grid to complete before it
  // reads) may start on the SMs that free up
  asm volatile("griddepcontrol.launch_dependents;");
  // Launched as a programmatic dependent of the kernel before it on the
  // stream: this launch may have started while that kernel (a previous
  // chunk's attention, which lets its dependents start early) was still
  // running -- none of this kernel's inputs is its output.  It completes only
  // once that kernel has, so whatever follows on the stream sees both done.
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// A view (d, phase, group, head) of a [heads, tokens, D]-strided bf16 tensor,
// or (d, head, phase, group) when heads are closer than tokens (a
// [tokens, heads, D] layout), so that the strides of the view grow; returns
// whether the head comes second.  box_rows groups of one phase per box.
bool encode_phase_view(CUtensorMap *m, const void *base, int D, int S, int64_t groups,
                       int heads, int64_t hs, int64_t ts, int box_rows, bool *head_inner) {
  *head_inner = hs < ts;
  if (*head_inner) {
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)S,
                                (cuuint64_t)groups};
    const cuuint64_t str[3] = {(cuuint64_t)hs * 2, (cuuint64_t)ts * 2, (cuuint64_t)S * ts * 2};
    const cuuint32_t box[4] = {KSTEP, 1, 1, (cuuint32_t)box_rows};
    return encode_bf16(m, base, 4, dims, str, box);
  }
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)groups,
                              (cuuint64_t)heads};
  const cuuint64_t str[3] = {(cuuint64_t)ts * 2, (cuuint64_t)S * ts * 2, (cuuint64_t)hs * 2};
  const cuuint32_t box[4] = {KSTEP, 1, (cuuint32_t)box_rows, 1};
  return encode_bf16(m, base, 4, dims, str, box);
}

}  // namespace

cudaError_t launch_score_gemm(const Geo &g, int ntiles, const __nv_bfloat16 *q,
                              const __nv_bfloat16 *kcur, const __nv_bfloat16 *kpool,
                              const KeySeq *kseq, float scale, float *bpart, float2 *tstat,
                              bool early, cudaStream_t st) {
  if (ntiles == 0) return cudaSuccess;
  const int S = g.S, D = g.D, BRc = g.Bk / S;
  const int64_t tot_q = (int64_t)g.req[g.B - 1].q0 + g.req[g.B - 1].lq;
  Maps mp;
  memset(&mp, 0, sizeof(mp));
  bool hi = false;
  // q as (d, phase i, group, head)
  if (!encode_phase_view(&mp.q, q, D, S, tot_q / S, g.H, g.q_hs, D, ROWS, &hi))
    return cudaErrorInvalidValue;
  if (kseq) {
    // the keys of every request in logical order: as many groups as the
    // furthest request reaches
    int64_t groups = 1;
    for (int r = 0; r < g.B; ++r) {
      const int64_t e = (int64_t)g.req[r].ks0 + (g.req[r].kh + g.req[r].lq) / S;
      if (e > groups) groups = e;
    }
    if (!encode_phase_view(&mp.ks, kseq->base, D, S, groups, g.Hkv, kseq->hs, kseq->ts, COLS,
                           &hi))
      return cudaErrorInvalidValue;
    mp.ks_head_inner = hi;
    if (!encode_phase_view(&mp.ksh, kseq->base, D, S, groups, g.Hkv, kseq->hs, kseq->ts,
                           COLS / 2, &hi))
      return cudaErrorInvalidValue;
    if (g.ns > 0) {
      // sampled history: (d, phase, group of the block, block, head), or the
      // head second for token-major keys; a box takes the first ns groups of
      // rows / ns consecutive blocks, landing as [block][group] rows
      const int64_t nblk = (groups + BRc - 1) / BRc, hs = kseq->hs, ts = kseq->ts;
      for (int half = 0; half < 2; ++half) {
        const cuuint32_t nb = (cuuint32_t)((half ? COLS / 2 : COLS) / g.ns);
        CUtensorMap *m = half ? &mp.khh : &mp.kh;
        bool ok;
        if (hi) {
          const cuuint64_t dims[5] = {(cuuint64_t)D, (cuuint64_t)g.Hkv, (cuuint64_t)S,
                                      (cuuint64_t)BRc, (cuuint64_t)nblk};
          const cuuint64_t str[4] = {(cuuint64_t)hs * 2, (cuuint64_t)ts * 2,
                                     (cuuint64_t)S * ts * 2, (cuuint64_t)g.Bk * ts * 2};
          const cuuint32_t box[5] = {KSTEP, 1, 1, (cuuint32_t)g.ns, nb};
          ok = encode_bf16(m, kseq->base, 5, dims, str, box);
        } else {
          const cuuint64_t dims[5] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)BRc,
                                      (cuuint64_t)nblk, (cuuint64_t)g.Hkv};
          const cuuint64_t str[4] = {(cuuint64_t)ts * 2, (cuuint64_t)S * ts * 2,
                                     (cuuint64_t)g.Bk * ts * 2, (cuuint64_t)hs * 2};
          const cuuint32_t box[5] = {KSTEP, 1, (cuuint32_t)g.ns, nb, 1};
          ok = encode_bf16(m, kseq->base, 5, dims, str, box);
        }
        if (!ok) return cudaErrorInvalidValue;
      }
    }
  } else {
    // current-chunk keys, Br groups per box
    if (!encode_phase_view(&mp.kc, kcur, D, S, tot_q / S, g.Hkv, g.kv_hs, g.kv_ts, BRc, &hi))
      return cudaErrorInvalidValue;
    mp.kc_head_inner = hi;
    if (g.num_pages > 0 && kpool) {  // pool keys as (d, kv head, phase i, group, page)
      const cuuint64_t dims[5] = {(cuuint64_t)D, (cuuint64_t)g.Hkv, (cuuint64_t)S,
                                  (cuuint64_t)BRc, (cuuint64_t)g.num_pages};
      const cuuint64_t str[4] = {(cuuint64_t)D * 2, (cuuint64_t)g.Hkv * D * 2,
                                 (cuuint64_t)S * g.Hkv * D * 2, (cuuint64_t)g.Bk * g.Hkv * D * 2};
      const cuuint32_t box[5] = {KSTEP, 1, 1, (cuuint32_t)BRc, 1};
      if (!encode_bf16(&mp.kp, kpool, 5, dims, str, box)) return cudaErrorInvalidValue;
    } else {
      mp.kp = mp.kc;  // no history anywhere: never used
    }
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidValue;
  auto run = [&](auto kernel) {
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    // A last wave that fills at most half of the SMs runs as half-width tiles
    // (twice as many, each half the time).
    const int rem = ntiles % sms;
    const int nfull = (rem > 0 && 2 * rem <= sms) ? ntiles - rem : ntiles;
    const int nwork = nfull + 2 * (ntiles - nfull);
    const int n = nwork < sms ? nwork : sms;
    // programmatic dependent launch: free SMs of a kernel that is finishing
    // (the previous chunk's attention) start this one (see the kernel's end)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM_ALLOC;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = early ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, g, mp, nwork, nfull, scale, bpart, tstat);
  };
  const bool sq = kseq != nullptr;
  if (g.ns > 0) {  // sampled history (keys in token order only): Br / 4 or Br / 2, >= 4
    if (!sq) return cudaErrorInvalidValue;
    switch (g.Bk / S * 100 + g.ns) {
      case 804: return run(score_gemm_kernel<8, true, 4>);
      case 1604: return run(score_gemm_kernel<16, true, 4>);
      case 1608: return run(score_gemm_kernel<16, true, 8>);
      case 3208: return run(score_gemm_kernel<32, true, 8>);
      case 3216: return run(score_gemm_kernel<32, true, 16>);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (g.Bk / S) {  // Br: reshaped columns per KV block
    case 8: return sq ? run(score_gemm_kernel<8, true, 0>) : run(score_gemm_kernel<8, false, 0>);
    case 16: return sq ? run(score_gemm_kernel<16, true, 0>) : run(score_gemm_kernel<16, false, 0>);
    case 32: return sq ? run(score_gemm_kernel<32, true, 0>) : run(score_gemm_kernel<32, false, 0>);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace xattn
