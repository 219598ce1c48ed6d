// Block-sparse chunk attention of XAttention BSA ("XAttention BSA Policy 设计文档",
// compute_chunked_prefill): softmax attention of the current query chunk over
// the selected history pages (non-causal) and the current chunk (causal),
// merged online by log-sum-exp in one pass -- the result equals
// flash_attn_with_lse(history) merged with flash_attn_with_lse(current, causal)
// by merge_attention_outputs.
//
// tcgen05 design.  One CTA = two 128-row query tiles (A and B) of one
// (request, head), sharing every K/V tile:
//   warp 0        TMA producer: both Q tiles once, then K(t), V(t) for each KV
//                 tile t (one page of up to 128 keys) through a 5-slot ring of
//                 128B-swizzled tiles.  History tiles are gathered page by page
//                 through the selection's page list, then the current chunk up
//                 to the diagonal.
//   warp 1        MMA issuer, in the order PV_A(t), S_A(t+1), PV_B(t), S_B(t+1):
//                 S_x = Q_x K^T into TMEM (128 lanes x NK fp32 columns), then
//                 O_x += P_x V into a TMEM accumulator with P_x read from TMEM.
//                 While one tile's softmax runs, the tensor pipe works for the
//                 other tile.
//   warps 4..7    softmax of tile A, warps 8..11 softmax of tile B: thread i
//                 owns query row i (TMEM lane i).  It loads its S row, masks
//                 the causal diagonal tile, keeps a running max (rescaling O in
//                 TMEM only when the max grows by more than 2^8), writes P as
//                 bf16 back into the TMEM columns its S row came from (the P V
//                 MMA reads its A operand there, so P costs no shared-memory
//                 bandwidth), and at the end normalises O and writes O, LSE.
// Each thread's tcgen05 ops complete in issue order: S_x(t) being ready
// implies PV_x(t-1) has finished, so O_x may be rescaled and S_x's columns
// reused for P_x(t) without further waits.
// Every mbarrier wait is bounded; a timeout records XATTN_ETIMEOUT and the CTA
// unwinds (draining its TMA loads and MMAs, then freeing TMEM).
#include "tc_common.cuh"

namespace xattn {
namespace {
using namespace tc;

constexpr int BM = 128;       // rows per query tile (MMA M)
constexpr int ROWS = 2 * BM;  // query rows per CTA
static_assert(ROWS == kAttnRows, "host grid sizing assumes kAttnRows rows per CTA");
constexpr int NSLOT = 5;      // K/V ring slots
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
  static constexpr int BYTES = OFF_BAR + 256;
  static constexpr int SMEM_ALLOC = BYTES + 1024;  // slack to align the base to 1024
};

struct Bars {
  uint64_t q_full;
  uint64_t full[NSLOT];
  uint64_t empty[NSLOT];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t pv_done[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

struct TMaps {
  CUtensorMap q, kc, vc, kp, vp;
};

template <int D, int NK>
__global__ void __launch_bounds__(THREADS, 1)
    attn_tc_kernel(const __grid_constant__ Geo g, const __grid_constant__ TMaps tm,
                   const int32_t *__restrict__ sel_page, const int32_t *__restrict__ n_sel,
                   float scale_log2, __nv_bfloat16 *__restrict__ o, float *__restrict__ lse) {
  using LY = Layout<D, NK>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars &bar = *reinterpret_cast<Bars *>(smem + LY::OFF_BAR);
  volatile int *abort = &bar.abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x;
  const int r = find_req(g, cta, [](const ReqDesc &d) { return d.att0; });
  const ReqDesc &R = g.req[r];
  const int mt_n = (R.lq + ROWS - 1) / ROWS;
  const int local = cta - R.att0;
  const int G = g.H / g.Hkv;
  // longest causal tiles first, all heads of a row tile together
  const int h = local % g.H;
  const int mt = mt_n - 1 - local / g.H;
  const int kvh = h / G;
  const int m0 = mt * ROWS;
  const bool has_b = m0 + BM < R.lq;

  const int kbh = R.kh / g.Bk;
  int nh = n_sel[r];
  nh = nh < 0 ? 0 : (nh > kbh ? kbh : nh);
  const int sub = g.Bk / NK;
  const int n_hist = nh * sub;
  // current-chunk tiles up to the last row of each query tile
  const int n_a = n_hist + (min(m0 + BM, R.lq) - 1) / NK + 1;
  const int n_b = has_b ? n_hist + (min(m0 + ROWS, R.lq) - 1) / NK + 1 : 0;
  const int n_tiles = has_b ? n_b : n_a;
  const int32_t *pages = sel_page + (int64_t)r * g.bt_stride;

  if (tid == 0) {
    mbar_init(&bar.q_full, 1);
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(&bar.full[s], 1);
      mbar_init(&bar.empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bar.s_full[x], 1);
      mbar_init(&bar.p_full[x], 4);  // one arrival per softmax warp
      mbar_init(&bar.pv_done[x], 1);
    }
    mbar_init(&bar.drain, 1);
    bar.abort = 0;
    fence_mbar_init();
  }
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
      if (n_hist) {
        tma_prefetch_desc(&tm.kp);
        tma_prefetch_desc(&tm.vp);
      }
      mbar_expect_tx(&bar.q_full, (has_b ? 2 : 1) * LY::Q_BYTES);
      for (int x = 0; x < (has_b ? 2 : 1); ++x)
        for (int hf = 0; hf < LY::HALVES; ++hf)
          tma_load_3d(smem + LY::OFF_Q + x * LY::Q_BYTES + hf * (BM * 128), &tm.q, &bar.q_full,
                      hf * 64, R.q0 + m0 + x * BM, h);
    }
    int issued = 0;  // loads: K(t) = 2t, V(t) = 2t+1
    int pg = 0;      // page id of tile (t & ~31) + lane
    for (int i = 0; i < 2 * n_tiles; ++i) {
      const int t = i >> 1;
      if ((i & 63) == 0) {  // next 32 tiles' page ids, one per lane
        const int tt = t + lane;
        pg = tt < n_hist ? __ldg(pages + tt / sub) : 0;
      }
      const int p_t = __shfl_sync(0xffffffffu, pg, t & 31);
      const int s = i % NSLOT;
      int ok = 1;  // lane 0 waits, the warp follows its verdict
      if (lane == 0 && i >= NSLOT) ok = mbar_wait(&bar.empty[s], ((i / NSLOT) - 1) & 1, abort, g.err);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (lane == 0) {
        const bool is_v = i & 1;
        uint8_t *dst = smem + LY::OFF_KV + s * LY::KV_BYTES;
        mbar_expect_tx(&bar.full[s], LY::KV_BYTES);
        if (t < n_hist) {
          const int p = (p_t < 0 || p_t >= g.num_pages) ? 0 : p_t;  // masked by the softmax
          const int tok = (t % sub) * NK;
          for (int hf = 0; hf < LY::HALVES; ++hf)
            tma_load_4d(dst + hf * (NK * 128), is_v ? &tm.vp : &tm.kp, &bar.full[s], hf * 64,
                        kvh, tok, p);
        } else {
          const int j0 = (t - n_hist) * NK;
          for (int hf = 0; hf < LY::HALVES; ++hf)
            tma_load_3d(dst + hf * (NK * 128), is_v ? &tm.vc : &tm.kc, &bar.full[s], hf * 64,
                        R.q0 + j0, kvh);
        }
      }
      issued = i + 1;
    }
    // drain: every load issued must land before shared memory is released
    // (only the last NSLOT can still be in flight)
    if (lane == 0) {
      for (uint32_t k = 0; k < kSpinLimit && !mbar_try_wait(&bar.q_full, 0); ++k) {
      }
      for (int i = max(0, issued - NSLOT); i < issued; ++i) {
        const uint32_t par = (i / NSLOT) & 1;
        for (uint32_t k = 0; k < kSpinLimit && !mbar_try_wait(&bar.full[i % NSLOT], par); ++k) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(BM, NK, 0, 0);
      constexpr uint32_t idPV = idesc_bf16(BM, D, 0, 1);
      const uint32_t sQ = smem_addr(smem + LY::OFF_Q);
      const uint32_t sKV = smem_addr(smem + LY::OFF_KV);
      auto slot_wait = [&](int i) {
        return mbar_wait(&bar.full[i % NSLOT], (i / NSLOT) & 1, abort, g.err);
      };
      // Descriptors are built once; a k-step only adds its byte offset / 16 to
      // the start-address field (all operands lie below 256 KB of shared memory).
      const uint64_t dQ0 = sdesc_sw128(sQ, 16, 1024);
      const uint64_t dK0 = sdesc_sw128(sKV, 16, 1024);
      const uint64_t dV0 = sdesc_sw128(sKV, NK * 128, 1024);
      auto issue_S = [&](int x, int t) {
        const uint64_t a0 = dQ0 + (uint64_t)((x * LY::Q_BYTES) >> 4);
        const uint64_t b0 = dK0 + (uint64_t)((((2 * t) % NSLOT) * LY::KV_BYTES) >> 4);
        const uint32_t d = tmem + x * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_f16_ss(d, a0 + (uint64_t)(((kk / 4) * (BM * 128) + (kk % 4) * 32) >> 4),
                     b0 + (uint64_t)(((kk / 4) * (NK * 128) + (kk % 4) * 32) >> 4), idS,
                     kk > 0 ? 1u : 0u);
        mma_commit(&bar.s_full[x]);
      };
      auto issue_PV = [&](int x, int t) {
        const uint64_t b0 = dV0 + (uint64_t)((((2 * t + 1) % NSLOT) * LY::KV_BYTES) >> 4);
        const uint32_t d = tmem + 256 + x * 128;
        const uint32_t a = tmem + x * 128;
        // A = P in TMEM (16 keys = 8 columns per step); B = V, MN-major
        // (d contiguous): the two 64-wide d blocks are NK*128 bytes apart,
        // 8-key groups 1024 apart
#pragma unroll
        for (int kk = 0; kk < NK / 16; ++kk)
          mma_f16_ts(d, a + kk * 8, b0 + (uint64_t)((kk * 2048) >> 4), idPV,
                     (t > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bar.pv_done[x]);
      };
      bool ok = mbar_wait(&bar.q_full, 0, abort, g.err);
      if (ok && n_tiles > 0) {
        ok = slot_wait(0);
        if (ok) {
          tc_fence_after();
          issue_S(0, 0);
          if (has_b) issue_S(1, 0);
          mma_commit(&bar.empty[0]);
        }
      }
      for (int t = 0; ok && t < n_tiles; ++t) {
        const bool a_now = t < n_a, a_next = t + 1 < n_a;
        const bool b_now = t < n_b, b_next = t + 1 < n_b;
        const bool next = t + 1 < n_tiles;
        if (!slot_wait(2 * t + 1)) break;  // V(t)
        if (a_now) {
          if (!mbar_wait(&bar.p_full[0], t & 1, abort, g.err)) break;
          tc_fence_after();
          issue_PV(0, t);
        }
        if (next && !slot_wait(2 * t + 2)) break;  // K(t+1)
        if (a_next) {  // the softmax has consumed S_A(t): it arrived p_full
          tc_fence_after();
          issue_S(0, t + 1);
        }
        if (b_now) {
          if (!mbar_wait(&bar.p_full[1], t & 1, abort, g.err)) break;
          tc_fence_after();
          issue_PV(1, t);
        }
        mma_commit(&bar.empty[(2 * t + 1) % NSLOT]);  // V(t) consumed
        if (b_next) {
          tc_fence_after();
          issue_S(1, t + 1);
        }
        if (next) mma_commit(&bar.empty[(2 * t + 2) % NSLOT]);  // K(t+1) consumed
      }
      // every MMA issued has completed before TMEM is freed
      mma_commit(&bar.drain);
      for (uint32_t k = 0; k < kSpinLimit && !mbar_try_wait(&bar.drain, 0); ++k) {
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int x = (warp - 4) >> 2;         // query tile: 0 = A, 1 = B
    const int n_x = x ? n_b : n_a;
    const int row = tid - 128 - x * BM;    // row within the tile == TMEM lane
    const int qrow = m0 + x * BM + row;    // chunk-local query index
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const uint32_t s_col = x * 128, o_col = 256 + x * 128;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    int p_next = (n_hist > 0) ? __ldg(pages) : 0;
    for (int t = 0; t < n_x; ++t) {
      const int p_cur = p_next;
      if (t + 1 < n_hist) p_next = __ldg(pages + (t + 1) / sub);
      if (!mbar_wait(&bar.s_full[x], t & 1, abort, g.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[NK];
#pragma unroll
      for (int c = 0; c < NK / 32; ++c)
        tmem_ld32(lane_addr + s_col + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
      tmem_ld_wait();

      if (t < n_hist) {
        if (p_cur < 0 || p_cur >= g.num_pages) {  // invalid page: skip its keys
#pragma unroll
          for (int j = 0; j < NK; ++j) sr[j] = __float_as_uint(-INFINITY);
          if (row == 0 && (t % sub) == 0) record_error(g.err, XATTN_EPAGE);
        }
      } else {
        const int lim = qrow - (t - n_hist) * NK + 1;  // keys [0, lim) are visible
        if (lim < NK) {
#pragma unroll
          for (int j = 0; j < NK; ++j)
            if (j >= lim) sr[j] = __float_as_uint(-INFINITY);
        }
      }
      // softmax_scale > 0, so the row max of the scaled logits is the scaled max
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int j = 0; j < NK; j += 8)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          m4[e] = fmax3(m4[e], __uint_as_float(sr[j + 2 * e]), __uint_as_float(sr[j + 2 * e + 1]));
      const float mt = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3])) * scale_log2;
      const float mnew = fmaxf(m_run, mt);
      const bool need = mnew > m_run + 8.f;
      const float alpha = need ? ex2(m_run - mnew) : 1.f;
      const float m_use = need ? mnew : m_run;
      const float nb = m_use == -INFINITY ? 0.f : -m_use;
      const uint64_t sc2 = f2(scale_log2, scale_log2), nb2 = f2(nb, nb);
      uint64_t sum2[4] = {0ull, 0ull, 0ull, 0ull};
      // P row -> the S row's TMEM columns (two bf16 per column), the A operand
      // of P V, 64 keys at a time; PV_x(t-1) finished before S_x(t) did
#pragma unroll
      for (int hb = 0; hb < NK / 64; ++hb) {
        uint32_t pk[32];
#pragma unroll
        for (int j = 0; j < 64; j += 2) {
          float x0, x1;
          unf2(ffma2(f2(__uint_as_float(sr[hb * 64 + j]), __uint_as_float(sr[hb * 64 + j + 1])),
                     sc2, nb2),
               x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          sum2[(j >> 1) & 3] = fadd2(sum2[(j >> 1) & 3], f2(p0, p1));
          pk[j >> 1] = pack_bf16x2(p0, p1);
        }
        tmem_st32(lane_addr + s_col + hb * 32, pk);
      }
      float s0, s1, s2, s3;
      unf2(fadd2(sum2[0], sum2[1]), s0, s1);
      unf2(fadd2(sum2[2], sum2[3]), s2, s3);
      l_run = l_run * alpha + ((s0 + s1) + (s2 + s3));
      m_run = m_use;
      if (t > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(lane_addr + o_col + c * 32, ov);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
          tmem_st32(lane_addr + o_col + c * 32, ov);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.p_full[x]);
    }
    // epilogue: wait for the last P V, normalise, write O and LSE
    if (ok && n_x > 0 && mbar_wait(&bar.pv_done[x], (n_x - 1) & 1, abort, g.err)) {
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      const bool wr = qrow < R.lq;
      __nv_bfloat16 *orow = o + (int64_t)h * g.q_hs + (int64_t)(R.q0 + qrow) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(lane_addr + o_col + c * 32, ov);
        tmem_ld_wait();
        if (wr) {
#pragma unroll
          for (int j = 0; j < 32; j += 8) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(ov[j]) * inv, __uint_as_float(ov[j + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(ov[j + 2]) * inv, __uint_as_float(ov[j + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(ov[j + 4]) * inv, __uint_as_float(ov[j + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(ov[j + 6]) * inv, __uint_as_float(ov[j + 7]) * inv);
            *reinterpret_cast<uint4 *>(orow + c * 32 + j) = v;
          }
        }
      }
      if (wr)
        lse[(int64_t)h * g.lse_hs + R.q0 + qrow] =
            l_run > 0.f ? (m_run + __log2f(l_run)) * 0.6931471805599453f : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

// ---------------------------------------------------------------------------
// Host side: tensor maps and launch
// ---------------------------------------------------------------------------
template <int D, int NK>
cudaError_t launch_tc(const Geo &g, int nctas, const __nv_bfloat16 *q, const __nv_bfloat16 *kcur,
                      const __nv_bfloat16 *vcur, const __nv_bfloat16 *kpool,
                      const __nv_bfloat16 *vpool, const int32_t *sel_page, const int32_t *n_sel,
                      float scale, __nv_bfloat16 *o, float *lse, cudaStream_t st) {
  TMaps tm;
  const int64_t tot_q = (int64_t)g.req[g.B - 1].q0 + g.req[g.B - 1].lq;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)tot_q, (cuuint64_t)g.H};
    const cuuint64_t str[2] = {(cuuint64_t)D * 2, (cuuint64_t)g.q_hs * 2};
    const cuuint32_t box[3] = {64, BM, 1};
    if (!encode_bf16(&tm.q, q, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)tot_q, (cuuint64_t)g.Hkv};
    const cuuint64_t str[2] = {(cuuint64_t)D * 2, (cuuint64_t)g.kv_hs * 2};
    const cuuint32_t box[3] = {64, NK, 1};
    if (!encode_bf16(&tm.kc, kcur, 3, dims, str, box)) return cudaErrorInvalidValue;
    if (!encode_bf16(&tm.vc, vcur, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  if (g.num_pages > 0 && kpool && vpool) {
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)g.Hkv, (cuuint64_t)g.Bk,
                                (cuuint64_t)g.num_pages};
    const cuuint64_t str[3] = {(cuuint64_t)D * 2, (cuuint64_t)g.Hkv * D * 2,
                               (cuuint64_t)g.Bk * g.Hkv * D * 2};
    const cuuint32_t box[4] = {64, 1, NK, 1};
    if (!encode_bf16(&tm.kp, kpool, 4, dims, str, box)) return cudaErrorInvalidValue;
    if (!encode_bf16(&tm.vp, vpool, 4, dims, str, box)) return cudaErrorInvalidValue;
  } else {
    tm.kp = tm.kc;
    tm.vp = tm.vc;
  }
  using LY = Layout<D, NK>;
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D, NK>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, LY::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  attn_tc_kernel<D, NK><<<nctas, THREADS, LY::SMEM_ALLOC, st>>>(
      g, tm, sel_page, n_sel, scale * 1.4426950408889634f, o, lse);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const Geo &g, int nctas, const __nv_bfloat16 *q,
                             const __nv_bfloat16 *kcur, const __nv_bfloat16 *vcur,
                             const __nv_bfloat16 *kpool, const __nv_bfloat16 *vpool,
                             const int32_t *sel_page, const int32_t *n_sel, float scale,
                             __nv_bfloat16 *o, float *lse, cudaStream_t st) {
  if (nctas == 0) return cudaSuccess;
  const bool wide = g.Bk % 128 == 0;  // KV tile: 128 keys, else 64
  if (g.D == 128)
    return wide ? launch_tc<128, 128>(g, nctas, q, kcur, vcur, kpool, vpool, sel_page, n_sel,
                                      scale, o, lse, st)
                : launch_tc<128, 64>(g, nctas, q, kcur, vcur, kpool, vpool, sel_page, n_sel,
                                     scale, o, lse, st);
  if (g.D == 64)
    return wide ? launch_tc<64, 128>(g, nctas, q, kcur, vcur, kpool, vpool, sel_page, n_sel,
                                     scale, o, lse, st)
                : launch_tc<64, 64>(g, nctas, q, kcur, vcur, kpool, vpool, sel_page, n_sel,
                                    scale, o, lse, st);
  return cudaErrorInvalidValue;
}

}  // namespace xattn
