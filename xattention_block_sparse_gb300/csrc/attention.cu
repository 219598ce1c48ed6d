// Block-sparse chunk attention of XAttention BSA ("XAttention BSA Policy 设计文档",
// compute_chunked_prefill): softmax attention of the current query chunk over
// the selected history pages (non-causal) and the current chunk (causal),
// merged online by log-sum-exp in one pass -- the result equals
// flash_attn_with_lse(history) merged with flash_attn_with_lse(current, causal)
// by merge_attention_outputs.
//
// tcgen05 design.  One CTA = 128 query rows of one (request, head).
//   warp 0       TMA producer: Q tile once, then K and V tiles (one page of up to
//                128 keys each) through an NST-stage ring; history tiles are
//                gathered page by page from the pool through the selection's
//                page list, then the current chunk up to the diagonal.
//   warp 1       MMA issuer: S = Q K^T into one of two TMEM buffers (128 lanes x
//                NK fp32 columns), then O += P V into a TMEM accumulator.
//   warps 4..7   softmax: thread i owns query row i (TMEM lane i).  It loads its
//                S row, applies scale and causal mask, keeps a running max
//                (rescaling O in TMEM only when the max grows by more than
//                2^8), writes P as bf16 into 128B-swizzled shared memory for
//                the P V MMA, and finally normalises O and writes O and LSE.
// Every mbarrier wait is bounded; a timeout records XATTN_ETIMEOUT and the CTA
// unwinds (waiting for its own TMA loads and MMAs, then freeing TMEM).
#include <cudaTypedefs.h>

#include "tc_common.cuh"

namespace xattn {
namespace {
using namespace tc;

constexpr int BM = 128;      // query rows per CTA
constexpr int NST = 2;       // K/V pipeline stages
constexpr int THREADS = 256;
constexpr int TMEM_COLS = 512;
constexpr int TM_S = 0;      // S buffers at columns 0 and 128
constexpr int TM_O = 256;    // O accumulator at columns 256 .. 256+D

template <int D, int NK>
struct Layout {
  static constexpr int HALVES = D / 64;             // 64-element (128 B) column blocks
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int KV_BYTES = NK * D * 2;
  static constexpr int P_BYTES = BM * NK * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + NST * KV_BYTES;
  static constexpr int OFF_P = OFF_V + NST * KV_BYTES;
  static constexpr int OFF_BAR = OFF_P + P_BYTES;
  static constexpr int BYTES = OFF_BAR + 256;
  static constexpr int SMEM_ALLOC = BYTES + 1024;  // slack to align the base to 1024
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[NST];
  uint64_t v_full[NST];
  uint64_t kv_empty[NST];
  uint64_t s_full[2];
  uint64_t p_full;
  uint64_t pv_done;
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
  const int mt_n = (R.lq + BM - 1) / BM;
  const int local = cta - R.att0;
  const int h = local % g.H;
  const int mt = mt_n - 1 - local / g.H;  // longest causal tiles first
  const int kvh = h / (g.H / g.Hkv);
  const int m0 = mt * BM;

  const int kbh = R.kh / g.Bk;
  int nh = n_sel[r];
  nh = nh < 0 ? 0 : (nh > kbh ? kbh : nh);
  const int sub = g.Bk / NK;
  const int n_hist = nh * sub;
  const int n_cur = min((m0 + BM + NK - 1) / NK, R.lq / NK);
  const int n_tiles = n_hist + n_cur;
  const int32_t *pages = sel_page + (int64_t)r * g.bt_stride;

  if (tid == 0) {
    mbar_init(&bar.q_full, 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&bar.k_full[s], 1);
      mbar_init(&bar.v_full[s], 1);
      mbar_init(&bar.kv_empty[s], 1);
    }
    mbar_init(&bar.s_full[0], 1);
    mbar_init(&bar.s_full[1], 1);
    mbar_init(&bar.p_full, 4);  // one arrival per softmax warp
    mbar_init(&bar.pv_done, 1);
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
    if (lane == 0) {
      tma_prefetch_desc(&tm.q);
      tma_prefetch_desc(&tm.kc);
      tma_prefetch_desc(&tm.vc);
      if (n_hist) {
        tma_prefetch_desc(&tm.kp);
        tma_prefetch_desc(&tm.vp);
      }
      uint8_t *sQ = smem + LY::OFF_Q;
      mbar_expect_tx(&bar.q_full, LY::Q_BYTES);
      for (int hf = 0; hf < LY::HALVES; ++hf)
        tma_load_3d(sQ + hf * (BM * 128), &tm.q, &bar.q_full, hf * 64, R.q0 + m0, h);
      int issued = 0;
      for (int t = 0; t < n_tiles; ++t) {
        const int s = t % NST;
        if (t >= NST && !mbar_wait(&bar.kv_empty[s], ((t / NST) - 1) & 1, abort, g.err)) break;
        uint8_t *sK = smem + LY::OFF_K + s * LY::KV_BYTES;
        uint8_t *sV = smem + LY::OFF_V + s * LY::KV_BYTES;
        mbar_expect_tx(&bar.k_full[s], LY::KV_BYTES);
        mbar_expect_tx(&bar.v_full[s], LY::KV_BYTES);
        if (t < n_hist) {
          int p = __ldg(pages + t / sub);
          if (p < 0 || p >= g.num_pages) p = 0;  // masked by the softmax warps
          const int tok = (t % sub) * NK;
          for (int hf = 0; hf < LY::HALVES; ++hf)
            tma_load_4d(sK + hf * (NK * 128), &tm.kp, &bar.k_full[s], hf * 64, kvh, tok, p);
          for (int hf = 0; hf < LY::HALVES; ++hf)
            tma_load_4d(sV + hf * (NK * 128), &tm.vp, &bar.v_full[s], hf * 64, kvh, tok, p);
        } else {
          const int j0 = (t - n_hist) * NK;
          for (int hf = 0; hf < LY::HALVES; ++hf)
            tma_load_3d(sK + hf * (NK * 128), &tm.kc, &bar.k_full[s], hf * 64, R.q0 + j0, kvh);
          for (int hf = 0; hf < LY::HALVES; ++hf)
            tma_load_3d(sV + hf * (NK * 128), &tm.vc, &bar.v_full[s], hf * 64, R.q0 + j0, kvh);
        }
        issued = t + 1;
      }
      // drain: every load issued must have landed before the CTA's shared
      // memory is released (only the last NST can still be in flight)
      mbar_wait(&bar.q_full, 0, abort, g.err);
      for (int t = max(0, issued - NST); t < issued; ++t) {
        const int s = t % NST;
        const uint32_t par = (t / NST) & 1;
        for (uint32_t i = 0; i < kSpinLimit && !mbar_try_wait(&bar.k_full[s], par); ++i) {
        }
        for (uint32_t i = 0; i < kSpinLimit && !mbar_try_wait(&bar.v_full[s], par); ++i) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(BM, NK, 0, 0);
      constexpr uint32_t idPV = idesc_bf16(BM, D, 0, 1);
      const uint32_t sQ = smem_addr(smem + LY::OFF_Q);
      const uint32_t sP = smem_addr(smem + LY::OFF_P);
      bool ok = mbar_wait(&bar.q_full, 0, abort, g.err);
      auto issue_S = [&](int t) -> bool {
        const int s = t % NST;
        if (!mbar_wait(&bar.k_full[s], (t / NST) & 1, abort, g.err)) return false;
        tc_fence_after();
        const uint32_t sK = smem_addr(smem + LY::OFF_K + s * LY::KV_BYTES);
        const uint32_t d = tmem + TM_S + (t & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t a = sdesc_sw128(sQ + (kk / 4) * (BM * 128) + (kk % 4) * 32, 16, 1024);
          const uint64_t b = sdesc_sw128(sK + (kk / 4) * (NK * 128) + (kk % 4) * 32, 16, 1024);
          mma_f16_ss(d, a, b, idS, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bar.s_full[t & 1]);
        return true;
      };
      auto issue_PV = [&](int t) -> bool {
        const int s = t % NST;
        if (!mbar_wait(&bar.v_full[s], (t / NST) & 1, abort, g.err)) return false;
        if (!mbar_wait(&bar.p_full, t & 1, abort, g.err)) return false;
        tc_fence_after();
        const uint32_t sV = smem_addr(smem + LY::OFF_V + s * LY::KV_BYTES);
#pragma unroll
        for (int kk = 0; kk < NK / 16; ++kk) {
          // A = P, K-major over keys; B = V, MN-major (d contiguous): the two
          // 64-wide d blocks are NK*128 bytes apart, 8-key groups 1024 apart
          const uint64_t a = sdesc_sw128(sP + (kk / 4) * (BM * 128) + (kk % 4) * 32, 16, 1024);
          const uint64_t b = sdesc_sw128(sV + kk * 2048, NK * 128, 1024);
          mma_f16_ss(tmem + TM_O, a, b, idPV, (t > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bar.pv_done);
        mma_commit(&bar.kv_empty[s]);
        return true;
      };
      if (ok && n_tiles > 0) ok = issue_S(0);
      for (int t = 0; ok && t < n_tiles; ++t) {
        if (t + 1 < n_tiles && !issue_S(t + 1)) break;
        if (!issue_PV(t)) break;
      }
      // every MMA issued has completed before TMEM is freed
      mma_commit(&bar.drain);
      for (uint32_t i = 0; i < kSpinLimit && !mbar_try_wait(&bar.drain, 0); ++i) {
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int row = tid - 128;             // query row within the tile == TMEM lane
    const int qrow = m0 + row;             // chunk-local query index
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp - 4)) << 16);
    uint8_t *sP = smem + LY::OFF_P;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int t = 0; t < n_tiles; ++t) {
      if (!mbar_wait(&bar.s_full[t & 1], (t >> 1) & 1, abort, g.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sraw[NK / 32][32];
#pragma unroll
      for (int c = 0; c < NK / 32; ++c) tmem_ld32(lane_addr + TM_S + (t & 1) * 128 + c * 32, sraw[c]);
      tmem_ld_wait();

      // visibility of this tile's keys
      bool all_vis = true, none_vis = false;
      int lim = NK;  // keys [0, lim) visible
      if (t < n_hist) {
        const int p = __ldg(pages + t / sub);
        if (p < 0 || p >= g.num_pages) {
          none_vis = true;
          if (row == 0 && (t % sub) == 0) record_error(g.err, XATTN_EPAGE);
        }
      } else {
        const int j0 = (t - n_hist) * NK;
        lim = qrow - j0 + 1;
        if (lim < NK) all_vis = false;
        if (lim <= 0) none_vis = true;
      }
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < NK / 32; ++c)
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          float x = __uint_as_float(sraw[c][j]) * scale_log2;
          if (none_vis || (!all_vis && c * 32 + j >= lim)) x = -INFINITY;
          sraw[c][j] = __float_as_uint(x);
          mt = fmaxf(mt, x);
        }
      const float mnew = fmaxf(m_run, mt);
      const bool need = mnew > m_run + 8.f;
      const float alpha = need ? ex2(m_run - mnew) : 1.f;
      const float m_use = need ? mnew : m_run;
      const float base = m_use == -INFINITY ? 0.f : m_use;
      float rs = 0.f;
      uint32_t pk[NK / 2];
#pragma unroll
      for (int c = 0; c < NK / 32; ++c)
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float p0 = ex2(__uint_as_float(sraw[c][j]) - base);
          const float p1 = ex2(__uint_as_float(sraw[c][j + 1]) - base);
          rs += p0 + p1;
          pk[(c * 32 + j) / 2] = pack_bf16x2(p0, p1);
        }
      l_run = l_run * alpha + rs;
      m_run = m_use;

      // P buffer and O are free once the previous P V has completed
      if (t > 0 && !mbar_wait(&bar.pv_done, (t - 1) & 1, abort, g.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (t > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(lane_addr + TM_O + c * 32, ov);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
          tmem_st32(lane_addr + TM_O + c * 32, ov);
        }
        tmem_st_wait();
      }
      // P row -> 128B-swizzled K-major tile (64-key column blocks)
#pragma unroll
      for (int ch = 0; ch < NK / 8; ++ch) {
        const int blk = ch / 8, cc = ch % 8;
        uint8_t *dst = sP + blk * (BM * 128) + row * 128 + ((cc ^ (row & 7)) << 4);
        *reinterpret_cast<uint4 *>(dst) =
            make_uint4(pk[ch * 4], pk[ch * 4 + 1], pk[ch * 4 + 2], pk[ch * 4 + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.p_full);
    }
    // epilogue: wait for the last P V, normalise, write O and LSE
    if (ok && n_tiles > 0 && mbar_wait(&bar.pv_done, (n_tiles - 1) & 1, abort, g.err)) {
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      const bool wr = qrow < R.lq;
      __nv_bfloat16 *orow = o + (int64_t)h * g.q_hs + (int64_t)(R.q0 + qrow) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(lane_addr + TM_O + c * 32, ov);
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
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

bool encode_bf16(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims,
                 const cuuint64_t *strides, const cuuint32_t *box) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(base), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

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
