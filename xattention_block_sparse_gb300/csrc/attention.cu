// Block-sparse chunk attention of XAttention BSA ("XAttention BSA Policy 设计文档",
// compute_chunked_prefill): softmax attention of the current query chunk over
// the selected history pages (non-causal) and the current chunk (causal),
// with the two parts merged online by log-sum-exp inside one pass, so the
// output equals flash_attn_with_lse(history) merged with
// flash_attn_with_lse(current, causal) by merge_attention_outputs.
//
// One CTA = 128 query rows of one (request, head); 8 warps x 16 rows.  KV is
// walked in 64-token tiles: the selected pages first (gathered through the
// selection's page list), then the current chunk up to the diagonal.
#include "common.cuh"

namespace xattn {
namespace {

constexpr int AM = 128;  // query rows per CTA
constexpr int AN = 64;   // keys per tile
constexpr int ATHR = 256;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
  const int sz = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(sz));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// row-major [rows][D] bf16 tile, 16-byte chunk c of row r stored at c ^ (r & 7)
template <int D>
__device__ __forceinline__ int swz(int row, int chunk) {
  return row * D + ((chunk ^ (row & 7)) << 3);
}

template <int D>
__global__ void __launch_bounds__(ATHR) attn_kernel(
    const __grid_constant__ Geo g, const __nv_bfloat16 *__restrict__ q,
    const __nv_bfloat16 *__restrict__ kcur, const __nv_bfloat16 *__restrict__ vcur,
    const __nv_bfloat16 *__restrict__ kpool, const __nv_bfloat16 *__restrict__ vpool,
    const int32_t *__restrict__ sel_page, const int32_t *__restrict__ n_sel, float scale_log2,
    __nv_bfloat16 *__restrict__ o, float *__restrict__ lse) {
  constexpr int NCH = D / 8;  // 16-byte chunks per row
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __nv_bfloat16 *sQ = reinterpret_cast<__nv_bfloat16 *>(smem_raw);
  __nv_bfloat16 *sK = sQ + AM * D;      // [2][AN*D]
  __nv_bfloat16 *sV = sK + 2 * AN * D;  // [2][AN*D]

  const int cta = blockIdx.x;
  const int r = find_req(g, cta, [](const ReqDesc &d) { return d.att0; });
  const ReqDesc &R = g.req[r];
  const int mt_n = (R.lq + AM - 1) / AM;
  const int local = cta - R.att0;
  const int h = local % g.H;
  const int mt = mt_n - 1 - local / g.H;  // longest causal tiles first
  const int kvh = h / (g.H / g.Hkv);
  const int m0 = mt * AM;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  const int kbh = R.kh / g.Bk;
  int nh = n_sel[r];
  nh = nh < 0 ? 0 : (nh > kbh ? kbh : nh);
  const int sub = g.Bk / AN;
  const int n_hist = nh * sub;
  const int n_cur = min((m0 + AM + AN - 1) / AN, R.lq / AN);
  const int n_tiles = n_hist + n_cur;

  // ---- Q tile
  const __nv_bfloat16 *qh = q + (int64_t)h * g.q_hs + (int64_t)R.q0 * D;
  for (int id = tid; id < AM * NCH; id += ATHR) {
    const int row = id / NCH, c = id % NCH;
    const bool ok = m0 + row < R.lq;
    cp_async16(smem_u32(&sQ[swz<D>(row, c)]), qh + (int64_t)(ok ? m0 + row : 0) * D + c * 8, ok);
  }

  auto tile_src = [&](int t, const __nv_bfloat16 *&kb, const __nv_bfloat16 *&vb, int64_t &rs,
                      bool &ok) {
    if (t < n_hist) {
      const int p = sel_page[(int64_t)r * g.bt_stride + t / sub];
      ok = p >= 0 && p < g.num_pages;
      const int64_t base = ((int64_t)(ok ? p : 0) * g.Bk + (t % sub) * AN) * g.Hkv + kvh;
      kb = kpool + base * D;
      vb = vpool + base * D;
      rs = (int64_t)g.Hkv * D;
    } else {
      const int j0 = (t - n_hist) * AN;
      const int64_t base = (int64_t)R.q0 + j0;
      kb = kcur + (int64_t)kvh * g.kv_hs + base * D;
      vb = vcur + (int64_t)kvh * g.kv_hs + base * D;
      rs = D;
      ok = true;
    }
  };
  auto load_tile = [&](int t, int stage) {
    const __nv_bfloat16 *kb, *vb;
    int64_t rs;
    bool ok;
    tile_src(t, kb, vb, rs, ok);
    __nv_bfloat16 *dk = sK + stage * AN * D, *dv = sV + stage * AN * D;
    for (int id = tid; id < AN * NCH; id += ATHR) {
      const int row = id / NCH, c = id % NCH;
      cp_async16(smem_u32(&dk[swz<D>(row, c)]), kb + row * rs + c * 8, ok);
      cp_async16(smem_u32(&dv[swz<D>(row, c)]), vb + row * rs + c * 8, ok);
    }
  };

  if (n_tiles > 0) load_tile(0, 0);
  cp_commit();

  // Q fragments stay in registers for the whole KV walk
  uint32_t qf[D / 16][4];
  float oacc[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) oacc[i][e] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  const int row_a = m0 + warp * 16 + (lane >> 2);  // rows row_a and row_a + 8

  for (int t = 0; t < n_tiles; ++t) {
    if (t + 1 < n_tiles) load_tile(t + 1, (t + 1) & 1);
    cp_commit();
    cp_wait<1>();
    __syncthreads();
    if (t == 0) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int row = warp * 16 + (lane & 15);
        ldsm_x4(smem_u32(&sQ[swz<D>(row, kk * 2 + (lane >> 4))]), qf[kk][0], qf[kk][1], qf[kk][2],
                qf[kk][3]);
      }
    }
    const __nv_bfloat16 *K = sK + (t & 1) * AN * D;
    const __nv_bfloat16 *V = sV + (t & 1) * AN * D;

    // S = Q K^T  (16 x 64 per warp)
    float s[AN / 8][4];
#pragma unroll
    for (int i = 0; i < AN / 8; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[i][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int nj = 0; nj < AN / 16; ++nj) {
        uint32_t b0, b1, b2, b3;
        const int row = nj * 16 + (lane & 7) + ((lane >> 4) << 3);
        ldsm_x4(smem_u32(&K[swz<D>(row, kk * 2 + ((lane >> 3) & 1))]), b0, b1, b2, b3);
        mma_bf16(s[2 * nj], qf[kk], b0, b1);
        mma_bf16(s[2 * nj + 1], qf[kk], b2, b3);
      }
    }

    // visibility: history tiles are visible unless their page was invalid;
    // current tiles are causal (key j visible from query i iff j <= i)
    bool page_ok = true;
    int j0 = -1;
    if (t < n_hist) {
      const int p = sel_page[(int64_t)r * g.bt_stride + t / sub];
      page_ok = p >= 0 && p < g.num_pages;
      if (!page_ok && tid == 0) record_error(g.err, XATTN_EPAGE);
    } else {
      j0 = (t - n_hist) * AN;
    }
#pragma unroll
    for (int ni = 0; ni < AN / 8; ++ni)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = row_a + (e >> 1) * 8;
        const int j = j0 + ni * 8 + (lane & 3) * 2 + (e & 1);
        const bool vis = page_ok && (j0 < 0 || j <= i);
        s[ni][e] = vis ? s[ni][e] * scale_log2 : -INFINITY;
      }

    // online softmax (base 2)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      float mx = -INFINITY;
#pragma unroll
      for (int ni = 0; ni < AN / 8; ++ni) mx = fmaxf(mx, fmaxf(s[ni][hf * 2], s[ni][hf * 2 + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float mnew = fmaxf(mrow[hf], mx);
      const float base = mnew == -INFINITY ? 0.f : mnew;
      const float alpha = exp2f(mrow[hf] - base);
      mrow[hf] = mnew;
      float ls = 0.f;
#pragma unroll
      for (int ni = 0; ni < AN / 8; ++ni) {
        s[ni][hf * 2] = exp2f(s[ni][hf * 2] - base);
        s[ni][hf * 2 + 1] = exp2f(s[ni][hf * 2 + 1] - base);
        ls += s[ni][hf * 2] + s[ni][hf * 2 + 1];
      }
      lrow[hf] = lrow[hf] * alpha + ls;
#pragma unroll
      for (int di = 0; di < D / 8; ++di) {
        oacc[di][hf * 2] *= alpha;
        oacc[di][hf * 2 + 1] *= alpha;
      }
    }

    // O += P V
#pragma unroll
    for (int kk = 0; kk < AN / 16; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int dj = 0; dj < D / 16; ++dj) {
        uint32_t b0, b1, b2, b3;
        const int row = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int chunk = dj * 2 + (lane >> 4);
        ldsm_x4_t(smem_u32(&V[swz<D>(row, chunk)]), b0, b1, b2, b3);
        mma_bf16(oacc[2 * dj], pa, b0, b1);
        mma_bf16(oacc[2 * dj + 1], pa, b2, b3);
      }
    }
    __syncthreads();
  }
  cp_wait<0>();

  // ---- epilogue: O / l, LSE = ln(sum exp(logit))
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    float l = lrow[hf];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    const int i = row_a + hf * 8;
    if (i < R.lq) {
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16 *orow = o + (int64_t)h * g.q_hs + (int64_t)(R.q0 + i) * D;
#pragma unroll
      for (int di = 0; di < D / 8; ++di) {
        const int d = di * 8 + (lane & 3) * 2;
        *reinterpret_cast<__nv_bfloat162 *>(orow + d) =
            __floats2bfloat162_rn(oacc[di][hf * 2] * inv, oacc[di][hf * 2 + 1] * inv);
      }
      if ((lane & 3) == 0)
        lse[(int64_t)h * g.lse_hs + R.q0 + i] =
            l > 0.f ? (mrow[hf] + log2f(l)) * 0.6931471805599453f : -INFINITY;
    }
  }
}

template <int D>
cudaError_t launch_attn_d(const Geo &g, int nctas, const __nv_bfloat16 *q,
                          const __nv_bfloat16 *kcur, const __nv_bfloat16 *vcur,
                          const __nv_bfloat16 *kpool, const __nv_bfloat16 *vpool,
                          const int32_t *sel_page, const int32_t *n_sel, float scale,
                          __nv_bfloat16 *o, float *lse, cudaStream_t st) {
  const size_t smem = (size_t)(AM * D + 4 * AN * D) * sizeof(__nv_bfloat16);
  cudaError_t e =
      cudaFuncSetAttribute(attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  attn_kernel<D><<<nctas, ATHR, smem, st>>>(g, q, kcur, vcur, kpool, vpool, sel_page, n_sel,
                                            scale * 1.4426950408889634f, o, lse);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const Geo &g, int nctas, const __nv_bfloat16 *q,
                             const __nv_bfloat16 *kcur, const __nv_bfloat16 *vcur,
                             const __nv_bfloat16 *kpool, const __nv_bfloat16 *vpool,
                             const int32_t *sel_page, const int32_t *n_sel, float scale,
                             __nv_bfloat16 *o, float *lse, cudaStream_t st) {
  if (nctas == 0) return cudaSuccess;
  if (g.D == 128)
    return launch_attn_d<128>(g, nctas, q, kcur, vcur, kpool, vpool, sel_page, n_sel, scale, o, lse,
                              st);
  if (g.D == 64)
    return launch_attn_d<64>(g, nctas, q, kcur, vcur, kpool, vpool, sel_page, n_sel, scale, o, lse,
                             st);
  return cudaErrorInvalidValue;
}

}  // namespace xattn
