// Estimation kernels of XAttention BSA ("XAttention BSA Policy 设计文档",
// select_blocks Steps 1-2; "XAttention Offload Stream Synchronization Fix",
// 技术细节: partial stats per KV tile -> merged stats -> normalise + block sum).
//
//   score_gemm_kernel  reshaped scores s[a,b] = scale * sum_i q[S a+S-1-i] . k[S b+i]
//                      for one (request, head, 64-row x 128-column tile), written to
//                      the fp32 score matrix, plus the tile's per-row (max, sum exp)
//   block_sum_kernel   per (request, head, query block): merges the tile statistics
//                      of its rows, then sums exp(s-m)/l over every block's cells
#include "common.cuh"

namespace xattn {
namespace {

constexpr int GM = 64;    // reshaped rows per CTA
constexpr int GN = 128;   // reshaped columns per CTA (== kTileCols)
constexpr int GK = 64;    // bf16 elements of the reshaped K dimension per stage
constexpr int GTHR = 256;
static_assert(GN == kTileCols, "statistics tile must match the GEMM N tile");

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

// 64-element (128 B) rows; 16-byte chunk c of row r lives at chunk c ^ (r & 7).
__device__ __forceinline__ int swz64(int row, int chunk) {
  return row * GK + ((chunk ^ (row & 7)) << 3);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
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

__global__ void __launch_bounds__(GTHR) score_gemm_kernel(const __grid_constant__ Geo g,
                                                          const __nv_bfloat16 *__restrict__ q,
                                                          const __nv_bfloat16 *__restrict__ kcur,
                                                          const __nv_bfloat16 *__restrict__ kpool,
                                                          float scale, float *__restrict__ scores,
                                                          float2 *__restrict__ tstat) {
  __shared__ alignas(128) __nv_bfloat16 sA[2][GM * GK];
  __shared__ alignas(128) __nv_bfloat16 sB[2][GN * GK];
  __shared__ float red[4][GM];
  __shared__ float rowm[GM];

  const int cta = blockIdx.x;
  const int r = find_req(g, cta, [](const ReqDesc &d) { return d.gemm0; });
  const ReqDesc &R = g.req[r];
  const int S = g.S, D = g.D;
  const int rq = R.lq / S, ch = R.kh / S, ncol = (R.kh + R.lq) / S;
  const int mt_n = (rq + GM - 1) / GM, nt_n = (ncol + GN - 1) / GN;
  int local = cta - R.gemm0;
  const int nt = local % nt_n;
  local /= nt_n;
  const int mt = local % mt_n;
  const int h = local / mt_n;
  const int kvh = h / (g.H / g.Hkv);
  const int m0 = mt * GM, n0 = nt * GN;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // A tile entirely right of the causal diagonal of the current chunk: no
  // visible cell, so only empty statistics are recorded.
  const int last_row = min(m0 + GM, rq) - 1;
  if (n0 >= ch && n0 - ch > last_row) {
    for (int i = tid; i < GM; i += GTHR) {
      const int a = m0 + i;
      if (a < rq)
        tstat[R.tstat_off + ((int64_t)h * rq + a) * nt_n + nt] = make_float2(-INFINITY, 0.f);
    }
    return;
  }

  // ---- loader state: each thread owns 16-byte chunk c of 2 A rows and 4 B rows
  const int c = tid & 7;
  const __nv_bfloat16 *a_base[2];
  bool a_ok[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int a = m0 + (tid >> 3) + 32 * k;
    a_ok[k] = a < rq;
    // row a of the reversed-stride reshape starts at token S*a + S-1 and walks back
    a_base[k] = q + (int64_t)h * g.q_hs + (int64_t)(R.q0 + S * (a_ok[k] ? a : 0) + S - 1) * D;
  }
  const __nv_bfloat16 *b_base[4];
  int64_t b_tstride[4];
  bool b_ok[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int b = n0 + (tid >> 3) + 32 * k;
    b_ok[k] = b < ncol;
    b_base[k] = kcur;
    b_tstride[k] = D;
    if (b_ok[k]) {
      const int t = S * b;  // first token of reshaped column b
      if (b < ch) {
        const int p = page_of(g, r, t / g.Bk);
        if (p < 0) {
          b_ok[k] = false;
        } else {
          b_base[k] = kpool + ((int64_t)(p * g.Bk + t % g.Bk) * g.Hkv + kvh) * D;
          b_tstride[k] = (int64_t)g.Hkv * D;
        }
      } else {
        b_base[k] = kcur + (int64_t)kvh * g.kv_hs + (int64_t)(R.q0 + t - R.kh) * D;
      }
    }
  }

  const int KS = S * D / GK;
  auto load_stage = [&](int ks, int stage) {
    const int kk = ks * GK + c * 8;
    const int i = kk / D, d = kk % D;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int row = (tid >> 3) + 32 * k;
      cp_async16(smem_u32(&sA[stage][swz64(row, c)]), a_base[k] - (int64_t)i * D + d, a_ok[k]);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int row = (tid >> 3) + 32 * k;
      cp_async16(smem_u32(&sB[stage][swz64(row, c)]), b_base[k] + (int64_t)i * b_tstride[k] + d,
                 b_ok[k]);
    }
  };

  float acc[2][4][4];
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int ni = 0; ni < 4; ++ni)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mi][ni][e] = 0.f;

  const int wm = warp >> 2, wn = warp & 3;
  load_stage(0, 0);
  cp_commit();
  for (int ks = 0; ks < KS; ++ks) {
    if (ks + 1 < KS) load_stage(ks + 1, (ks + 1) & 1);
    cp_commit();
    cp_wait<1>();
    __syncthreads();
    const __nv_bfloat16 *A = sA[ks & 1];
    const __nv_bfloat16 *Bm = sB[ks & 1];
#pragma unroll
    for (int kk = 0; kk < GK / 16; ++kk) {
      uint32_t af[2][4];
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) {
        const int row = wm * 32 + mi * 16 + (lane & 15);
        ldsm_x4(smem_u32(&A[swz64(row, kk * 2 + (lane >> 4))]), af[mi][0], af[mi][1], af[mi][2],
                af[mi][3]);
      }
      uint32_t bfr[4][2];
#pragma unroll
      for (int nj = 0; nj < 2; ++nj) {
        const int row = wn * 32 + nj * 16 + (lane & 7) + ((lane >> 4) << 3);
        ldsm_x4(smem_u32(&Bm[swz64(row, kk * 2 + ((lane >> 3) & 1))]), bfr[2 * nj][0],
                bfr[2 * nj][1], bfr[2 * nj + 1][0], bfr[2 * nj + 1][1]);
      }
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) mma_bf16(acc[mi][ni], af[mi], bfr[ni][0], bfr[ni][1]);
    }
    __syncthreads();
  }

  // ---- epilogue: scale, store, per-row tile statistics over visible cells

#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int al = wm * 32 + mi * 16 + (lane >> 2) + hf * 8;
      const int a = m0 + al;
      float mx = -INFINITY;
#pragma unroll
      for (int ni = 0; ni < 4; ++ni) {
        const int b = n0 + wn * 32 + ni * 8 + (lane & 3) * 2;
        float v0 = acc[mi][ni][hf * 2] * scale, v1 = acc[mi][ni][hf * 2 + 1] * scale;
        acc[mi][ni][hf * 2] = v0;
        acc[mi][ni][hf * 2 + 1] = v1;
        if (a < rq && b < ncol) {
          *reinterpret_cast<float2 *>(scores + R.score_off + ((int64_t)h * rq + a) * ncol + b) =
              make_float2(v0, v1);
          if (b < ch || b - ch <= a) mx = fmaxf(mx, v0);
          if (b + 1 < ch || b + 1 - ch <= a) mx = fmaxf(mx, v1);
        }
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      if ((lane & 3) == 0) red[wn][al] = mx;
    }
  __syncthreads();
  if (tid < GM) rowm[tid] = fmaxf(fmaxf(red[0][tid], red[1][tid]), fmaxf(red[2][tid], red[3][tid]));
  __syncthreads();
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int al = wm * 32 + mi * 16 + (lane >> 2) + hf * 8;
      const int a = m0 + al;
      const float m = rowm[al];
      float sum = 0.f;
      if (m > -INFINITY) {
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
          const int b = n0 + wn * 32 + ni * 8 + (lane & 3) * 2;
          if (a < rq && b < ncol) {
            if (b < ch || b - ch <= a) sum += __expf(acc[mi][ni][hf * 2] - m);
            if (b + 1 < ch || b + 1 - ch <= a) sum += __expf(acc[mi][ni][hf * 2 + 1] - m);
          }
        }
      }
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      sum += __shfl_xor_sync(0xffffffffu, sum, 2);
      if ((lane & 3) == 0) red[wn][al] = sum;
    }
  __syncthreads();
  if (tid < GM) {
    const int a = m0 + tid;
    if (a < rq) {
      const float l = red[0][tid] + red[1][tid] + red[2][tid] + red[3][tid];
      tstat[R.tstat_off + ((int64_t)h * rq + a) * nt_n + nt] = make_float2(rowm[tid], l);
    }
  }
}

// ---------------------------------------------------------------------------
// Merge of tile statistics + normalise and block-sum (one CTA per (r, h, qb)).
// ---------------------------------------------------------------------------
constexpr int BTHR = 256;

template <int BR>
__global__ void __launch_bounds__(BTHR) block_sum_kernel(const __grid_constant__ Geo g,
                                                         const float *__restrict__ scores,
                                                         const float2 *__restrict__ tstat,
                                                         float2 *__restrict__ rstat,
                                                         float *__restrict__ bs) {
  __shared__ float sm[BR], sil[BR];
  const int cta = blockIdx.x;
  const int r = find_req(g, cta, [](const ReqDesc &d) { return d.bsum0; });
  const ReqDesc &R = g.req[r];
  const int S = g.S;
  const int rq = R.lq / S, ch = R.kh / S, ncol = (R.kh + R.lq) / S;
  const int ntiles = (ncol + kTileCols - 1) / kTileCols;
  const int Qb = R.lq / g.Bk, Kb = ncol / BR;
  const int local = cta - R.bsum0;
  const int qb = local % Qb, h = local / Qb;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // merge: m = max_t m_t, l = sum_t l_t exp(m_t - m)
  for (int j = warp; j < BR; j += BTHR / 32) {
    const int a = qb * BR + j;
    const float2 *ts = tstat + R.tstat_off + ((int64_t)h * rq + a) * ntiles;
    float m = -INFINITY;
    for (int t = lane; t < ntiles; t += 32) m = fmaxf(m, ts[t].x);
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float l = 0.f;
    for (int t = lane; t < ntiles; t += 32) {
      const float2 v = ts[t];
      if (v.x > -INFINITY) l += v.y * __expf(v.x - m);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) {
      sm[j] = m;
      sil[j] = 1.f / l;
      rstat[R.rstat_off + (int64_t)h * rq + a] = make_float2(m, l);
    }
  }
  __syncthreads();

  constexpr int TPB = BR / 4;  // threads sharing one block's columns
  const float *base = scores + R.score_off + ((int64_t)h * rq + qb * BR) * ncol;
  // columns past the last row's diagonal are invisible to every row of this block
  const int col_end = min(ncol, ch + qb * BR + BR);
  float *out = bs + R.bs_off + ((int64_t)h * Qb + qb) * Kb;
  for (int c0 = 0; c0 < ncol / 4; c0 += BTHR) {
    const int c4 = c0 + tid;
    const int b0 = c4 * 4;
    float acc = 0.f;
    if (b0 < col_end) {
#pragma unroll
      for (int j = 0; j < BR; ++j) {
        const int a = qb * BR + j;
        const float4 v = __ldcs(reinterpret_cast<const float4 *>(base + (int64_t)j * ncol + b0));
        const float m = sm[j], il = sil[j];
        const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int b = b0 + e;
          const bool vis = b < ch || b - ch <= a;
          acc += vis ? __expf(vv[e] - m) * il : 0.f;
        }
      }
    }
#pragma unroll
    for (int o = TPB / 2; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if ((tid % TPB) == 0 && b0 < ncol) out[b0 / BR] = acc;
  }
}

}  // namespace

cudaError_t launch_score_gemm(const Geo &g, int nctas, const __nv_bfloat16 *q,
                              const __nv_bfloat16 *kcur, const __nv_bfloat16 *kpool, float scale,
                              float *scores, float2 *tstat, cudaStream_t st) {
  if (nctas == 0) return cudaSuccess;
  score_gemm_kernel<<<nctas, GTHR, 0, st>>>(g, q, kcur, kpool, scale, scores, tstat);
  return cudaGetLastError();
}

cudaError_t launch_block_sum(const Geo &g, int nctas, const float *scores, const float2 *tstat,
                             float2 *rstat, float *block_sums, cudaStream_t st) {
  if (nctas == 0) return cudaSuccess;
  const int br = g.Bk / g.S;
  switch (br) {
    case 4: block_sum_kernel<4><<<nctas, BTHR, 0, st>>>(g, scores, tstat, rstat, block_sums); break;
    case 8: block_sum_kernel<8><<<nctas, BTHR, 0, st>>>(g, scores, tstat, rstat, block_sums); break;
    case 16: block_sum_kernel<16><<<nctas, BTHR, 0, st>>>(g, scores, tstat, rstat, block_sums); break;
    case 32: block_sum_kernel<32><<<nctas, BTHR, 0, st>>>(g, scores, tstat, rstat, block_sums); break;
    case 64: block_sum_kernel<64><<<nctas, BTHR, 0, st>>>(g, scores, tstat, rstat, block_sums); break;
    case 128: block_sum_kernel<128><<<nctas, BTHR, 0, st>>>(g, scores, tstat, rstat, block_sums); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace xattn
