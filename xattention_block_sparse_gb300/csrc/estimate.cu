// Block-sum kernel of XAttention BSA estimation ("XAttention BSA Policy 设计文档",
// select_blocks Step 2 softmax_fuse_block_sum; "XAttention Offload Stream
// Synchronization Fix", 技术细节 Stages 2 and 3: merge of the per-tile softmax
// statistics, then normalise and block-sum with the merged statistics).
// The score GEMM that produces the scores and tile statistics is in
// score_gemm.cu.
//
//   block_sum_kernel   per (request, head, query block): merges the tile statistics
//                      of its rows, then sums exp(s-m)/l over every block's cells
#include "common.cuh"

namespace xattn {
namespace {

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

  // merge: m = max_t m_t, l = sum_t l_t exp(m_t - m), over the statistics
  // tiles that hold visible cells of the row (columns up to ch + a)
  for (int j = warp; j < BR; j += BTHR / 32) {
    const int a = qb * BR + j;
    const float2 *ts = tstat + R.tstat_off + ((int64_t)h * rq + a) * ntiles;
    const int nt_a = min(ntiles, (ch + a) / kTileCols + 1);
    float m = -INFINITY;
    for (int t = lane; t < nt_a; t += 32) m = fmaxf(m, ts[t].x);
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float l = 0.f;
    for (int t = lane; t < nt_a; t += 32) {
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
