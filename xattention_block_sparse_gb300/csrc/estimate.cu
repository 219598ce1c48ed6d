// Block sums of XAttention BSA estimation ("XAttention BSA Policy 设计文档",
// select_blocks Step 2 softmax_fuse_block_sum; "XAttention Offload Stream
// Synchronization Fix", 技术细节 Stages 2 and 3: merge of the per-tile softmax
// statistics, then normalise and block-sum with the merged statistics).
//
// The score GEMM (score_gemm.cu) leaves, per reshaped row a and 128-column
// statistics tile t, the tile max m_t and sum l_t over the visible cells, and
// per KV block kb the partial sum P[a][kb] = sum exp(s - m_t(kb)) over the
// block's visible cells.  block_sum_kernel, one CTA per (request, head, query
// block):
//   A2  per row a of the block: m = max_t m_t, l = sum_t l_t e^(m_t - m)
//       over the tiles that hold visible cells of the row;
//   A3  per KV block kb: BS = sum over the block's Br rows of
//       P[a][kb] e^(m_t(kb) - m_a) / l_a,
// which is the sum of exp(s - m)/l over the block's visible cells.
// With a sampled history (ReqDesc::samp) the GEMM's columns are the sampled
// history columns (g.ns per block, padded to hc) then the current chunk's;
// the partials and tile sums already carry the samples' weight, and only the
// tile of each block moves.
#include "common.cuh"

namespace xattn {
namespace {

constexpr int BTHR = 256;

template <int BR>
__global__ void __launch_bounds__(BTHR) block_sum_kernel(const __grid_constant__ Geo g,
                                                         const float *__restrict__ bpart,
                                                         const float2 *__restrict__ tstat,
                                                         float *__restrict__ bs) {
  static_assert(BR >= 8 && BR <= 32 && BR % 4 == 0, "block-sum geometry");
  __shared__ float sm[BR], sil[BR];
  // launched as a programmatic dependent of the score GEMM before it: its
  // partials and statistics are complete and visible once this returns
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int cta = blockIdx.x;
  const int r = find_req(g, cta, [](const ReqDesc &d) { return d.bsum0; });
  const ReqDesc &R = g.req[r];
  const int S = g.S;
  const int rq = R.lq / S, ch = R.hc, ncol = R.hc + rq;  // ch: columns before the chunk's
  const int ntile = (ncol + kTileCols - 1) / kTileCols;
  const int Qb = R.lq / g.Bk, Kbh = R.kh / g.Bk, Kb = Kbh + Qb;
  const int hw = R.samp ? g.ns : BR;  // history columns of a block in the GEMM
  const int local = cta - R.bsum0;
  const int qb = local % Qb, h = local / Qb;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float2 *ts_h = tstat + R.tstat_off + (int64_t)h * rq * ntile;

  // A2: one warp per row of the query block
  for (int rr = warp; rr < BR; rr += BTHR / 32) {
    const int a = qb * BR + rr;
    const float2 *ts = ts_h + (int64_t)a * ntile;
    const int nt_a = min(ntile, (ch + a) / kTileCols + 1);
    float m = -INFINITY;
    for (int t = lane; t < nt_a; t += 32) m = fmaxf(m, ts[t].x);
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float l = 0.f;
    for (int t = lane; t < nt_a; t += 32) {
      const float2 w = ts[t];
      if (w.x > -INFINITY) l += w.y * __expf(w.x - m);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) {
      sm[rr] = m;
      sil[rr] = 1.f / l;  // every row sees at least its own diagonal cell: l > 0
    }
  }
  __syncthreads();

  // A3: one thread per KV block; its Br partials are contiguous
  const float *pq = bpart + R.bpart_off + (int64_t)(h * Qb + qb) * Kb * BR;
  float *out = bs + R.bs_off + ((int64_t)h * Qb + qb) * Kb;
  for (int kb = tid; kb < Kb; kb += BTHR) {
    const float4 *pp = reinterpret_cast<const float4 *>(pq + (int64_t)kb * BR);
    float4 v[BR / 4];
#pragma unroll
    for (int q = 0; q < BR / 4; ++q) v[q] = __ldcs(pp + q);
    // the statistics tile of the block's columns
    const int t = (kb < Kbh ? kb * hw : ch + (kb - Kbh) * BR) / kTileCols;
    float acc = 0.f;
#pragma unroll
    for (int q = 0; q < BR / 4; ++q) {
      const float vv[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = 4 * q + e, a = qb * BR + j;
        // a block starting right of the row's diagonal holds no visible cell
        // (and its partial was never written)
        if (kb < Kbh || (kb - Kbh) * BR <= a)
          acc += vv[e] * __expf(ts_h[(int64_t)a * ntile + t].x - sm[j]) * sil[j];
      }
    }
    out[kb] = acc;
  }
}

}  // namespace

cudaError_t launch_block_sum(const Geo &g, int nctas, const float *bpart, const float2 *tstat,
                             float *block_sums, cudaStream_t st) {
  if (nctas == 0) return cudaSuccess;
  // a programmatic dependent of the kernel before it on the stream (the score
  // GEMM of the same call): its CTAs take SMs as the GEMM's free up
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nctas);
  cfg.blockDim = dim3(BTHR);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (g.Bk / g.S) {
    case 8: return cudaLaunchKernelEx(&cfg, block_sum_kernel<8>, g, bpart, tstat, block_sums);
    case 16: return cudaLaunchKernelEx(&cfg, block_sum_kernel<16>, g, bpart, tstat, block_sums);
    case 32: return cudaLaunchKernelEx(&cfg, block_sum_kernel<32>, g, bpart, tstat, block_sums);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace xattn
