// Block-sum kernel of XAttention BSA estimation ("XAttention BSA Policy 设计文档",
// select_blocks Step 2 softmax_fuse_block_sum; "XAttention Offload Stream
// Synchronization Fix", 技术细节 Stages 2 and 3: merge of the per-tile softmax
// statistics, then normalise and block-sum with the merged statistics).
// The score GEMM that produces the scores and tile statistics is in
// score_gemm.cu.
//
//   merge_stats_kernel  per reshaped row: merges the tile statistics (A2)
//   block_sum_kernel    per (request, head, query block, 256 columns): sums
//                       exp(s-m)/l over the visible cells of every block (A3)
#include "common.cuh"

namespace xattn {
namespace {

// ---------------------------------------------------------------------------
// A2: merge of the per-tile statistics, one warp per reshaped row:
//   m = max_t m_t,  l = sum_t l_t exp(m_t - m)
// over the 128-column tiles that hold visible cells of the row (columns up to
// ch + a).  Rows are numbered request by request, head-major.
// ---------------------------------------------------------------------------
constexpr int MTHR = 256;

__global__ void __launch_bounds__(MTHR) merge_stats_kernel(const __grid_constant__ Geo g,
                                                           int64_t nrows,
                                                           const float2 *__restrict__ tstat,
                                                           float2 *__restrict__ rstat) {
  const int64_t row = ((int64_t)blockIdx.x * MTHR + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= nrows) return;  // whole warps leave together
  // request owning this row: rows of request r start at its rstat offset
  int r = 0;
  for (int i = 1; i < g.B; ++i)
    if (row >= g.req[i].rstat_off) r = i;
  const ReqDesc &R = g.req[r];
  const int S = g.S;
  const int rq = R.lq / S, ch = R.kh / S, ncol = (R.kh + R.lq) / S;
  const int ntiles = (ncol + kTileCols - 1) / kTileCols;
  const int64_t local = row - R.rstat_off;  // h * rq + a
  const int a = (int)(local % rq);
  const float2 *ts = tstat + R.tstat_off + local * ntiles;
  const int nt_a = min(ntiles, (ch + a) / kTileCols + 1);
  float2 tv[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int t = lane + 32 * u;
    tv[u] = t < nt_a ? ts[t] : make_float2(-INFINITY, 0.f);
  }
  float m = fmaxf(fmaxf(tv[0].x, tv[1].x), fmaxf(tv[2].x, tv[3].x));
  for (int t = lane + 128; t < nt_a; t += 32) m = fmaxf(m, ts[t].x);
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float l = 0.f;
#pragma unroll
  for (int u = 0; u < 4; ++u)
    if (tv[u].x > -INFINITY) l += tv[u].y * __expf(tv[u].x - m);
  for (int t = lane + 128; t < nt_a; t += 32) {
    const float2 w = ts[t];
    if (w.x > -INFINITY) l += w.y * __expf(w.x - m);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  if (lane == 0) rstat[row] = make_float2(m, l);
}

// ---------------------------------------------------------------------------
// A3: normalise + block-sum.  One CTA per (request, head, query block, chunk
// of BTHR columns).  Scores are stored [H][Qb][ncol][Br]: a thread owns one
// column and reads its Br rows as Br/4 float4s (issued before anything else);
// the Br columns of a block are Br consecutive lanes, summed with shuffles.
// ---------------------------------------------------------------------------
constexpr int BTHR = 256;

template <int BR>
__global__ void __launch_bounds__(BTHR) block_sum_kernel(const __grid_constant__ Geo g,
                                                         const float *__restrict__ scores,
                                                         const float2 *__restrict__ rstat,
                                                         float *__restrict__ bs) {
  constexpr int QPC = BR / 4;  // float4s per column
  static_assert(BR >= 8 && BR <= 32, "block-sum geometry");
  __shared__ float sm[BR], sil[BR];
  const int cta = blockIdx.x;
  const int r = find_req(g, cta, [](const ReqDesc &d) { return d.bsum0; });
  const ReqDesc &R = g.req[r];
  const int S = g.S;
  const int rq = R.lq / S, ch = R.kh / S, ncol = (R.kh + R.lq) / S;
  const int Qb = R.lq / g.Bk, Kb = ncol / BR;
  const int nchunk = (ncol + BTHR - 1) / BTHR;
  int local = cta - R.bsum0;
  const int cc = local % nchunk;
  local /= nchunk;
  const int qb = local % Qb, h = local / Qb;
  const int tid = threadIdx.x, lane = tid & 31;

  const int b = cc * BTHR + tid;
  // columns past the last row's diagonal are invisible to every row of this block
  const int col_end = min(ncol, ch + qb * BR + BR);
  const float4 *col = reinterpret_cast<const float4 *>(
      scores + R.score_off + ((int64_t)(h * Qb + qb) * ncol + b) * BR);
  float4 v[QPC];
#pragma unroll
  for (int q = 0; q < QPC; ++q) v[q] = b < col_end ? __ldcs(col + q) : make_float4(0.f, 0.f, 0.f, 0.f);
  if (tid < BR) {
    const float2 ml = rstat[R.rstat_off + (int64_t)h * rq + qb * BR + tid];
    sm[tid] = ml.x;
    sil[tid] = 1.f / ml.y;
  }
  __syncthreads();
  float acc = 0.f;
  if (b < col_end) {
#pragma unroll
    for (int q = 0; q < QPC; ++q) {
      const float vv[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = 4 * q + e;
        acc += (b <= ch + qb * BR + j) ? __expf(vv[e] - sm[j]) * sil[j] : 0.f;
      }
    }
  }
  // a block's Br columns are Br consecutive lanes (chunks start at multiples of Br)
#pragma unroll
  for (int o = BR / 2; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((lane % BR) == 0 && b < ncol) bs[R.bs_off + ((int64_t)h * Qb + qb) * Kb + b / BR] = acc;
}

}  // namespace

cudaError_t launch_block_sum(const Geo &g, int nctas, int64_t nrows, const float *scores,
                             const float2 *tstat, float2 *rstat, float *block_sums,
                             cudaStream_t st) {
  if (nrows > 0) {
    const int64_t blocks = (nrows * 32 + MTHR - 1) / MTHR;
    merge_stats_kernel<<<(unsigned)blocks, MTHR, 0, st>>>(g, nrows, tstat, rstat);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (nctas == 0) return cudaSuccess;
  const int br = g.Bk / g.S;
  switch (br) {
    case 8: block_sum_kernel<8><<<nctas, BTHR, 0, st>>>(g, scores, rstat, block_sums); break;
    case 16: block_sum_kernel<16><<<nctas, BTHR, 0, st>>>(g, scores, rstat, block_sums); break;
    case 32: block_sum_kernel<32><<<nctas, BTHR, 0, st>>>(g, scores, rstat, block_sums); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace xattn
