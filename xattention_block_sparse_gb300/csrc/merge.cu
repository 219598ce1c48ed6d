// merge_attention_outputs of "XAttention BSA Policy 设计文档"
// (compute_chunked_prefill, steps 1 and 3): two partial attention results over
// disjoint key sets, each normalised with its own log-sum-exp, combined into
// the result over the union.  Memory-bound: one warp per row, float4 accesses.
#include "common.cuh"

namespace xattn {
namespace {

// One warp per row: every lane reads the row's two LSEs before lane 0 writes
// the merged one, so lse_out may alias lse1 or lse2.
__global__ void lse_merge_kernel(const float *__restrict__ o1, const float *__restrict__ l1,
                                 const float *__restrict__ o2, const float *__restrict__ l2,
                                 int64_t rows, int D, void *o_out, int bf16_out,
                                 float *l_out) {
  const int lane = threadIdx.x & 31;
  const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (row >= rows) return;  // whole warps leave together
  const float a = l1[row], b = l2[row];
  const float mx = fmaxf(a, b);
  float w1 = 0.f, w2 = 0.f, lse = -INFINITY;
  if (mx > -INFINITY) {
    const float e1 = __expf(a - mx), e2 = __expf(b - mx);
    const float s = e1 + e2;
    lse = mx + __logf(s);
    w1 = e1 / s;
    w2 = e2 / s;
  }
  __syncwarp();
  for (int c = lane * 4; c < D; c += 128) {
    const float4 x = *reinterpret_cast<const float4 *>(o1 + row * D + c);
    const float4 y = *reinterpret_cast<const float4 *>(o2 + row * D + c);
    const float4 z = make_float4(x.x * w1 + y.x * w2, x.y * w1 + y.y * w2, x.z * w1 + y.z * w2,
                                 x.w * w1 + y.w * w2);
    if (bf16_out) {
      __nv_bfloat162 *p = reinterpret_cast<__nv_bfloat162 *>(
          reinterpret_cast<__nv_bfloat16 *>(o_out) + row * D + c);
      p[0] = __floats2bfloat162_rn(z.x, z.y);
      p[1] = __floats2bfloat162_rn(z.z, z.w);
    } else {
      *reinterpret_cast<float4 *>(reinterpret_cast<float *>(o_out) + row * D + c) = z;
    }
  }
  if (lane == 0) l_out[row] = lse;
}

}  // namespace

cudaError_t launch_lse_merge(const float *o1, const float *l1, const float *o2, const float *l2,
                             int64_t rows, int D, void *o_out, int bf16_out, float *l_out,
                             cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const int thr = 256;  // 8 rows per block
  const int64_t blocks = (rows * 32 + thr - 1) / thr;
  lse_merge_kernel<<<(unsigned)blocks, thr, 0, st>>>(o1, l1, o2, l2, rows, D, o_out, bf16_out,
                                                     l_out);
  return cudaGetLastError();
}

}  // namespace xattn
