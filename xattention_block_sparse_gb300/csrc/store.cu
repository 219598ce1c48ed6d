// KV store of a prefill chunk ("Task Plan: Layerwise Offload Refactoring",
// Phase 1.2, offload_layer_kv_async): the chunk's keys and values, strided
// views (KV head, token, d) -- [Hkv, tokens, D] or [tokens, Hkv, D] -- are
// written block by block into the pool pages
// the block table assigns to their positions, [page, row, Hkv, D].
//
// A page is a contiguous block_size * Hkv * D run of the pool, cut into slices
// of kSlice 16-byte pieces, one CTA per (request, chunk block, slice) so the
// copy spreads over every SM; each thread reads its kPer pieces of k_cur and
// v_cur (from their (KV head, token) rows) before it writes any, so its loads
// are in flight together.  Memory-bound: every byte is read once and written
// once.
#include "common.cuh"

namespace xattn {
namespace {

constexpr int kStoreThreads = 256;
constexpr int kPer = 4;                          // pieces per thread and tensor
constexpr int kSlice = kStoreThreads * kPer;     // pieces per CTA and tensor

__global__ void __launch_bounds__(kStoreThreads)
    store_kv_kernel(const __grid_constant__ Geo g, int slices, const uint4 *__restrict__ kc,
                    const uint4 *__restrict__ vc, uint4 *__restrict__ kp, uint4 *__restrict__ vp) {
  const int r = blockIdx.y, j = blockIdx.x / slices, sl = blockIdx.x - j * slices;
  const ReqDesc &R = g.req[r];
  if (j >= R.lq / g.Bk) return;
  const int page = page_of(g, r, R.kh / g.Bk + j);  // -1 (and a recorded error) if invalid
  if (page < 0) return;
  const int per_tok = g.Hkv * g.D / 8;     // 16-byte pieces of one pool row
  const int per_page = g.Bk * per_tok;
  const int dq = g.D / 8;                   // pieces per head row
  const int64_t hs = g.kv_hs / 8;           // pieces between heads of k_cur / v_cur
  const int64_t ts = g.kv_ts / 8;           // pieces between their tokens
  const int64_t tok0 = (int64_t)R.q0 + (int64_t)j * g.Bk;  // chunk block's first token
  const int64_t dst0 = (int64_t)page * per_page;
  const int u0 = sl * kSlice + threadIdx.x;
  uint4 a[kPer], b[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int u = u0 + k * kStoreThreads;
    if (u < per_page) {
      const int row = u / per_tok, rem = u - row * per_tok;
      const int kvh = rem / dq, c = rem - kvh * dq;
      const int64_t src = kvh * hs + (tok0 + row) * ts + c;
      a[k] = __ldg(kc + src);
      b[k] = __ldg(vc + src);
    }
  }
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int u = u0 + k * kStoreThreads;
    if (u < per_page) {
      kp[dst0 + u] = a[k];
      vp[dst0 + u] = b[k];
    }
  }
}

}  // namespace

cudaError_t launch_store_kv(const Geo &g, int max_blocks, const __nv_bfloat16 *kc,
                            const __nv_bfloat16 *vc, __nv_bfloat16 *kp, __nv_bfloat16 *vp,
                            cudaStream_t st) {
  if (max_blocks == 0) return cudaSuccess;
  const int per_page = g.Bk * g.Hkv * g.D / 8;
  const int slices = (per_page + kSlice - 1) / kSlice;
  store_kv_kernel<<<dim3(max_blocks * slices, g.B), kStoreThreads, 0, st>>>(
      g, slices, reinterpret_cast<const uint4 *>(kc), reinterpret_cast<const uint4 *>(vc),
      reinterpret_cast<uint4 *>(kp), reinterpret_cast<uint4 *>(vp));
  return cudaGetLastError();
}

}  // namespace xattn
