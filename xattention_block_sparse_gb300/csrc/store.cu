// KV store of a prefill chunk ("Task Plan: Layerwise Offload Refactoring",
// Phase 1.2, offload_layer_kv_async): the chunk's keys and values, stored
// head-major [Hkv, tokens, D], are written block by block into the pool pages
// the block table assigns to their positions, [page, row, Hkv, D].
//
// One CTA per (request, chunk block): the block's page is a contiguous
// block_size * Hkv * D run of the pool, written in order with 16-byte stores;
// each 16-byte piece is read from its (KV head, token) row of k_cur / v_cur.
// Memory-bound: every byte is read once and written once.
#include "common.cuh"

namespace xattn {
namespace {

constexpr int kStoreThreads = 256;

__global__ void __launch_bounds__(kStoreThreads)
    store_kv_kernel(const __grid_constant__ Geo g, const uint4 *__restrict__ kc,
                    const uint4 *__restrict__ vc, uint4 *__restrict__ kp, uint4 *__restrict__ vp) {
  const int r = blockIdx.y, j = blockIdx.x;
  const ReqDesc &R = g.req[r];
  if (j >= R.lq / g.Bk) return;
  const int page = page_of(g, r, R.kh / g.Bk + j);  // -1 (and a recorded error) if invalid
  if (page < 0) return;
  const int per_tok = g.Hkv * g.D / 8;     // 16-byte pieces of one pool row
  const int per_page = g.Bk * per_tok;
  const int dq = g.D / 8;                   // pieces per head row
  const int64_t hs = g.kv_hs / 8;           // pieces between heads of k_cur / v_cur
  const int64_t tok0 = (int64_t)R.q0 + (int64_t)j * g.Bk;  // chunk block's first token
  const int64_t dst0 = (int64_t)page * per_page;
  for (int u = threadIdx.x; u < per_page; u += kStoreThreads) {
    const int row = u / per_tok, rem = u - row * per_tok;
    const int kvh = rem / dq, c = rem - kvh * dq;
    const int64_t src = kvh * hs + (tok0 + row) * dq + c;
    const uint4 a = __ldg(kc + src), b = __ldg(vc + src);
    kp[dst0 + u] = a;
    vp[dst0 + u] = b;
  }
}

}  // namespace

cudaError_t launch_store_kv(const Geo &g, int max_blocks, const __nv_bfloat16 *kc,
                            const __nv_bfloat16 *vc, __nv_bfloat16 *kp, __nv_bfloat16 *vp,
                            cudaStream_t st) {
  if (max_blocks == 0) return cudaSuccess;
  store_kv_kernel<<<dim3(max_blocks, g.B), kStoreThreads, 0, st>>>(
      g, reinterpret_cast<const uint4 *>(kc), reinterpret_cast<const uint4 *>(vc),
      reinterpret_cast<uint4 *>(kp), reinterpret_cast<uint4 *>(vp));
  return cudaGetLastError();
}

}  // namespace xattn
