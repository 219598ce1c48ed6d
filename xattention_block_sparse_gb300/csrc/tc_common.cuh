// Blackwell (sm_100a / sm_103a) building blocks written as inline PTX:
// mbarriers with bounded waits, TMA tiled loads into this CTA's shared memory,
// tcgen05 TMEM allocation, MMA issue/commit and TMEM loads/stores, and the
// shared-memory matrix and instruction descriptors of tcgen05.mma.kind::f16.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "common.cuh"

namespace xattn {
namespace tc {

// Budget of every mbarrier wait: kSpinLimit polls, each of which may suspend
// the thread for up to the hardware's time limit (or kSuspendNs when set),
// a few seconds in all.  A wait that runs out records XATTN_ETIMEOUT in the
// device error word and raises the CTA's abort flag, so the kernel unwinds
// instead of hanging.
#ifndef XATTN_SUSPEND_NS
#define XATTN_SUSPEND_NS 0
#endif
constexpr uint32_t kSuspendNs = XATTN_SUSPEND_NS;  // 0: no hint, the system limit applies
constexpr uint32_t kSpinLimit = kSuspendNs ? (1u << 17) : (1u << 24);

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_addr(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  if (kSuspendNs) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(kSuspendNs)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
  }
  return ok != 0;
}
// Non-blocking test for the completion of the phase with the given parity.
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase with the given parity.  Returns false (and sets
// *abort) if the budget ran out or another thread already aborted.  A phase
// that has already completed is seen by the non-blocking test.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                          int32_t *err) {
  if (mbar_test(bar, parity)) return true;
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
  }
  *abort = 1;
  record_error(err, XATTN_ETIMEOUT);
  return false;
}

// ---------------------------------------------------------------------------
// TMA (tensor maps are __grid_constant__ kernel parameters)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *m) {
  asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *m, uint64_t *bar, int c0,
                                            int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *m, uint64_t *bar, int c0,
                                            int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5}], [%6];\n" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_5d(void *dst, const CUtensorMap *m, uint64_t *bar, int c0,
                                            int c1, int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5, %6}], [%7];\n" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
      "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: TMEM allocation, MMA, commit, loads/stores, fences
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                   smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T per the instruction descriptor (kind::f16).
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T: A (M x K, K-major) is read from tensor
// memory, one row per lane, two bf16 per 32-bit column.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// One accumulation of 4 or 8 MMAs (K = 16 each) as one block of PTX, so that
// the issuing thread spends few instructions per MMA: a descriptor advances by
// a 32-bit add on its low word (the start-address field, in 16-byte units:
// shared memory is under 256 KB, so it never carries out), and the accumulate
// predicates are set once.  The first MMA accumulates iff acc0 != 0, the rest
// always.
#define XATTN_GRP_DECL "{\n\t.reg .pred p0, pt;\n\t.reg .b32 al, bl;\n\t.reg .b64 da, db;\n\t"
// S-type: D (+)= A B^T, A and B from shared memory (%1/%2 A lo/hi, %3/%4 B lo/hi)
#define XATTN_SS_FIRST                                                  \
  "setp.ne.b32 p0, %6, 0;\n\tsetp.eq.b32 pt, %6, %6;\n\t"               \
  "mov.b64 da, {%1, %2};\n\tmov.b64 db, {%3, %4};\n\t"                  \
  "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p0;\n\t"
#define XATTN_SS_NEXT(AO, BO)                                           \
  "add.u32 al, %1, " #AO ";\n\tadd.u32 bl, %3, " #BO ";\n\t"            \
  "mov.b64 da, {al, %2};\n\tmov.b64 db, {bl, %4};\n\t"                  \
  "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, pt;\n\t"
#define XATTN_SS_ARGS                                                                \
  "r"(d_tmem), "r"((uint32_t)a_desc), "r"((uint32_t)(a_desc >> 32)),                  \
      "r"((uint32_t)b_desc), "r"((uint32_t)(b_desc >> 32)), "r"(idesc), "r"(acc0)
// P.V-type: D (+)= A B^T, A (P) in tensor memory (%1), B from shared memory
// (%2/%3 lo/hi)
#define XATTN_TS_FIRST                                                  \
  "setp.ne.b32 p0, %5, 0;\n\tsetp.eq.b32 pt, %5, %5;\n\t"               \
  "mov.b64 db, {%2, %3};\n\t"                                           \
  "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p0;\n\t"
#define XATTN_TS_NEXT(AO, BO)                                           \
  "add.u32 al, %1, " #AO ";\n\tadd.u32 bl, %2, " #BO ";\n\t"            \
  "mov.b64 db, {bl, %3};\n\t"                                           \
  "tcgen05.mma.cta_group::1.kind::f16 [%0], [al], db, %4, pt;\n\t"
#define XATTN_TS_ARGS                                                                 \
  "r"(d_tmem), "r"(a_tmem), "r"((uint32_t)b_desc), "r"((uint32_t)(b_desc >> 32)),      \
      "r"(idesc), "r"(acc0)

// S = Q K^T over head_dim 128 (two 64-wide 128B-swizzle halves per operand):
// MMA k at K offset (k / 4) * half + (k % 4) * 32 bytes; half = 128 rows * 128 B
// for A, NK rows * 128 B for B (1024 or 512 in 16-byte units).
__device__ __forceinline__ void mma_ss_d128_nk128(uint32_t d_tmem, uint64_t a_desc,
                                                  uint64_t b_desc, uint32_t idesc,
                                                  uint32_t acc0) {
  asm volatile(XATTN_GRP_DECL XATTN_SS_FIRST XATTN_SS_NEXT(2, 2) XATTN_SS_NEXT(4, 4)
                   XATTN_SS_NEXT(6, 6) XATTN_SS_NEXT(1024, 1024) XATTN_SS_NEXT(1026, 1026)
                       XATTN_SS_NEXT(1028, 1028) XATTN_SS_NEXT(1030, 1030) "}\n" ::XATTN_SS_ARGS
               : "memory");
}
__device__ __forceinline__ void mma_ss_d128_nk64(uint32_t d_tmem, uint64_t a_desc,
                                                 uint64_t b_desc, uint32_t idesc,
                                                 uint32_t acc0) {
  asm volatile(XATTN_GRP_DECL XATTN_SS_FIRST XATTN_SS_NEXT(2, 2) XATTN_SS_NEXT(4, 4)
                   XATTN_SS_NEXT(6, 6) XATTN_SS_NEXT(1024, 512) XATTN_SS_NEXT(1026, 514)
                       XATTN_SS_NEXT(1028, 516) XATTN_SS_NEXT(1030, 518) "}\n" ::XATTN_SS_ARGS
               : "memory");
}
// head_dim 64: one swizzle half, four MMAs
__device__ __forceinline__ void mma_ss_d64(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t acc0) {
  asm volatile(XATTN_GRP_DECL XATTN_SS_FIRST XATTN_SS_NEXT(2, 2) XATTN_SS_NEXT(4, 4)
                   XATTN_SS_NEXT(6, 6) "}\n" ::XATTN_SS_ARGS
               : "memory");
}
// O (+)= P V over NK keys: MMA k reads P columns 8k.. (16 keys) and the V rows
// of keys 16k.. (2048 bytes on: 128 in 16-byte units)
__device__ __forceinline__ void mma_ts_nk128(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t acc0) {
  asm volatile(XATTN_GRP_DECL XATTN_TS_FIRST XATTN_TS_NEXT(8, 128) XATTN_TS_NEXT(16, 256)
                   XATTN_TS_NEXT(24, 384) XATTN_TS_NEXT(32, 512) XATTN_TS_NEXT(40, 640)
                       XATTN_TS_NEXT(48, 768) XATTN_TS_NEXT(56, 896) "}\n" ::XATTN_TS_ARGS
               : "memory");
}
__device__ __forceinline__ void mma_ts_nk64(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t acc0) {
  asm volatile(XATTN_GRP_DECL XATTN_TS_FIRST XATTN_TS_NEXT(8, 128) XATTN_TS_NEXT(16, 256)
                   XATTN_TS_NEXT(24, 384) "}\n" ::XATTN_TS_ARGS
               : "memory");
}

// Arrive once on the mbarrier when every tcgen05 op issued so far by this thread
// has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
          smem_addr(bar))
      : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (warp-collective).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]),
      "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]),
      "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// ---------------------------------------------------------------------------
// Descriptors
// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor, 128-byte swizzle: start address, leading and
// stride byte offsets (16-byte units), version 1, layout type SWIZZLE_128B (2).
// Operand tiles are 1024-byte aligned, so the base offset field stays 0.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor of kind::f16 with bf16 A/B, fp32 accumulator.
// a_mn / b_mn select MN-major (transposed) operands.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4)                      // D format: f32
         | (1u << 7)                    // A format: bf16
         | (1u << 10)                   // B format: bf16
         | ((uint32_t)a_mn << 15)       // A major
         | ((uint32_t)b_mn << 16)       // B major
         | ((uint32_t)(N >> 3) << 17)   // N / 8
         | ((uint32_t)(M >> 4) << 24);  // M / 16
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32 pairs (Blackwell f32x2 arithmetic) and the 3-input max.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unf2(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// ---------------------------------------------------------------------------
// Host: tiled tensor maps (bf16, 128-byte swizzle), encoded through the driver
// entry point so the library does not link libcuda.
// ---------------------------------------------------------------------------
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// dims/box innermost first; strides in bytes for dims 1..rank-1.
inline bool encode_bf16(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims,
                        const cuuint64_t *strides, const cuuint32_t *box) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(base), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc
}  // namespace xattn
