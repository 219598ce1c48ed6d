// Selection kernels of XAttention BSA ("XAttention BSA Policy 设计文档",
// select_blocks Step 3 find_blocks_chunked and Step 4 GQA-aware aggregation +
// majority voting).
//
//   select_kernel  one CTA per (request, KV head, query block).  For each query
//                  head of the group: integer masses q_j = rne(bs_j * 2^32),
//                  visited in (q_j desc, j asc) order; block j is kept iff the
//                  mass visited before it, prefix_j, is < fl64(tau * T).  Rows
//                  of up to kRankMax blocks get prefix_j directly as the sum of
//                  the masses whose key (q, -index) exceeds j's -- all the
//                  group's rows at once, no barrier in the loop; longer rows
//                  go through a bitonic sort and a prefix scan.  The group's
//                  "any" over its heads then votes once per history block.
//                  The CTA that finishes last (a counter) runs the vote of every
//                  request: test votes*den > num*Hkv*Qb ((1, 2): strict
//                  majority), sink and last history block forced (when asked),
//                  ascending compaction, page lookup.
//   vote_kernel    the same vote alone, for a call with no query rows.
//
// Every step is integer or exactly rounded, so the result does not depend on
// the order in which threads add or compare.
#include "common.cuh"

namespace xattn {
namespace {

constexpr int STHR = 512;
constexpr int SWARPS = STHR / 32;
constexpr int kRankMax = 512;    // longest row ranked directly (Kb^2 compare-adds per row)
constexpr int kRankKeys = 4096;  // keys of all G rows held at once
constexpr int kRankMaxG = 64;    // largest GQA group taking the direct path

__device__ __forceinline__ unsigned long long warp_incl_scan(unsigned long long v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Exclusive block-wide prefix of one value per thread; *total gets the sum.
__device__ unsigned long long block_excl_scan(unsigned long long v, unsigned long long *wbuf,
                                              unsigned long long *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned long long incl = warp_incl_scan(v, lane);
  if (lane == 31) wbuf[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    unsigned long long w = lane < SWARPS ? wbuf[lane] : 0ull;
    const unsigned long long wi = warp_incl_scan(w, lane);
    if (lane < SWARPS) wbuf[lane] = wi - w;
    if (lane == SWARPS - 1) wbuf[SWARPS] = wi;
  }
  __syncthreads();
  const unsigned long long res = wbuf[warp] + incl - v;
  *total = wbuf[SWARPS];
  __syncthreads();
  return res;
}

// The vote of request r by the whole CTA (STHR threads): keep history block j
// when votes_j * den > num * Hkv * Qb, or when forced (sink / last block);
// ascending compaction into sel_idx, page lookup into sel_page, count in n_sel.
// kvh >= 0: the vote of that KV head alone (its votes over its Qb query
// blocks, out of Qb), in row r * Hkv + kvh of the counters and outputs.
__device__ void vote_request(const Geo &g, int r, int kvh, const int32_t *counts, int vote_num,
                             int vote_den, int force, int32_t *sel_idx, int32_t *sel_page,
                             int32_t *n_sel, unsigned long long *wbuf) {
  const ReqDesc &R = g.req[r];
  const int kbh = R.kh / g.Bk, Qb = R.lq / g.Bk;
  const int64_t votes_total = kvh < 0 ? (int64_t)g.Hkv * Qb : (int64_t)Qb;
  const int64_t row = kvh < 0 ? r : (int64_t)r * g.Hkv + kvh;
  const int tid = threadIdx.x;
  const int per = (kbh + STHR - 1) / STHR;
  const int beg = min(tid * per, kbh), end = min(beg + per, kbh);
  const int32_t *cnt = counts + row * g.bt_stride;
  auto keep = [&](int j) {
    return (int64_t)__ldcg(cnt + j) * vote_den > (int64_t)vote_num * votes_total ||
           (force && (j == 0 || j == kbh - 1));
  };
  unsigned long long mine = 0;
  for (int j = beg; j < end; ++j) mine += keep(j) ? 1 : 0;
  unsigned long long total;
  unsigned long long pos = block_excl_scan(mine, wbuf, &total);
  for (int j = beg; j < end; ++j) {
    if (keep(j)) {
      const int64_t o = row * g.bt_stride + (int64_t)pos;
      sel_idx[o] = j;
      int p = g.block_table[(int64_t)r * g.bt_stride + j];
      if (p < 0 || p >= g.num_pages) {
        record_error(g.err, XATTN_EPAGE);
        p = -1;
      }
      sel_page[o] = p;
      ++pos;
    }
  }
  if (tid == 0) n_sel[row] = (int32_t)total;
}

__global__ void __launch_bounds__(STHR) select_kernel(const __grid_constant__ Geo g,
                                                      const float *__restrict__ bs, double tau,
                                                      uint8_t *__restrict__ mask,
                                                      int32_t *__restrict__ counts, int nkeys,
                                                      int vote_num, int vote_den, int force,
                                                      int per_kv,
                                                      int32_t *__restrict__ sel_idx,
                                                      int32_t *__restrict__ sel_page,
                                                      int32_t *__restrict__ n_sel,
                                                      int32_t *__restrict__ done) {
  extern __shared__ __align__(16) uint8_t sel_smem[];  // any-flags [npad], then keys
  __shared__ unsigned long long wbuf[SWARPS + 1];
  const int cta = blockIdx.x;
  const int r = find_req(g, cta, [](const ReqDesc &d) { return d.sel0; });
  const ReqDesc &R = g.req[r];
  const int Qb = R.lq / g.Bk, kbh = R.kh / g.Bk, Kb = kbh + Qb;
  const int local = cta - R.sel0;
  const int qb = local % Qb, kvh = local / Qb;
  const int G = g.H / g.Hkv;
  int npad = 1;
  while (npad < Kb) npad <<= 1;
  uint8_t *anyf = sel_smem;
  unsigned long long *keys = reinterpret_cast<unsigned long long *>(sel_smem + ((npad + 15) & ~15));
  const int tid = threadIdx.x;

  for (int j = tid; j < kbh; j += STHR) anyf[j] = 0;

  // (the keys of G rows must fit the shared memory the launch sized: nkeys)
  if (Kb <= kRankMax && G * Kb <= kRankKeys && G <= kRankMaxG && G * Kb <= nkeys) {
    // direct ranks: keys of every head of the group in shared memory
    unsigned long long *gk = keys;  // [G][Kb]
    __shared__ unsigned long long tot[kRankMaxG];
    for (int idx = tid; idx < G * Kb; idx += STHR) {
      const int gi = idx / Kb, j = idx - gi * Kb;
      const float v = bs[R.bs_off + ((int64_t)(kvh * G + gi) * Qb + qb) * Kb + j];
      // v * 2^32 is exact in fp32; the conversion rounds half to even
      const unsigned long long qv = v > 0.f ? __float2ull_rn(v * 4294967296.0f) : 0ull;
      gk[idx] = (qv << 16) | (unsigned long long)(0xFFFF - j);
    }
    __syncthreads();
    // row totals T, one warp per row
    for (int gi = tid >> 5; gi < G; gi += SWARPS) {
      unsigned long long t = 0ull;
      for (int j = tid & 31; j < Kb; j += 32) t += gk[gi * Kb + j] >> 16;
#pragma unroll
      for (int o = 16; o; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
      if ((tid & 31) == 0) tot[gi] = t;
    }
    __syncthreads();
    for (int idx = tid; idx < G * Kb; idx += STHR) {
      const int gi = idx / Kb, j = idx - gi * Kb;
      const unsigned long long *row = gk + gi * Kb;
      const unsigned long long kj = row[j];
      // four independent partial sums over the row (shared-memory broadcasts)
      unsigned long long p4[4] = {0ull, 0ull, 0ull, 0ull};
      int i = 0;
      for (; i + 4 <= Kb; i += 4) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const unsigned long long ki = row[i + u];
          p4[u] += ki > kj ? (ki >> 16) : 0ull;
        }
      }
      for (; i < Kb; ++i) {
        const unsigned long long ki = row[i];
        p4[0] += ki > kj ? (ki >> 16) : 0ull;
      }
      const unsigned long long pre = (p4[0] + p4[1]) + (p4[2] + p4[3]);
      const unsigned long long qv = kj >> 16;
      const bool keep =
          tau >= 1.0 ? (qv > 0ull) : ((double)pre < __dmul_rn(tau, (double)tot[gi]));
      const int64_t row_off = R.bs_off + ((int64_t)(kvh * G + gi) * Qb + qb) * Kb;
      if (mask) mask[row_off + j] = keep ? 1 : 0;
      if (keep && j < kbh) anyf[j] = 1;
    }
    __syncthreads();
  } else
  for (int gi = 0; gi < G; ++gi) {
    const int h = kvh * G + gi;
    const int64_t row_off = R.bs_off + ((int64_t)h * Qb + qb) * Kb;
    const float *row = bs + row_off;
    unsigned long long tsum = 0;
    for (int j = tid; j < npad; j += STHR) {
      unsigned long long key = 0ull;
      if (j < Kb) {
        const float v = row[j];
        // v * 2^32 is exact in fp32; the conversion rounds half to even
        const unsigned long long qv = v > 0.f ? __float2ull_rn(v * 4294967296.0f) : 0ull;
        tsum += qv;
        key = (qv << 16) | (unsigned long long)(0xFFFF - j);
      }
      keys[j] = key;
    }
    unsigned long long T;
    block_excl_scan(tsum, wbuf, &T);  // also orders the key writes before the sort

    // bitonic sort, descending
    for (int k = 2; k <= npad; k <<= 1) {
      for (int jj = k >> 1; jj > 0; jj >>= 1) {
        for (int i = tid; i < npad; i += STHR) {
          const int ixj = i ^ jj;
          if (ixj > i) {
            const unsigned long long x = keys[i], y = keys[ixj];
            const bool desc = (i & k) == 0;
            if (desc ? (x < y) : (x > y)) {
              keys[i] = y;
              keys[ixj] = x;
            }
          }
        }
        __syncthreads();
      }
    }

    // exclusive prefix of the sorted masses; each thread owns a contiguous run
    const int per = (npad + STHR - 1) / STHR;
    const int beg = min(tid * per, npad), end = min(beg + per, npad);
    unsigned long long run = 0;
    for (int i = beg; i < end; ++i) run += keys[i] >> 16;
    unsigned long long tot;
    unsigned long long pre = block_excl_scan(run, wbuf, &tot);
    const double Rth = __dmul_rn(tau, (double)T);
    for (int i = beg; i < end; ++i) {
      const unsigned long long key = keys[i];
      const unsigned long long qv = key >> 16;
      const int idx = 0xFFFF - (int)(key & 0xFFFFull);
      if (idx < Kb) {
        const bool keep = tau >= 1.0 ? (qv > 0ull) : ((double)pre < Rth);
        if (mask) mask[row_off + idx] = keep ? 1 : 0;
        if (keep && idx < kbh) anyf[idx] = 1;
      }
      pre += qv;
    }
    __syncthreads();
  }
  // votes: per request (over its KV heads), or per (request, KV head)
  int32_t *crow = counts + (per_kv ? (int64_t)r * g.Hkv + kvh : (int64_t)r) * g.bt_stride;
  for (int j = tid; j < kbh; j += STHR)
    if (anyf[j]) atomicAdd(crow + j, 1);

  // the CTA that finishes last has every vote counted: it runs the votes
  __shared__ int last;
  __threadfence();
  __syncthreads();
  if (tid == 0) last = atomicAdd(done, 1) == (int)gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (int rr = 0; rr < g.B; ++rr) {
    if (per_kv) {
      for (int k = 0; k < g.Hkv; ++k)
        vote_request(g, rr, k, counts, vote_num, vote_den, force, sel_idx, sel_page, n_sel, wbuf);
    } else {
      vote_request(g, rr, -1, counts, vote_num, vote_den, force, sel_idx, sel_page, n_sel, wbuf);
    }
  }
}

__global__ void __launch_bounds__(STHR) vote_kernel(const __grid_constant__ Geo g,
                                                    const int32_t *__restrict__ counts,
                                                    int vote_num, int vote_den, int force,
                                                    int per_kv,
                                                    int32_t *__restrict__ sel_idx,
                                                    int32_t *__restrict__ sel_page,
                                                    int32_t *__restrict__ n_sel) {
  __shared__ unsigned long long wbuf[SWARPS + 1];
  const int r = per_kv ? blockIdx.x / g.Hkv : blockIdx.x;
  vote_request(g, r, per_kv ? (int)(blockIdx.x % g.Hkv) : -1, counts, vote_num, vote_den, force,
               sel_idx, sel_page, n_sel, wbuf);
}

}  // namespace

cudaError_t launch_select(const Geo &g, int nctas, int max_kb, const float *block_sums,
                          double threshold, uint8_t *mask, int32_t *counts, int vote_num,
                          int vote_den, int force_sink_last, int per_kv, int32_t *sel_idx,
                          int32_t *sel_page, int32_t *n_sel, cudaStream_t st) {
  if (nctas == 0) {  // no query rows: the vote alone (every count is zero)
    vote_kernel<<<per_kv ? g.B * g.Hkv : g.B, STHR, 0, st>>>(
        g, counts, vote_num, vote_den, force_sink_last, per_kv, sel_idx, sel_page, n_sel);
    return cudaGetLastError();
  }
  int npad = 1;
  while (npad < max_kb) npad <<= 1;
  const int G = g.H / g.Hkv;
  // keys: the sort's npad, or the direct ranks' G rows (see select_kernel)
  size_t nkeys = (size_t)npad;
  if (max_kb <= kRankMax && G * max_kb <= kRankKeys && G <= kRankMaxG && (size_t)G * max_kb > nkeys)
    nkeys = (size_t)G * max_kb;
  const size_t smem = (((size_t)npad + 15) & ~(size_t)15) + nkeys * sizeof(unsigned long long);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  // the finishing counter sits right after the vote counters (zeroed with them)
  int32_t *done = counts + (size_t)g.B * (per_kv ? (size_t)g.Hkv : 1) * (size_t)g.bt_stride;
  select_kernel<<<nctas, STHR, smem, st>>>(g, block_sums, threshold, mask, counts, (int)nkeys,
                                           vote_num, vote_den, force_sink_last, per_kv, sel_idx,
                                           sel_page, n_sel, done);
  return cudaGetLastError();
}

}  // namespace xattn
