// Selection kernels of XAttention BSA ("XAttention BSA Policy 设计文档",
// select_blocks Step 3 find_blocks_chunked and Step 4 GQA-aware aggregation +
// majority voting).
//
// Per row (request, query head, query block) of Kb block sums: integer masses
// q_j = rne(bs_j * 2^32), visited in (q_j desc, j asc) order; block j is kept
// iff the mass visited before it, prefix_j, is < fl64(tau * T), T = sum q_j.
// The GQA group's "any" over its query heads then votes once per history
// block, and the CTA that finishes last (a counter) runs the vote of every
// request: test votes*den > num*Hkv*Qb ((1, 2): strict majority), sink and
// last history block forced (when asked), ascending compaction, page lookup.
//
//   select_warp_kernel  rows of up to kWarpSortMax blocks: one warp per row.
//                       The row's keys (q << 16 | 0xFFFF - j) sit in the
//                       warp's registers, E = npad/32 per lane; a bitonic
//                       network sorts them in descending order (shuffles
//                       between lanes, register swaps within a lane), a warp
//                       scan gives every position its prefix mass.  A CTA
//                       holds whole GQA groups, so their "any" is a
//                       shared-memory OR.
//   select_kernel       longer rows: one CTA per (request, KV head, query
//                       block), a bitonic sort of each head's row in shared
//                       memory and a block-wide prefix scan.
//   vote_kernel         the vote alone, for a call with no query rows.
//
// Every step is integer or exactly rounded, so the result does not depend on
// the order in which threads add or compare.
#include "common.cuh"

namespace xattn {
namespace {

constexpr int STHR = 512;            // select_kernel threads
constexpr int kWarpSortMax = 1024;   // longest row one warp sorts (32 keys per lane)
constexpr int kWarpRowsMax = 8;      // rows (warps) of one select_warp_kernel CTA
constexpr int kMaxWarps = 32;

__device__ __forceinline__ unsigned long long shfl_xor_u64(unsigned long long v, int m) {
  const unsigned lo = __shfl_xor_sync(0xffffffffu, (unsigned)v, m);
  const unsigned hi = __shfl_xor_sync(0xffffffffu, (unsigned)(v >> 32), m);
  return ((unsigned long long)hi << 32) | lo;
}

__device__ __forceinline__ unsigned long long warp_incl_scan(unsigned long long v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Exclusive block-wide prefix of one value per thread (blockDim.x a multiple
// of 32); *total gets the sum.
__device__ unsigned long long block_excl_scan(unsigned long long v, unsigned long long *wbuf,
                                              unsigned long long *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const unsigned long long incl = warp_incl_scan(v, lane);
  if (lane == 31) wbuf[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    unsigned long long w = lane < nw ? wbuf[lane] : 0ull;
    const unsigned long long wi = warp_incl_scan(w, lane);
    if (lane < nw) wbuf[lane] = wi - w;
    if (lane == nw - 1) wbuf[kMaxWarps] = wi;
  }
  __syncthreads();
  const unsigned long long res = wbuf[warp] + incl - v;
  *total = wbuf[kMaxWarps];
  __syncthreads();
  return res;
}

// The vote of request r by the whole CTA: keep history block j when
// votes_j * den > num * Hkv * Qb, or when forced (sink / last block);
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
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int per = (kbh + nthr - 1) / nthr;
  const int beg = min(tid * per, kbh), end = min(beg + per, kbh);
  const int32_t *cnt = counts + row * g.bt_stride;
  const int32_t *bt = g.block_table + (int64_t)r * g.bt_stride;
  auto keep = [&](int j, int c) {
    return (int64_t)c * vote_den > (int64_t)vote_num * votes_total ||
           (force && (j == 0 || j == kbh - 1));
  };
  // the thread's votes and page ids, loaded together before the scan (up to
  // kVotePer of each held in registers; longer runs read them again)
  constexpr int kVotePer = 4;
  int cv[kVotePer], pv[kVotePer];
#pragma unroll
  for (int e = 0; e < kVotePer; ++e) {
    const int j = beg + e;
    cv[e] = j < end ? __ldcg(cnt + j) : 0;
    pv[e] = j < end ? __ldg(bt + j) : 0;
  }
  unsigned long long mine = 0;
  for (int j = beg; j < end; ++j) {
    const int e = j - beg;
    mine += keep(j, e < kVotePer ? cv[e] : __ldcg(cnt + j)) ? 1 : 0;
  }
  unsigned long long total;
  unsigned long long pos = block_excl_scan(mine, wbuf, &total);
  for (int j = beg; j < end; ++j) {
    const int e = j - beg;
    if (keep(j, e < kVotePer ? cv[e] : __ldcg(cnt + j))) {
      const int64_t o = row * g.bt_stride + (int64_t)pos;
      sel_idx[o] = j;
      int p = e < kVotePer ? pv[e] : __ldg(bt + j);
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

// Counts the launch's finished CTAs; the last one has every vote counted and
// runs the votes of every request.
__device__ void finish_and_vote(const Geo &g, const int32_t *counts, int vote_num, int vote_den,
                                int force, int per_kv, int32_t *sel_idx, int32_t *sel_page,
                                int32_t *n_sel, int32_t *done, unsigned long long *wbuf) {
  __shared__ int last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(done, 1) == (int)gridDim.x - 1;
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

// Compare-exchange of registers e < f of one lane: the larger key to e when
// desc, to f otherwise.
template <int E>
__device__ __forceinline__ void lane_ce(unsigned long long (&x)[E], int e, int f, bool desc) {
  const unsigned long long a = x[e], b = x[f];
  const bool sw = desc ? (a < b) : (a > b);
  x[e] = sw ? b : a;
  x[f] = sw ? a : b;
}

// Bitonic merge of one lane's E keys (strides E/2 .. 1) into one run.
template <int E>
__device__ __forceinline__ void lane_merge(unsigned long long (&x)[E], bool desc) {
#pragma unroll
  for (int ls = 0; (1 << ls) < E; ++ls) {
    const int s = E >> (ls + 1);
#pragma unroll
    for (int e = 0; e < E; ++e)
      if ((e & s) == 0) lane_ce<E>(x, e, e | s, desc);
  }
}

// Descending bitonic sort of the 32*E keys of a warp, E per lane, position
// lane*E + e.  A merge pass of size k orders a run of k positions descending
// when (position & k) == 0, ascending otherwise, so the last pass (k = 32*E)
// leaves the whole warp descending.  Passes up to k = E stay inside a lane;
// a pass of k >= 2E first pairs lanes (shuffles, strides k/2 .. E), then
// merges each lane's registers.  Only the register steps are unrolled: the
// lane passes run as loops, which keeps the code small enough for the
// instruction cache.
template <int E>
__device__ __forceinline__ void warp_sort_desc(unsigned long long (&x)[E], int lane) {
#pragma unroll
  for (int lk = 1; (1 << lk) < E; ++lk) {  // k < E: direction by register index
    const int k = 1 << lk;
#pragma unroll
    for (int ls = lk - 1; ls >= 0; --ls) {
      const int s = 1 << ls;
#pragma unroll
      for (int e = 0; e < E; ++e)
        if ((e & s) == 0) lane_ce<E>(x, e, e | s, (e & k) == 0);
    }
  }
  if (E > 1) lane_merge<E>(x, (lane & 1) == 0);  // k = E: one run per lane
#pragma unroll 1
  for (int k = 2 * E; k <= 32 * E; k <<= 1) {
    const bool desc = ((lane * E) & k) == 0;  // e < E <= k/2 does not reach bit k
#pragma unroll 1
    for (int m = k / (2 * E); m >= 1; m >>= 1) {  // lane distance
      const bool keep_max = ((lane & m) == 0) == desc;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const unsigned long long y = shfl_xor_u64(x[e], m);
        x[e] = ((x[e] > y) == keep_max) ? x[e] : y;
      }
    }
    lane_merge<E>(x, desc);
  }
}

// Threshold selection of one row by one warp: mask bytes (when asked) and the
// history blocks it keeps OR-ed into anyf.
template <int E>
__device__ __forceinline__ void select_row_warp(const float *__restrict__ row, int Kb, int kbh,
                                                double tau, uint8_t *__restrict__ mrow,
                                                uint8_t *anyf, int lane) {
  unsigned long long x[E];
  unsigned long long tsum = 0ull;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    // coalesced loads; the sort does not care where a key starts
    const int j = e * 32 + lane;
    unsigned long long key = 0ull;  // padding: below every real key
    if (j < Kb) {
      const float v = __ldg(row + j);
      // v * 2^32 is exact in fp32; the conversion rounds half to even
      const unsigned long long qv = v > 0.f ? __float2ull_rn(v * 4294967296.0f) : 0ull;
      tsum += qv;
      key = (qv << 16) | (unsigned long long)(0xFFFF - j);
    }
    x[e] = key;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) tsum += shfl_xor_u64(tsum, o);
  warp_sort_desc<E>(x, lane);
  unsigned long long loc = 0ull;
#pragma unroll
  for (int e = 0; e < E; ++e) loc += x[e] >> 16;
  unsigned long long pre = warp_incl_scan(loc, lane) - loc;  // mass before this lane's run
  const double Rth = __dmul_rn(tau, (double)tsum);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const unsigned long long key = x[e], qv = key >> 16;
    if (key != 0ull) {
      const int j = 0xFFFF - (int)(key & 0xFFFFull);
      const bool keep = tau >= 1.0 ? (qv > 0ull) : ((double)pre < Rth);
      if (mrow) mrow[j] = keep ? 1 : 0;
      if (keep && j < kbh) anyf[j] = 1;
    }
    pre += qv;
  }
}

// One CTA per `gpc` consecutive GQA groups (request, KV head, query block),
// one warp per row of a group (warps loop when a group has more rows).
__global__ void __launch_bounds__(kWarpRowsMax * 32, 1) select_warp_kernel(
    const __grid_constant__ Geo g, const float *__restrict__ bs, double tau,
    uint8_t *__restrict__ mask, int32_t *__restrict__ counts, int ngroups, int gpc,
    int flag_stride, int vote_num, int vote_den, int force, int per_kv,
    int32_t *__restrict__ sel_idx, int32_t *__restrict__ sel_page, int32_t *__restrict__ n_sel,
    int32_t *__restrict__ done) {
  extern __shared__ __align__(16) uint8_t anyf_all[];  // [gpc][flag_stride]
  __shared__ unsigned long long wbuf[kMaxWarps + 1];
  __shared__ int64_t s_crow[kWarpRowsMax];
  __shared__ int s_kbh[kWarpRowsMax];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  const int G = g.H / g.Hkv;
  const int g0 = blockIdx.x * gpc;
  const int ng = min(gpc, ngroups - g0);
  for (int i = tid; i < gpc * flag_stride; i += blockDim.x) anyf_all[i] = 0;
  if (tid < ng) {
    const int grp = g0 + tid;
    const int r = find_req(g, grp, [](const ReqDesc &d) { return d.sel0; });
    const ReqDesc &R = g.req[r];
    const int Qb = R.lq / g.Bk, kvh = (grp - R.sel0) / Qb;
    s_crow[tid] = (per_kv ? (int64_t)r * g.Hkv + kvh : (int64_t)r) * g.bt_stride;
    s_kbh[tid] = R.kh / g.Bk;
  }
  __syncthreads();
  for (int rr = warp; rr < ng * G; rr += nw) {
    const int s = rr / G, gi = rr - s * G;
    const int grp = g0 + s;
    const int r = find_req(g, grp, [](const ReqDesc &d) { return d.sel0; });
    const ReqDesc &R = g.req[r];
    const int Qb = R.lq / g.Bk, kbh = R.kh / g.Bk, Kb = kbh + Qb;
    const int local = grp - R.sel0;
    const int qb = local % Qb, kvh = local / Qb;
    const int64_t row_off = R.bs_off + ((int64_t)(kvh * G + gi) * Qb + qb) * Kb;
    const float *row = bs + row_off;
    uint8_t *mrow = mask ? mask + row_off : nullptr;
    uint8_t *anyf = anyf_all + s * flag_stride;
    if (Kb <= 32)
      select_row_warp<1>(row, Kb, kbh, tau, mrow, anyf, lane);
    else if (Kb <= 64)
      select_row_warp<2>(row, Kb, kbh, tau, mrow, anyf, lane);
    else if (Kb <= 128)
      select_row_warp<4>(row, Kb, kbh, tau, mrow, anyf, lane);
    else if (Kb <= 256)
      select_row_warp<8>(row, Kb, kbh, tau, mrow, anyf, lane);
    else if (Kb <= 512)
      select_row_warp<16>(row, Kb, kbh, tau, mrow, anyf, lane);
    else
      select_row_warp<32>(row, Kb, kbh, tau, mrow, anyf, lane);
  }
  __syncthreads();
  // votes: one per (group, history block) kept by any of the group's heads;
  // consecutive groups that share a counter row are added up first
  for (int j = tid; j < flag_stride; j += blockDim.x) {
    int c = 0;
    for (int s = 0; s < ng; ++s) {
      if (j < s_kbh[s]) c += anyf_all[s * flag_stride + j];
      if (s + 1 == ng || s_crow[s + 1] != s_crow[s]) {
        if (c) atomicAdd(counts + s_crow[s] + j, c);
        c = 0;
      }
    }
  }
  finish_and_vote(g, counts, vote_num, vote_den, force, per_kv, sel_idx, sel_page, n_sel, done,
                  wbuf);
}

__global__ void __launch_bounds__(STHR) select_kernel(const __grid_constant__ Geo g,
                                                      const float *__restrict__ bs, double tau,
                                                      uint8_t *__restrict__ mask,
                                                      int32_t *__restrict__ counts,
                                                      int vote_num, int vote_den, int force,
                                                      int per_kv,
                                                      int32_t *__restrict__ sel_idx,
                                                      int32_t *__restrict__ sel_page,
                                                      int32_t *__restrict__ n_sel,
                                                      int32_t *__restrict__ done) {
  extern __shared__ __align__(16) uint8_t sel_smem[];  // any-flags [npad], then keys
  __shared__ unsigned long long wbuf[kMaxWarps + 1];
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
  finish_and_vote(g, counts, vote_num, vote_den, force, per_kv, sel_idx, sel_page, n_sel, done,
                  wbuf);
}

__global__ void __launch_bounds__(STHR) vote_kernel(const __grid_constant__ Geo g,
                                                    const int32_t *__restrict__ counts,
                                                    int vote_num, int vote_den, int force,
                                                    int per_kv,
                                                    int32_t *__restrict__ sel_idx,
                                                    int32_t *__restrict__ sel_page,
                                                    int32_t *__restrict__ n_sel) {
  __shared__ unsigned long long wbuf[kMaxWarps + 1];
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
  // the finishing counter sits right after the vote counters (zeroed with them)
  int32_t *done = counts + (size_t)g.B * (per_kv ? (size_t)g.Hkv : 1) * (size_t)g.bt_stride;
  const int G = g.H / g.Hkv;
  if (max_kb <= kWarpSortMax) {
    // nctas GQA groups; as many whole groups per CTA as fit its warps, fewer
    // when that would leave SMs without a CTA
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return cudaErrorInvalidValue;
    int gpc = G >= kWarpRowsMax ? 1 : kWarpRowsMax / G;
    while (gpc > 1 && (nctas + gpc - 1) / gpc < sms) gpc /= 2;
    const int warps = G * gpc < kWarpRowsMax ? G * gpc : kWarpRowsMax;
    const int flag_stride = (max_kb + 15) & ~15;
    const int grid = (nctas + gpc - 1) / gpc;
    select_warp_kernel<<<grid, warps * 32, (size_t)gpc * flag_stride, st>>>(
        g, block_sums, threshold, mask, counts, nctas, gpc, flag_stride, vote_num, vote_den,
        force_sink_last, per_kv, sel_idx, sel_page, n_sel, done);
    return cudaGetLastError();
  }
  int npad = 1;
  while (npad < max_kb) npad <<= 1;
  const size_t smem = (((size_t)npad + 15) & ~(size_t)15) + (size_t)npad * sizeof(unsigned long long);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  select_kernel<<<nctas, STHR, smem, st>>>(g, block_sums, threshold, mask, counts, vote_num,
                                           vote_den, force_sink_last, per_kv, sel_idx, sel_page,
                                           n_sel, done);
  return cudaGetLastError();
}

}  // namespace xattn
