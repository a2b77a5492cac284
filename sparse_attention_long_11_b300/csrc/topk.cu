// Exact per-query top-k selection (DeepSeek-V3.2 summary card, "How DSA
// Works": keep only the 2048 most relevant tokens per query; news article on
// DeepSeek-V3.2: the fine-grained selector keeps the top-k key/value
// positions of every query).
//
// One block per query row.  Scores become order-preserving 32-bit keys (-0
// folded onto +0).
//
//   1. A threshold guess G: of 1024 evenly spaced samples of the row, the
//      r-th largest (its 22 leading bits: two radix rounds), r a few standard
//      deviations above the expected rank of the k-th largest key (1024 k / n).
//   2. One pass over the row collects every key >= G with its position into
//      a per-warp list (warp w owns a contiguous segment, so the lists hold
//      positions in ascending order).  With at least k of them, the row's
//      top k are all among them.
//   3. Three radix rounds (11 + 11 + 10 bits) over the collected keys find
//      the exact key T of the k-th largest and how many keys equal to T are
//      still needed; the output is every collected key above T and the
//      lowest-positioned `need` keys equal to T, in ascending position: ties
//      resolve to the lower position and the selected set is unique.
//
// When the guess misses (fewer than k collected, or a list overflows) the
// block falls back to the same radix rounds over the whole row, followed by
// an ordered compaction of the whole row.  Rows are read with 16-byte loads
// straight from global memory (inside the fused forward the indexer has just
// written them).  Blocks of 512 threads let four rows share an SM; batches
// with few rows, rows longer than 65536 keys, or lists too large for several
// blocks an SM use 1024-thread blocks instead.  The list is sized at launch from k and the
// longest row, and a row whose expected candidates would nearly fill it goes
// straight to the exact rounds.
#include <algorithm>
#include <cmath>

#include "launch.h"
#include "topk_core.cuh"

namespace dsa {
namespace {

using namespace topk_core;

template <int NT>
__global__ void __launch_bounds__(NT, NT == kManyRowsThreads ? 2048 / NT : 1)
topk_kernel(QueryBatch qb, const float* __restrict__ scores, int64_t ld, int k, int32_t* __restrict__ idx,
            int R, int* err) {
  constexpr int NW = NT / 32;
  extern __shared__ __align__(16) uint32_t dsm[];   // [NW * R] candidate keys, then [NW * R] positions (R per warp)
  uint32_t* ckey = dsm;
  uint32_t* cpos = dsm + NW * R;
  __shared__ uint32_t hist[kBins];
  __shared__ uint32_t samp[kSamples];
  __shared__ uint32_t warp_tot[32];
  __shared__ TopkShared<NT> S;

  const int i = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int32_t* out = idx + (int64_t)i * k;
  const int pos = __ldg(qb.q_pos + i);
  if (pos < 0 || pos >= qb.max_kv) {
    if (tid == 0) flag_error(err, DSA_ERR_BOUNDS);
    for (int j = tid; j < k; j += NT) out[j] = -1;
    return;
  }
  const int n = pos + 1;
  if (n <= k) {
    for (int j = tid; j < k; j += NT) out[j] = j < n ? j : -1;
    return;
  }
  const float* row = scores + (int64_t)i * ld;
  const RowKeys rk{row, n, (reinterpret_cast<uintptr_t>(row) & 15) == 0};

  // ---- 1. a threshold guess from evenly spaced samples: the r-th largest
  // sample, r a safe margin above the expected rank of the k-th largest key.
  // When the r n / 1024 keys expected above it would nearly fill the list,
  // the guess would overflow it: take the exact rounds over the row at once.
  const float f = (float)kSamples * (float)k / (float)n;
  const int r = min(kSamples, (int)ceilf(f + 3.f * sqrtf(f) + 8.f));
  if (8 * (int64_t)r * n > 7 * (int64_t)kSamples * NW * R) {   // block-uniform
    radix_path<NT>(rk, k, out, err, hist, dsm, warp_tot, S);
    return;
  }
  for (int s = tid; s < kSamples; s += NT) samp[s] = score_key(__ldg(row + (int)(((int64_t)s * n) / kSamples)));
  if (tid == 0) {
    S.overflow = 0;
    S.sel_bin = 0;   // always overwritten by a consistent select; never left undefined
    S.sel_above = 0;
  }
  __syncthreads();
  uint32_t unused;
  const uint32_t G = select_in_list<NT>(kSamples, [&](int s, uint32_t& u) { u = samp[s]; return true; }, (uint32_t)r,
                                        hist, warp_tot, S, &unused, 2);

  // ---- 2. one pass over the row: every key >= G with its position, into
  // the warp's region of the list, in position order (warp w scans the
  // contiguous segment [w*seg, (w+1)*seg); seg a multiple of 128, four
  // candidates per lane and step, four steps' loads in flight)
  const int seg = ((n + NW - 1) / NW + 127) & ~127;
  const int beg = warp * seg, end = min(n, beg + seg);
  uint32_t cnt = 0;
#pragma unroll 1
  for (int j0 = beg; j0 < end; j0 += 512) {   // warp-uniform bound
    uint4 v[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int j = j0 + 128 * t + 4 * lane;
      v[t] = j < end ? rk.load4(j) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int j = j0 + 128 * t + 4 * lane;
      const uint32_t u[4] = {v[t].x, v[t].y, v[t].z, v[t].w};
      uint32_t m = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (j + e < end && u[e] >= G) m |= 1u << e;
      uint32_t tot;
      uint32_t slot = cnt + warp_excl_scan(__popc(m), &tot);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (m & (1u << e)) {
          if (slot < (uint32_t)R) {
            ckey[warp * R + slot] = u[e];
            cpos[warp * R + slot] = (uint32_t)(j + e);
          }
          ++slot;
        }
      cnt += tot;
    }
  }
  if (lane == 0) {
    S.w_cnt[warp] = cnt;
    if (cnt > (uint32_t)R) S.overflow = 1;
  }
  __syncthreads();
  uint32_t total = 0;
#pragma unroll 1
  for (int w = 0; w < NW; ++w) total += S.w_cnt[w];
  if (S.overflow || total < (uint32_t)k) {   // the guess missed (block-uniform): exact radix rounds over the row
    radix_path<NT>(rk, k, out, err, hist, ckey, warp_tot, S);
    return;
  }

  // ---- 3. the exact k-th largest key among the candidates (all keys >= G,
  // at least k of them, so the row's top k are among them)
  uint32_t need;
  // c / R as a multiply-high: exact, since c < 2^16 and the reciprocal's error
  // stays far below 1/R
  const uint32_t inv_r = (uint32_t)(0xffffffffull / (uint32_t)R) + 1u;
  const uint32_t T = select_in_list<NT>(
      NW * R,
      [&](int c, uint32_t& u) {
        const int w = (int)__umulhi((uint32_t)c, inv_r);
        if ((uint32_t)(c - w * R) >= S.w_cnt[w]) return false;
        u = ckey[c];
        return true;
      },
      (uint32_t)k, hist, warp_tot, S, &need);

  // ---- 4. ordered output: warp w walks its region (positions ascending)
  uint32_t gt = 0, eq = 0;
  for (uint32_t c = lane; c < cnt; c += 32) {
    const uint32_t u = ckey[warp * R + c];
    gt += u > T;
    eq += u == T;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    gt += __shfl_xor_sync(0xffffffffu, gt, o);
    eq += __shfl_xor_sync(0xffffffffu, eq, o);
  }
  if (lane == 0) {
    S.w_gt[warp] = gt;
    S.w_eq[warp] = eq;
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t e_w = lane < NW ? S.w_eq[lane] : 0u, g_w = lane < NW ? S.w_gt[lane] : 0u;
    uint32_t e_tot;
    const uint32_t e_ex = warp_excl_scan(e_w, &e_tot);
    const uint32_t take = need > e_ex ? min(need - e_ex, e_w) : 0u;
    uint32_t s_tot;
    const uint32_t s_ex = warp_excl_scan(g_w + take, &s_tot);
    if (lane < NW) {
      S.w_selbase[lane] = s_ex;
      S.w_eqbase[lane] = e_ex;
    }
  }
  __syncthreads();
  uint32_t eq_run = S.w_eqbase[warp], sel_run = S.w_selbase[warp];
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (uint32_t c0 = 0; c0 < cnt; c0 += 32) {   // warp-uniform bound
    const uint32_t c = c0 + lane;
    uint32_t u = 0;
    if (c < cnt) u = ckey[warp * R + c];
    const bool is_eq = c < cnt && u == T;
    const uint32_t eqb = __ballot_sync(0xffffffffu, is_eq);
    const bool take = (c < cnt && u > T) || (is_eq && eq_run + __popc(eqb & lt_mask) < need);
    const uint32_t selb = __ballot_sync(0xffffffffu, take);
    if (take) {
      const uint32_t slot = sel_run + __popc(selb & lt_mask);
      if (slot < (uint32_t)k) out[slot] = (int32_t)cpos[warp * R + c];
      else flag_error(err, DSA_ERR_BOUNDS);   // cannot happen for a consistent select; never write past the row
    }
    eq_run += __popc(eqb);
    sel_run += __popc(selb);
  }
}

int sm_count_topk() {
  static int cache[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (!cache[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 148;
  }
  return cache[dev];
}

// Per-warp list capacity for rows of up to max_kv keys: 4/3 of the keys
// expected above the sampled guess in the longest row, spread over the warps,
// rounded up to 32; at least the default and at most kMaxListBytes in all.
int list_per_warp(int nt, int k, int max_kv) {
  const int nw = nt / 32;
  const double n = (double)std::max(max_kv, 1);
  const double f = (double)kSamples * k / n;
  const double r = std::min((double)kSamples, std::ceil(f + 3.0 * std::sqrt(f) + 8.0));
  const double expect = std::min(n, r * n / kSamples);
  int per = (int)std::ceil(expect * 4.0 / 3.0 / nw);
  per = (per + 31) & ~31;
  const int lo = nt == kManyRowsThreads ? Region<kManyRowsThreads>::kPerWarp : Region<kFewRowsThreads>::kPerWarp;
  const int hi = kMaxListBytes / (8 * nw);
  return std::max(lo, std::min(per, hi));
}

template <int NT>
cudaError_t launch_topk_nt(const QueryBatch& qb, const float* scores, int64_t ld, int k, int32_t* idx, int per,
                           int* err, cudaStream_t stream) {
  const int smem = 2 * (NT / 32) * per * (int)sizeof(uint32_t);
  cudaError_t e = cudaFuncSetAttribute(topk_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  topk_kernel<NT><<<qb.num_q, NT, smem, stream>>>(qb, scores, ld, k, idx, per, err);
  return cudaGetLastError();
}

}  // namespace

// Many rows of at most kLongRow keys: 512-thread blocks, four per SM, while
// the list stays within 100 KiB; otherwise (few rows, long rows, or a list
// that would leave one narrow block per SM) 1024-thread blocks, whose 32
// warps keep more loads in flight for each row.
cudaError_t launch_topk(const QueryBatch& qb, const float* scores, int64_t ld, int k, int32_t* idx,
                        int* err, cudaStream_t stream) {
  if (qb.num_q >= 2 * sm_count_topk() && qb.max_kv <= kLongRow) {
    const int per = list_per_warp(kManyRowsThreads, k, qb.max_kv);
    if (8 * (kManyRowsThreads / 32) * per <= (100 << 10))
      return launch_topk_nt<kManyRowsThreads>(qb, scores, ld, k, idx, per, err, stream);
  }
  return launch_topk_nt<kFewRowsThreads>(qb, scores, ld, k, idx, list_per_warp(kFewRowsThreads, k, qb.max_kv), err,
                                         stream);
}

}  // namespace dsa
