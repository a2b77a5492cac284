// Exact per-query top-k selection (DeepSeek-V3.2 summary card, "How DSA
// Works": keep only the 2048 most relevant tokens per query; news article on
// DeepSeek-V3.2: the fine-grained selector keeps the top-k key/value
// positions of every query).
//
// One 1024-thread block per query row.  Scores become order-preserving
// 32-bit keys (-0 folded onto +0).  A three-round radix select (11 + 11 + 10
// bits, shared-memory histograms) finds the exact key T of the k-th largest
// candidate and how many candidates equal to T are still needed.  An ordered
// compaction then writes, in ascending position, every candidate above T and
// the lowest-positioned `need` candidates equal to T: ties resolve to the
// lower position and the selected set is unique.  Rows of up to
// kCacheCap candidates keep their keys in shared memory; longer rows are
// re-read from global memory on every round.
#include "launch.h"

namespace dsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;
constexpr int kCacheCap = 40960;   // keys cached in shared memory (160 KiB)

__device__ __forceinline__ uint32_t block_incl_scan(uint32_t v, uint32_t* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t t = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t u = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += u;
    }
    warp_tot[lane] = t;   // inclusive over warps
  }
  __syncthreads();
  uint32_t r = v + (warp > 0 ? warp_tot[warp - 1] : 0u);
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kThreads, 1)
topk_kernel(QueryBatch qb, const float* __restrict__ scores, int64_t ld, int k,
            int32_t* __restrict__ idx, int cache_cap, int* err) {
  extern __shared__ uint32_t skey[];           // [cache_cap]
  __shared__ uint32_t hist[kBins];
  __shared__ uint32_t warp_tot[32];
  __shared__ uint32_t sel_bin, sel_above;
  __shared__ uint32_t w_gt[kWarps], w_eq[kWarps], w_selbase[kWarps], w_eqbase[kWarps];

  const int i = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int32_t* out = idx + (int64_t)i * k;
  const int pos = __ldg(qb.q_pos + i);
  if (pos < 0 || pos >= qb.max_kv) {
    if (tid == 0) flag_error(err, DSA_ERR_BOUNDS);
    for (int j = tid; j < k; j += kThreads) out[j] = -1;
    return;
  }
  const int n = pos + 1;
  if (n <= k) {
    for (int j = tid; j < k; j += kThreads) out[j] = j < n ? j : -1;
    return;
  }
  const float* row = scores + (int64_t)i * ld;
  const bool cached = n <= cache_cap;

  uint32_t prefix = 0, pmask = 0;
  uint32_t krem = (uint32_t)k;
#pragma unroll 1
  for (int round = 0; round < 3; ++round) {
    const int shift = round == 0 ? 21 : (round == 1 ? 10 : 0);
    const int nb = round == 2 ? 1024 : 2048;
    for (int b = tid; b < kBins; b += kThreads) hist[b] = 0;
    __syncthreads();
    for (int j = tid; j < n; j += kThreads) {
      uint32_t u;
      if (round == 0) {
        u = score_key(__ldg(row + j));
        if (cached) skey[j] = u;
      } else {
        u = cached ? skey[j] : score_key(__ldg(row + j));
      }
      if ((u & pmask) == prefix) atomicAdd(&hist[(u >> shift) & (nb - 1)], 1u);
    }
    __syncthreads();
    // thread t owns the bins of descending rank 2t and 2t+1
    const int b0 = nb - 1 - 2 * tid, b1 = b0 - 1;
    const uint32_t h0 = b0 >= 0 ? hist[b0] : 0u, h1 = b1 >= 0 ? hist[b1] : 0u;
    const uint32_t incl = block_incl_scan(h0 + h1, warp_tot);
    const uint32_t excl = incl - h0 - h1;
    if (excl < krem && krem <= excl + h0) {
      sel_bin = (uint32_t)b0;
      sel_above = excl;
    } else if (excl + h0 < krem && krem <= incl) {
      sel_bin = (uint32_t)b1;
      sel_above = excl + h0;
    }
    __syncthreads();
    prefix |= sel_bin << shift;
    pmask |= (uint32_t)(nb - 1) << shift;
    krem -= sel_above;
    __syncthreads();
  }
  const uint32_t T = prefix;   // key of the k-th largest candidate
  const uint32_t need = krem;  // candidates equal to T to take (>= 1)

  // ordered compaction: warp w owns the contiguous segment [w*seg, (w+1)*seg)
  const int seg = ((n + kWarps - 1) / kWarps + 31) & ~31;
  const int beg = warp * seg, end = min(n, beg + seg);
  uint32_t gt = 0, eq = 0;
  for (int j = beg + lane; j < end; j += 32) {
    uint32_t u = cached ? skey[j] : score_key(__ldg(row + j));
    gt += u > T;
    eq += u == T;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    gt += __shfl_xor_sync(0xffffffffu, gt, o);
    eq += __shfl_xor_sync(0xffffffffu, eq, o);
  }
  if (lane == 0) { w_gt[warp] = gt; w_eq[warp] = eq; }
  __syncthreads();
  if (tid == 0) {
    uint32_t eb = 0, sb = 0;
    for (int w = 0; w < kWarps; ++w) {
      w_eqbase[w] = eb;
      w_selbase[w] = sb;
      uint32_t take = need > eb ? min(need - eb, w_eq[w]) : 0u;
      sb += w_gt[w] + take;
      eb += w_eq[w];
    }
  }
  __syncthreads();
  uint32_t eq_run = w_eqbase[warp], sel_run = w_selbase[warp];
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int j0 = beg; j0 < end; j0 += 32) {
    const int j = j0 + lane;
    uint32_t u = 0;
    if (j < end) u = cached ? skey[j] : score_key(__ldg(row + j));
    const bool is_eq = j < end && u == T;
    const uint32_t eqb = __ballot_sync(0xffffffffu, is_eq);
    const bool take = (j < end && u > T) || (is_eq && eq_run + __popc(eqb & lt_mask) < need);
    const uint32_t selb = __ballot_sync(0xffffffffu, take);
    if (take) {
      const uint32_t slot = sel_run + __popc(selb & lt_mask);
      if (slot < (uint32_t)k) out[slot] = j;
      else flag_error(err, DSA_ERR_BOUNDS);   // cannot happen for a consistent select; never write past the row
    }
    eq_run += __popc(eqb);
    sel_run += __popc(selb);
  }
}

}  // namespace

cudaError_t launch_topk(const QueryBatch& qb, const float* scores, int64_t ld, int k, int32_t* idx,
                        int* err, cudaStream_t stream) {
  int cap = qb.max_kv <= kCacheCap ? qb.max_kv : 0;
  size_t smem = (size_t)cap * sizeof(uint32_t);
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  topk_kernel<<<qb.num_q, kThreads, smem, stream>>>(qb, scores, ld, k, idx, cap, err);
  return cudaGetLastError();
}

}  // namespace dsa
