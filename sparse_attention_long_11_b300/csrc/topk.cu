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
constexpr int kCandCap = 8192;     // threshold-bin keys gathered for the finer rounds (32 KiB)

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

// Selects, among the nb bins of `hist` (counts of candidates sharing a
// digit), the one holding the krem-th largest candidate: sets *sel_bin and
// *sel_above (candidates in higher bins).  Thread t owns the bins of
// descending rank 2t and 2t+1.  Ends with a barrier.
__device__ __forceinline__ void select_bin(const uint32_t* hist, int nb, uint32_t krem, uint32_t* warp_tot,
                                           uint32_t* sel_bin, uint32_t* sel_above) {
  const int tid = threadIdx.x;
  const int b0 = nb - 1 - 2 * tid, b1 = b0 - 1;
  const uint32_t h0 = b0 >= 0 ? hist[b0] : 0u, h1 = b1 >= 0 ? hist[b1] : 0u;
  const uint32_t incl = block_incl_scan(h0 + h1, warp_tot);
  const uint32_t excl = incl - h0 - h1;
  if (excl < krem && krem <= excl + h0) {
    *sel_bin = (uint32_t)b0;
    *sel_above = excl;
  } else if (excl + h0 < krem && krem <= incl) {
    *sel_bin = (uint32_t)b1;
    *sel_above = excl + h0;
  }
  __syncthreads();
}

// Warp-wide exclusive prefix sum of v (and the warp total in *tot).
__device__ __forceinline__ uint32_t warp_excl_scan(uint32_t v, uint32_t* tot) {
  const int lane = threadIdx.x & 31;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += t;
  }
  *tot = __shfl_sync(0xffffffffu, x, 31);
  return x - v;
}

// Keys of candidates j .. j+3 (j a multiple of 4; entries >= n are don't-care).
struct RowKeys {
  const float* row;
  const uint32_t* skey;
  int n;
  bool cached, vec;
  __device__ __forceinline__ uint4 load4(int j) const {
    if (cached) return *reinterpret_cast<const uint4*>(skey + j);
    return load4_global(j);
  }
  __device__ __forceinline__ uint4 load4_global(int j) const {
    if (vec && j + 3 < n) {
      const float4 x = __ldg(reinterpret_cast<const float4*>(row + j));
      return make_uint4(score_key(x.x), score_key(x.y), score_key(x.z), score_key(x.w));
    }
    uint32_t u[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) u[e] = j + e < n ? score_key(__ldg(row + j + e)) : 0u;
    return make_uint4(u[0], u[1], u[2], u[3]);
  }
};

__global__ void __launch_bounds__(kThreads, 1)
topk_kernel(QueryBatch qb, const float* __restrict__ scores, int64_t ld, int k,
            int32_t* __restrict__ idx, int cache_cap, int* err) {
  extern __shared__ __align__(16) uint32_t smem[];   // [cache_cap] keys, then [kCandCap] candidates
  uint32_t* skey = smem;
  uint32_t* cand = smem + cache_cap;
  __shared__ uint32_t hist[kBins];
  __shared__ uint32_t warp_tot[32];
  __shared__ uint32_t sel_bin, sel_above, n_cand;
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
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15) == 0;
  const RowKeys rk{row, skey, n, cached, vec};
  const int n4 = (n + 3) >> 2;   // groups of four candidates

  // ---- round 0: histogram of the top 11 bits over the whole row (keys cached on the way)
  for (int b = tid; b < kBins; b += kThreads) hist[b] = 0;
  if (tid == 0) n_cand = 0;
  __syncthreads();
#pragma unroll 1
  for (int q0 = tid; q0 < n4; q0 += 2 * kThreads) {
    const int q1 = q0 + kThreads;
    // both loads in flight before any use; round 0 always reads the scores themselves
    const uint4 a = rk.load4_global(4 * q0);
    const uint4 c = q1 < n4 ? rk.load4_global(4 * q1) : make_uint4(0, 0, 0, 0);
    const uint32_t ua[4] = {a.x, a.y, a.z, a.w}, uc[4] = {c.x, c.y, c.z, c.w};
    if (cached) {
      reinterpret_cast<uint4*>(skey)[q0] = a;
      if (q1 < n4) reinterpret_cast<uint4*>(skey)[q1] = c;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (4 * q0 + e < n) atomicAdd(&hist[ua[e] >> 21], 1u);
      if (q1 < n4 && 4 * q1 + e < n) atomicAdd(&hist[uc[e] >> 21], 1u);
    }
  }
  __syncthreads();
  uint32_t krem = (uint32_t)k;
  select_bin(hist, kBins, krem, warp_tot, &sel_bin, &sel_above);
  uint32_t prefix = sel_bin << 21, pmask = 0xffe00000u;
  krem -= sel_above;
  const uint32_t c1 = hist[sel_bin];   // candidates in the threshold bin (>= 1)
  __syncthreads();

  // ---- rounds 1 (11 bits) and 2 (10 bits): over the threshold bin's keys,
  // gathered into a compact list when they fit, else over the whole row
  const bool compact = c1 <= (uint32_t)kCandCap;
  if (compact) {
#pragma unroll 1
    for (int q = tid; q - tid < n4; q += kThreads) {   // warp-uniform bound: every lane takes part in the scan
      uint4 v = make_uint4(0, 0, 0, 0);
      if (q < n4) v = rk.load4(4 * q);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
      uint32_t m = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (q < n4 && 4 * q + e < n && (u[e] & pmask) == prefix) m |= 1u << e;
      uint32_t tot;
      const uint32_t off = warp_excl_scan(__popc(m), &tot);
      uint32_t base = 0;
      if (lane == 0 && tot) base = atomicAdd(&n_cand, tot);
      base = __shfl_sync(0xffffffffu, base, 0) + off;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (m & (1u << e)) cand[base++] = u[e];
    }
    __syncthreads();
  }
#pragma unroll 1
  for (int round = 1; round < 3; ++round) {
    const int shift = round == 1 ? 10 : 0;
    const int nb = round == 1 ? 2048 : 1024;
    for (int b = tid; b < kBins; b += kThreads) hist[b] = 0;
    __syncthreads();
    if (compact) {
      for (int j = tid; j < (int)c1; j += kThreads) {
        const uint32_t u = cand[j];
        if ((u & pmask) == prefix) atomicAdd(&hist[(u >> shift) & (nb - 1)], 1u);
      }
    } else {
      for (int q = tid; q < n4; q += kThreads) {
        const uint4 v = rk.load4(4 * q);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (4 * q + e < n && (u[e] & pmask) == prefix) atomicAdd(&hist[(u[e] >> shift) & (nb - 1)], 1u);
      }
    }
    __syncthreads();
    select_bin(hist, nb, krem, warp_tot, &sel_bin, &sel_above);
    prefix |= sel_bin << shift;
    pmask |= (uint32_t)(nb - 1) << shift;
    krem -= sel_above;
    __syncthreads();
  }
  const uint32_t T = prefix;   // key of the k-th largest candidate
  const uint32_t need = krem;  // candidates equal to T to take (>= 1)

  // ---- ordered compaction: warp w owns the contiguous segment [w*seg, (w+1)*seg)
  // (seg a multiple of 128: each warp step covers 128 candidates, four per lane)
  const int seg = ((n + kWarps - 1) / kWarps + 127) & ~127;
  const int beg = warp * seg, end = min(n, beg + seg);
  uint32_t gt = 0, eq = 0;
  for (int j = beg + 4 * lane; j < end; j += 128) {
    const uint4 v = rk.load4(j);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const bool ok = j + e < end;
      gt += ok && u[e] > T;
      eq += ok && u[e] == T;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    gt += __shfl_xor_sync(0xffffffffu, gt, o);
    eq += __shfl_xor_sync(0xffffffffu, eq, o);
  }
  if (lane == 0) { w_gt[warp] = gt; w_eq[warp] = eq; }
  __syncthreads();
  if (warp == 0) {
    // exclusive scans over the warps: equal keys before each segment, and
    // selected entries before it (all greater keys + the first `need` equal ones)
    const uint32_t e_w = w_eq[lane], g_w = w_gt[lane];
    uint32_t e_tot;
    const uint32_t e_ex = warp_excl_scan(e_w, &e_tot);
    const uint32_t take = need > e_ex ? min(need - e_ex, e_w) : 0u;
    uint32_t s_tot;
    w_selbase[lane] = warp_excl_scan(g_w + take, &s_tot);
    w_eqbase[lane] = e_ex;
  }
  __syncthreads();
  uint32_t eq_run = w_eqbase[warp], sel_run = w_selbase[warp];
  for (int j0 = beg; j0 < end; j0 += 128) {   // warp-uniform bound
    const int j = j0 + 4 * lane;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (j < end) v = rk.load4(j);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
    uint32_t me = 0, mg = 0;   // this lane's equal / greater candidates (bit e = candidate j+e)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (j + e < end && u[e] == T) me |= 1u << e;
      if (j + e < end && u[e] > T) mg |= 1u << e;
    }
    uint32_t e_tot;
    const uint32_t e_before = eq_run + warp_excl_scan(__popc(me), &e_tot);
    // the equal candidates taken: the first `need` in position order
    uint32_t mt = mg, er = e_before;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (me & (1u << e)) {
        if (er < need) mt |= 1u << e;
        ++er;
      }
    uint32_t s_tot;
    uint32_t slot = sel_run + warp_excl_scan(__popc(mt), &s_tot);
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (mt & (1u << e)) {
        if (slot < (uint32_t)k) out[slot] = j + e;
        else flag_error(err, DSA_ERR_BOUNDS);   // cannot happen for a consistent select; never write past the row
        ++slot;
      }
    eq_run += e_tot;
    sel_run += s_tot;
  }
}

}  // namespace

cudaError_t launch_topk(const QueryBatch& qb, const float* scores, int64_t ld, int k, int32_t* idx,
                        int* err, cudaStream_t stream) {
  int cap = qb.max_kv <= kCacheCap ? ((qb.max_kv + 3) & ~3) : 0;   // a multiple of 4: the list behind it stays 16-B aligned
  size_t smem = ((size_t)cap + kCandCap) * sizeof(uint32_t);
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  topk_kernel<<<qb.num_q, kThreads, smem, stream>>>(qb, scores, ld, k, idx, cap, err);
  return cudaGetLastError();
}

}  // namespace dsa
