// Block-wide building blocks of the exact top-k selection, shared by the
// stand-alone top-k, the fused selection's threshold and select kernels and
// its fallback: radix rounds over order-preserving 32-bit keys (2048-bin
// histograms in shared memory, 11 + 11 + 10 bits), block and warp scans, and
// the whole-row exact selection with an ordered compaction (ties to the lower
// position).  Header-only device code; every function is called by all NT
// threads of a block (it synchronises the block).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace dsa {
namespace topk_core {

constexpr int kBins = 2048;
constexpr int kCandCap = 4096;   // threshold-bin keys gathered for the finer rounds (the candidate-list buffer)
constexpr int kManyRowsThreads = 512, kFewRowsThreads = 1024;
constexpr int kLongRow = 65536;   // rows beyond this many keys scan faster with 1024-thread blocks

template <int NT>
__device__ __forceinline__ uint32_t block_incl_scan(uint32_t v, uint32_t* warp_tot) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t t = lane < NW ? warp_tot[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t u = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += u;
    }
    if (lane < NW) warp_tot[lane] = t;   // inclusive over warps
  }
  __syncthreads();
  const uint32_t r = v + (warp > 0 ? warp_tot[warp - 1] : 0u);
  __syncthreads();
  return r;
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

// Selects, among the nb bins of `hist` (counts of candidates sharing a
// digit), the one holding the krem-th largest candidate: sets *sel_bin and
// *sel_above (candidates in higher bins).  Thread t owns the nb / NT bins of
// descending rank nb/NT * t onwards.  Ends with a barrier.
template <int NT>
__device__ __forceinline__ void select_bin(const uint32_t* hist, int nb, uint32_t krem, uint32_t* warp_tot,
                                           uint32_t* sel_bin, uint32_t* sel_above) {
  constexpr int BMAX = kBins / NT;
  const int tid = threadIdx.x;
  const int nper = (nb + NT - 1) / NT;   // nb a power of two up to kBins: at most BMAX bins each
  uint32_t h[BMAX], sum = 0;
#pragma unroll
  for (int r = 0; r < BMAX; ++r) {
    const int rank = nper * tid + r;
    h[r] = (r < nper && rank < nb) ? hist[nb - 1 - rank] : 0u;
    sum += h[r];
  }
  const uint32_t incl = block_incl_scan<NT>(sum, warp_tot);
  const uint32_t excl = incl - sum;
  if (excl < krem && krem <= incl) {   // exactly one thread's bins hold the krem-th candidate
    uint32_t c = excl;
#pragma unroll
    for (int r = 0; r < BMAX; ++r) {
      if (r < nper && nper * tid + r < nb && c < krem && krem <= c + h[r]) {
        *sel_bin = (uint32_t)(nb - 1 - (nper * tid + r));
        *sel_above = c;
      }
      c += h[r];
    }
  }
  __syncthreads();
}

// Keys of candidates j .. j+3 of one score row (j a multiple of 4; entries
// >= n read as 0 and must be masked by the caller).
struct RowKeys {
  const float* row;
  int n;
  bool vec;   // row start 16-byte aligned
  __device__ __forceinline__ uint4 load4(int j) const {
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

constexpr int kSamples = 1024;

// Smallest per-warp capacity of the candidate list (keys and positions in
// dynamic shared memory, 8 bytes a slot); the launch raises it for large k or
// long rows.  NW * kPerWarp >= kCandCap, which the fallback needs.
template <int NT> struct Region;
template <> struct Region<512> { static constexpr int kPerWarp = 256; };    // 32 KiB a block: four blocks per SM
template <> struct Region<1024> { static constexpr int kPerWarp = 256; };
constexpr int kMaxListBytes = 200 << 10;   // dynamic shared memory cap for the list

template <int NT>
struct TopkShared {
  uint32_t sel_bin, sel_above, n_cand, overflow;
  uint32_t w_cnt[NT / 32], w_gt[NT / 32], w_eq[NT / 32], w_selbase[NT / 32], w_eqbase[NT / 32];
};

// Exact selection over the whole row by radix rounds (used when the sampled
// threshold misses): writes the row's output.  `cand` holds kCandCap keys.
template <int NT>
__device__ __noinline__ void radix_path(const RowKeys rk, int k, int32_t* __restrict__ out, int* err,
                                        uint32_t* hist, uint32_t* cand, uint32_t* warp_tot, TopkShared<NT>& S) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = rk.n;
  const int n4 = (n + 3) >> 2;
  uint32_t& sel_bin = S.sel_bin;
  uint32_t& sel_above = S.sel_above;
  uint32_t& n_cand = S.n_cand;
  uint32_t* w_gt = S.w_gt;
  uint32_t* w_eq = S.w_eq;
  uint32_t* w_selbase = S.w_selbase;
  uint32_t* w_eqbase = S.w_eqbase;
  __syncthreads();
  // ---- round 0: histogram of the top 11 bits over the whole row
  for (int b = tid; b < kBins; b += NT) hist[b] = 0;
  if (tid == 0) {
    n_cand = 0;
    sel_bin = 0;   // always overwritten by a consistent select; never left undefined
    sel_above = 0;
  }
  __syncthreads();
#pragma unroll 1
  for (int q = tid; q < n4; q += 4 * NT) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {   // four 16-byte loads in flight before any use
      const int qq = q + u * NT;
      v[u] = qq < n4 ? rk.load4(4 * qq) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int qq = q + u * NT;
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (qq < n4 && 4 * qq + e < n) atomicAdd(&hist[w[e] >> 21], 1u);
    }
  }
  __syncthreads();
  uint32_t krem = (uint32_t)k;
  select_bin<NT>(hist, kBins, krem, warp_tot, &sel_bin, &sel_above);
  uint32_t prefix = sel_bin << 21, pmask = 0xffe00000u;
  krem -= sel_above;
  const uint32_t c1 = hist[sel_bin];   // candidates in the threshold bin (>= 1)
  __syncthreads();

  // ---- rounds 1 (11 bits) and 2 (10 bits): over the threshold bin's keys,
  // gathered into a compact list when they fit, else over the whole row
  const bool compact = c1 <= (uint32_t)kCandCap;
  if (compact) {
#pragma unroll 1
    for (int q = tid; q - tid < n4; q += NT) {   // warp-uniform bound: every lane takes part in the scan
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
    for (int b = tid; b < kBins; b += NT) hist[b] = 0;
    __syncthreads();
    if (compact) {
      for (int j = tid; j < (int)c1; j += NT) {
        const uint32_t u = cand[j];
        if ((u & pmask) == prefix) atomicAdd(&hist[(u >> shift) & (nb - 1)], 1u);
      }
    } else {
      for (int q = tid; q < n4; q += NT) {
        const uint4 v = rk.load4(4 * q);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (4 * q + e < n && (u[e] & pmask) == prefix) atomicAdd(&hist[(u[e] >> shift) & (nb - 1)], 1u);
      }
    }
    __syncthreads();
    select_bin<NT>(hist, nb, krem, warp_tot, &sel_bin, &sel_above);
    prefix |= sel_bin << shift;
    pmask |= (uint32_t)(nb - 1) << shift;
    krem -= sel_above;
    __syncthreads();
  }
  const uint32_t T = prefix;   // key of the k-th largest candidate
  const uint32_t need = krem;  // candidates equal to T to take (>= 1)

  // ---- ordered compaction: warp w owns the contiguous segment [w*seg, (w+1)*seg)
  // (seg a multiple of 128: each warp step covers 128 candidates, four per lane)
  const int seg = ((n + NW - 1) / NW + 127) & ~127;
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
  if (lane == 0) {
    w_gt[warp] = gt;
    w_eq[warp] = eq;
  }
  __syncthreads();
  if (warp == 0) {
    // exclusive scans over the warps: equal keys before each segment, and
    // selected entries before it (all greater keys + the first `need` equal ones)
    const uint32_t e_w = lane < NW ? w_eq[lane] : 0u, g_w = lane < NW ? w_gt[lane] : 0u;
    uint32_t e_tot;
    const uint32_t e_ex = warp_excl_scan(e_w, &e_tot);
    const uint32_t take = need > e_ex ? min(need - e_ex, e_w) : 0u;
    uint32_t s_tot;
    const uint32_t s_ex = warp_excl_scan(g_w + take, &s_tot);
    if (lane < NW) {
      w_selbase[lane] = s_ex;
      w_eqbase[lane] = e_ex;
    }
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

// k-th largest key of a list held in shared memory: radix rounds (11 + 11
// + 10 bits) over the entries i < total for which get(i) is valid.  With
// all three rounds the result is exact: the key T, and *need = how many
// entries equal to T belong to the top k_rank.  With two rounds it is the
// 22-bit prefix of that key (a lower bound on it, exact to 2^-13 relative).
template <int NT, class Get>
__device__ __forceinline__ uint32_t select_in_list(int total, Get get, uint32_t k_rank, uint32_t* hist,
                                                   uint32_t* warp_tot, TopkShared<NT>& S, uint32_t* need,
                                                   int rounds = 3, uint32_t* final_count = nullptr) {
  const int tid = threadIdx.x;
  uint32_t prefix = 0, pmask = 0, krem = k_rank;
#pragma unroll 1
  for (int round = 0; round < rounds; ++round) {
    const int shift = round == 0 ? 21 : (round == 1 ? 10 : 0);
    const int nb = round == 2 ? 1024 : 2048;
    for (int b = tid; b < kBins; b += NT) hist[b] = 0;
    __syncthreads();
    for (int i = tid; i < total; i += NT) {
      uint32_t u;
      if (get(i, u) && (u & pmask) == prefix) atomicAdd(&hist[(u >> shift) & (nb - 1)], 1u);
    }
    __syncthreads();
    select_bin<NT>(hist, nb, krem, warp_tot, &S.sel_bin, &S.sel_above);
    prefix |= S.sel_bin << shift;
    pmask |= (uint32_t)(nb - 1) << shift;
    krem -= S.sel_above;
    __syncthreads();
  }
  *need = krem;
  // entries whose key equals the result (after three rounds): the selected
  // bin's count in the last histogram, read before anyone rewrites it
  if (final_count) *final_count = hist[S.sel_bin];
  __syncthreads();
  return prefix;
}

// The k_rank-th largest of the 64-bit values get(i) over the valid entries
// 0 <= i < total (k_rank <= their number): exact.  The high words are
// selected first (three rounds); when the entries sharing the selected high
// word are not all taken, three more rounds select among their low words.
template <int NT, class Get>
__device__ __forceinline__ uint64_t select_kth_u64(int total, Get get, uint32_t k_rank, uint32_t* hist,
                                                   uint32_t* warp_tot, TopkShared<NT>& S, uint32_t* lo_min) {
  uint32_t need, eq;
  const uint32_t hi = select_in_list<NT>(
      total,
      [&](int i, uint32_t& u) {
        uint64_t v;
        if (!get(i, v)) return false;
        u = (uint32_t)(v >> 32);
        return true;
      },
      k_rank, hist, warp_tot, S, &need, 3, &eq);
  uint32_t lo;
  if (need == eq) {   // every entry with this high word is taken: the smallest low word among them
    if (threadIdx.x == 0) *lo_min = 0xffffffffu;
    __syncthreads();
    uint32_t m = 0xffffffffu;
    for (int i = threadIdx.x; i < total; i += NT) {
      uint64_t v;
      if (get(i, v) && (uint32_t)(v >> 32) == hi) m = min(m, (uint32_t)v);
    }
    atomicMin(lo_min, m);
    __syncthreads();
    lo = *lo_min;
    __syncthreads();
  } else {
    uint32_t need2;
    lo = select_in_list<NT>(
        total,
        [&](int i, uint32_t& u) {
          uint64_t v;
          if (!get(i, v) || (uint32_t)(v >> 32) != hi) return false;
          u = (uint32_t)v;
          return true;
        },
        need, hist, warp_tot, S, &need2);
  }
  return ((uint64_t)hi << 32) | lo;
}


}  // namespace topk_core
}  // namespace dsa
