// The fused forward's selection: the exact top-k of every query taken from
// the indexer's scores without writing them out (DeepSeek-V3.2 summary card,
// "How DSA Works": keep only the 2048 most relevant tokens per query; news
// article on DeepSeek-V3.2, sparse-attention section: a fine-grained selector
// keeps the top-k key/value positions of every query).
//
// Every key of a query is ranked by its composite key (score, then lower
// position), so the k largest composite keys are the selection, a unique set.
//
//   1. The indexer scores a sample of each query's keys: the key tiles 0, m,
//      2m, ... (kSample), into a small buffer of at most 32 tiles a row.
//   2. sel_threshold_kernel: per query, the r-th largest sampled composite
//      key G, r a margin of six standard deviations (plus 16) above the
//      expected number of samples that beat the row's k-th largest key, so
//      that at least k keys of the row are >= G.  It also clears the query's
//      candidate count (and block 0 the fallback queue).
//   3. The indexer scores all the other tiles (kFilter) and appends every key
//      whose composite key is >= G to the query's candidate list.
//   4. sel_select_kernel: the candidates plus the samples >= G hold every key
//      >= G.  With at least k of them (and no list overflow) the row's top k
//      are among them: an exact radix select of the k-th largest composite
//      key T, then every candidate >= T is written in ascending position
//      through a bitmap of the row's positions.  A row whose guess missed
//      (fewer than k keys >= G, or a full list) is queued for the fallback
//      (select_fallback.cu), which recomputes its scores and selects exactly.
//
// The result equals the top-k of the materialised score rows bit for bit:
// the same scores (same arithmetic), the same order (score, then position).
#include <algorithm>
#include <cmath>

#include "launch.h"
#include "topk_core.cuh"

namespace dsa {
namespace {

using namespace topk_core;

constexpr int kThrThreads = 256;
constexpr int kSelThreads = 512;
constexpr int kWinBits = 1 << 17;   // most positions per bitmap window of the ordered output (16 KiB)

// Sample layout of query row i: sampled tile o (key tile o*m) holds keys
// o*m*128 + j, j < 128, at samp[i*lds + o*128 + j].
__device__ __forceinline__ int sample_key(int x, int m) { return (x >> 7) * m * 128 + (x & 127); }
// Number of sample slots of a query at position pos (its sampled tiles hold keys <= pos).
__device__ __forceinline__ int sample_slots(int pos, int m) { return (pos / (m * 128) + 1) * 128; }

// The rank of the threshold among a query's samples: expected number of
// samples at or above the row's k-th largest key, f = S k / n, plus six
// standard deviations and 16; S when that reaches every sample.
__host__ __device__ __forceinline__ int threshold_rank(int S, int n, int k) {
  const double f = (double)S * (double)k / (double)n;
  const double r = ceil(f + 6.0 * sqrt(f) + 16.0);
  return r >= (double)S ? S : (int)r;
}

__global__ void __launch_bounds__(kThrThreads)
sel_threshold_kernel(QueryBatch qb, const float* __restrict__ samp, int64_t lds, int m, int k,
                     uint64_t* __restrict__ thr, uint32_t* __restrict__ cnt, uint32_t* __restrict__ fail_ctr) {
  __shared__ uint32_t hist[kBins];
  __shared__ uint32_t warp_tot[32];
  __shared__ TopkShared<kThrThreads> S;
  __shared__ uint32_t lo_min;
  __shared__ uint32_t hk[kSelSampleTiles * 128];   // the row's sample score keys
  const int i = blockIdx.x, tid = threadIdx.x;
  pdl_wait();
  pdl_release();
  if (tid == 0) {
    cnt[i] = 0;
    if (i == 0) {
      fail_ctr[0] = 0;   // rows queued for the fallback
      fail_ctr[1] = 0;   // rows the fallback has taken
    }
  }
  const int pos = __ldg(qb.q_pos + i);
  if (pos < k || pos >= qb.max_kv) return;   // nothing to select (n <= k) or an invalid row (flagged later)
  const int n = pos + 1;
  const int slots = sample_slots(pos, m);
  const int S_q = slots - 128 + min(128, pos - (slots / 128 - 1) * m * 128 + 1);   // samples at keys <= pos
  const int r = threshold_rank(S_q, n, k);
  if (r >= S_q) {   // every key is a candidate
    if (tid == 0) thr[i] = 0ull;
    return;
  }
  // the samples' score keys, converted once into shared memory for the
  // select's passes (each reads every sample)
  const float* row = samp + (int64_t)i * lds;
  for (int x = tid; x < slots; x += kThrThreads) hk[x] = score_key(__ldg(row + x));
  __syncthreads();
  const uint64_t G = select_kth_u64<kThrThreads>(
      slots,
      [&](int x, uint64_t& v) {
        const int s = sample_key(x, m);
        if (s > pos) return false;
        v = ((uint64_t)hk[x] << 32) | (uint64_t)(0xffffffffu - (uint32_t)s);
        return true;
      },
      (uint32_t)r, hist, warp_tot, S, &lo_min);
  if (tid == 0) thr[i] = G;
}

struct SelShared {
  uint32_t hist[kBins];
  uint32_t warp_tot[32];
  TopkShared<kSelThreads> S;
  uint32_t n_list, lo_min, out_base;
};

__global__ void __launch_bounds__(kSelThreads)
sel_select_kernel(QueryBatch qb, const float* __restrict__ samp, int64_t lds, int m, int k,
                  const uint64_t* __restrict__ thr, const uint32_t* __restrict__ cnt,
                  const uint64_t* __restrict__ cand, int cap, int list_cap, int win, int32_t* __restrict__ idx,
                  uint32_t* __restrict__ fail_ctr, uint32_t* __restrict__ fail_rows, int* err) {
  extern __shared__ __align__(16) unsigned char dsm[];
  uint32_t* bm = reinterpret_cast<uint32_t*>(dsm);                        // [win / 32] position bitmap
  uint64_t* list = reinterpret_cast<uint64_t*>(dsm + win / 8);           // [list_cap] candidate keys
  __shared__ SelShared Z;
  const int i = blockIdx.x, tid = threadIdx.x;
  pdl_wait();
  pdl_release();
  int32_t* out = idx + (int64_t)i * k;
  const int pos = __ldg(qb.q_pos + i);
  if (pos < 0 || pos >= qb.max_kv) {
    if (tid == 0) flag_error(err, DSA_ERR_BOUNDS);
    for (int j = tid; j < k; j += kSelThreads) out[j] = -1;
    return;
  }
  const int n = pos + 1;
  if (n <= k) {
    for (int j = tid; j < k; j += kSelThreads) out[j] = j < n ? j : -1;
    return;
  }
  const uint32_t c = __ldg(cnt + i);
  const uint64_t G = __ldg(thr + i);
  bool fail = c > (uint32_t)cap;   // the candidate list overflowed
  if (!fail) {
    // the candidates, then the samples >= G, into the shared list
    const uint64_t* cr = cand + (int64_t)i * cap;
    for (uint32_t j = tid; j < c && j < (uint32_t)list_cap; j += kSelThreads) list[j] = __ldg(cr + j);
    if (tid == 0) Z.n_list = c;
    __syncthreads();
    const float* srow = samp + (int64_t)i * lds;
    const int slots = sample_slots(pos, m);
    for (int x = tid; x < slots; x += kSelThreads) {
      const int s = sample_key(x, m);
      if (s > pos) continue;
      const uint64_t v = composite_key(__ldg(srow + x), s);
      if (v >= G) {
        const uint32_t at = atomicAdd(&Z.n_list, 1u);
        if (at < (uint32_t)list_cap) list[at] = v;
      }
    }
    __syncthreads();
    fail = Z.n_list < (uint32_t)k || Z.n_list > (uint32_t)list_cap;   // the guess missed (block-uniform)
  }
  if (fail) {
    if (tid == 0) fail_rows[atomicAdd(fail_ctr, 1u)] = (uint32_t)i;
    return;
  }
  const int total = (int)Z.n_list;
  // the k-th largest composite key: every key >= G is in the list and at
  // least k of them are, so it is the row's k-th largest
  const uint64_t T = select_kth_u64<kSelThreads>(
      total,
      [&](int j, uint64_t& v) {
        v = list[j];
        return true;
      },
      (uint32_t)k, Z.hist, Z.warp_tot, Z.S, &Z.lo_min);
  // ascending output: the selected positions of each window of the row's
  // positions marked in a bitmap, then written in order (one contiguous run
  // of words per thread, offsets from a block scan)
  if (tid == 0) Z.out_base = 0;
  for (int w0 = 0; w0 < n; w0 += win) {
    const int words = (min(win, n - w0) + 31) / 32;
    for (int j = tid; j < words; j += kSelThreads) bm[j] = 0u;
    __syncthreads();
    for (int j = tid; j < total; j += kSelThreads) {
      const uint64_t v = list[j];
      const int p = composite_pos(v) - w0;
      if (v >= T && p >= 0 && p < win) atomicOr(bm + (p >> 5), 1u << (p & 31));
    }
    __syncthreads();
    const int per = (words + kSelThreads - 1) / kSelThreads;
    const int wb = min(words, tid * per), we = min(words, wb + per);
    uint32_t mine = 0;
    for (int j = wb; j < we; ++j) mine += __popc(bm[j]);
    const uint32_t incl = block_incl_scan<kSelThreads>(mine, Z.warp_tot);
    uint32_t slot = Z.out_base + incl - mine;
    for (int j = wb; j < we; ++j) {
      uint32_t b = bm[j];
      while (b) {
        const int bit = __ffs(b) - 1;
        b &= b - 1;
        if (slot < (uint32_t)k) out[slot] = w0 + 32 * j + bit;
        else flag_error(err, DSA_ERR_BOUNDS);   // cannot happen for an exact select; never write past the row
        ++slot;
      }
    }
    __syncthreads();
    if (tid == kSelThreads - 1) Z.out_base += incl;
    __syncthreads();
  }
}

}  // namespace

SelectPlan plan_select(int max_kv, int k) {
  SelectPlan p;
  const int T = (max_kv + 127) / 128;
  p.m = std::max(1, (T + kSelSampleTiles - 1) / kSelSampleTiles);
  p.lds = (int64_t)((T + p.m - 1) / p.m) * 128;
  // capacity of a row's candidate list: over the possible row lengths n,
  // the expected number of keys >= G (r n / S) plus eight standard deviations
  // (sqrt(r) n / S), at most n
  int64_t cap = 256;
  for (int q = 0; q <= 64; ++q) {
    const int n = k + 1 + (int)((int64_t)(max_kv - k - 1) * q / 64);
    if (n <= k || n > max_kv) continue;
    const int pos = n - 1;
    const int slots = (pos / (p.m * 128) + 1) * 128;
    const int S_q = slots - 128 + std::min(128, pos - (slots / 128 - 1) * p.m * 128 + 1);
    const int r = threshold_rank(S_q, n, k);
    const double per = (double)n / S_q;
    const double want = std::min((double)n, r * per + 8.0 * std::sqrt((double)r) * per + 64.0);
    cap = std::max<int64_t>(cap, (int64_t)std::ceil(want));
  }
  p.cap = (int)((cap + 63) & ~int64_t(63));
  // The shared list holds the candidates and the samples >= G: exactly r of
  // them, r = threshold_rank(S, n, k).  A row's S is at most n/m + 128, so
  // f = S k / n < k/m + 128 =: F, and r <= ceil(F + 6 sqrt(F) + 16) (r grows
  // with f); r <= S <= lds as well.  Sized to that bound instead of to all
  // the samples, the list leaves room for three or four blocks an SM.
  const double F = (double)k / p.m + 128.0;
  const int64_t r_bound = std::min<int64_t>(p.lds, (int64_t)std::ceil(F + 6.0 * std::sqrt(F) + 16.0));
  p.list_cap = p.cap + (int)r_bound;
  // the bitmap covers a whole row when the cache is shorter than a window
  p.win = (int)std::min<int64_t>(kWinBits, ((int64_t)max_kv + 63) & ~int64_t(63));
  return p;
}

size_t select_shared_bytes(const SelectPlan& p) { return (size_t)p.win / 8 + (size_t)p.list_cap * 8; }

cudaError_t launch_sel_threshold(const QueryBatch& qb, const SelectPlan& p, const float* samp, int k, uint64_t* thr,
                                 uint32_t* cnt, uint32_t* fail_ctr, cudaStream_t stream) {
  return launch_pdl(sel_threshold_kernel, dim3(qb.num_q), dim3(kThrThreads), 0, stream, qb, samp, p.lds, p.m, k, thr,
                    cnt, fail_ctr);
}

cudaError_t launch_sel_select(const QueryBatch& qb, const SelectPlan& p, const float* samp, int k, const uint64_t* thr,
                              const uint32_t* cnt, const uint64_t* cand, int32_t* idx, uint32_t* fail_ctr,
                              uint32_t* fail_rows, int* err, cudaStream_t stream) {
  const int smem = (int)select_shared_bytes(p);
  cudaError_t e = cudaFuncSetAttribute(sel_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(sel_select_kernel, dim3(qb.num_q), dim3(kSelThreads), (size_t)smem, stream, qb, samp, p.lds, p.m,
                    k, thr, cnt, cand, p.cap, p.list_cap, p.win, idx, fail_ctr, fail_rows, err);
}

}  // namespace dsa
