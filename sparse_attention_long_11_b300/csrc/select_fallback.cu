// Exact selection for the rows whose sampled threshold missed in the fused
// forward (select.cu): too few keys at or above it, or more than the
// candidate list holds (an adversarial or heavily tied row).  Each such row's
// scores are recomputed on the tensor cores with the lightning indexer's own
// instruction and epilogue arithmetic (kind::f8f6f4 MMA, 128 keys x the
// query's 64 heads, then idx_epi::head_sum64 and the key scale), so they are
// the indexer's scores bit for bit; they are written to one score row per
// CTA, and the exact radix selection of the stand-alone top-k runs on it.
//
// Persistent: every CTA takes queued rows one at a time until the queue is
// empty (a launch that finds it empty returns at once, before any set-up).
// Warps 0-3 are the epilogue (TMEM lane quadrants 0-3), warp 4 lane 0 loads
// key tiles by TMA (two 64-row boxes, so paged caches are read block by
// block) and issues the MMAs into two 64-column accumulators; all 16 warps
// then run the selection.  All waits are bounded.
#include <algorithm>

#include "indexer_epi.cuh"
#include "launch.h"
#include "tc.cuh"
#include "tmap.h"
#include "topk_core.cuh"

namespace dsa {
namespace {
using namespace tc;
using namespace topk_core;

constexpr int kFbThreads = 512;
constexpr int kHI = 64, kKT = 128;
constexpr uint32_t kQBytes = kHI * 128;   // one query's 64 head rows of 128 codes
constexpr uint32_t kABytes = kKT * 128;   // one key tile
constexpr uint32_t kOffA = kQBytes;       // two key-tile stages after the query tile
constexpr uint32_t kSmemBytes = kOffA + 2 * kABytes;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;

struct FbShared {
  uint64_t a_full[2], a_free[2], d_full[2], d_empty[2], q_full, fin;
  alignas(16) float wq[kHI];
  uint32_t hist[kBins];
  uint32_t cand[kCandCap];
  uint32_t warp_tot[32];
  TopkShared<kFbThreads> T;
  uint32_t tmem_base;
  int row;
  int abort;
};

// Next queued row, or -1.
__device__ __forceinline__ int next_row(uint32_t* fail_ctr, const uint32_t* fail_rows) {
  const uint32_t n = *reinterpret_cast<volatile uint32_t*>(fail_ctr);
  const uint32_t at = atomicAdd(fail_ctr + 1, 1u);
  return at < n ? (int)fail_rows[at] : -1;
}

__global__ void __launch_bounds__(kFbThreads, 1)
sel_fallback_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k, QueryBatch qb,
                    CacheMap cm, const float* __restrict__ q_scale, const float* __restrict__ w,
                    const float* __restrict__ k_scale, int k, int32_t* __restrict__ idx, float* __restrict__ slots,
                    int64_t ld, uint32_t* fail_ctr, const uint32_t* __restrict__ fail_rows, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ FbShared S;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_wait();
  pdl_release();
  if (tid == 0) S.row = next_row(fail_ctr, fail_rows);
  __syncthreads();
  if (S.row < 0) return;   // nothing queued for this CTA

  volatile int* abort = &S.abort;
  const uint32_t sQ = smem_u32(sm), sA = smem_u32(sm + kOffA);
  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.a_full[b], 1);
      mbar_init(&S.a_free[b], 1);
      mbar_init(&S.d_full[b], 1);
      mbar_init(&S.d_empty[b], 128);
    }
    mbar_init(&S.q_full, 1);
    mbar_init(&S.fin, 1);
    S.abort = 0;
    fence_mbar_init();
  }
  if (warp == 4) {
    tmem_alloc(&S.tmem_base, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  float* slot = slots + (int64_t)blockIdx.x * ld;
  const uint32_t idesc = idesc_e4m3(128, kHI);

  uint32_t g0 = 0, nrow = 0;   // key tiles and rows done by this CTA (barrier phases)
  uint32_t issued = 0;         // key tiles whose TMA warp 4 has issued
  while (S.row >= 0 && !*abort) {
    const int i = S.row;
    const int seq = __ldg(qb.q_seq + i), pos = __ldg(qb.q_pos + i);
    const int n = pos + 1, T = (n + kKT - 1) / kKT;
    if (tid < kHI)
      S.wq[tid] = idx_epi::fold_weight(tid, __ldg(w + (int64_t)i * kHI + tid) * __ldg(q_scale + (int64_t)i * kHI + tid));
    __syncthreads();

    if (warp == 4) {
      // ---------------------------------------------------- TMA + MMA (lane 0)
      if (lane == 0) {
        auto load_tile = [&](uint32_t gt, int t) {
          const int st = gt & 1;
          int64_t rows[2];
          uint32_t bytes = 0;
          for (int hh = 0; hh < 2; ++hh) {
            const int sh = t * kKT + 64 * hh;
            rows[hh] = -1;
            if (sh > pos) continue;
            if (cm.block_size == 0) {
              rows[hh] = (int64_t)seq * cm.seq_stride + sh;
            } else {
              const int blk = sh / cm.block_size;
              const int phys = blk < cm.max_blocks ? __ldg(cm.block_table + (int64_t)seq * cm.max_blocks + blk) : -1;
              const int64_t r0 = (int64_t)phys * cm.block_size + (sh - blk * cm.block_size);
              if (phys < 0 || r0 + 64 > cm.num_rows) flag_error(err, DSA_ERR_BOUNDS);
              else rows[hh] = r0;
            }
            if (rows[hh] >= 0) bytes += 64 * 128;
          }
          mbar_arrive_expect_tx(&S.a_full[st], bytes);
          for (int hh = 0; hh < 2; ++hh)
            if (rows[hh] >= 0) tma_load_2d(sA + st * kABytes + hh * 8192, &tm_k, 0, (int32_t)rows[hh], &S.a_full[st]);
          ++issued;
        };
        mbar_arrive_expect_tx(&S.q_full, kQBytes);
        tma_load_2d(sQ, &tm_q, 0, i * kHI, &S.q_full);
        for (int t = 0; t < T && t < 2; ++t) load_tile(g0 + t, t);
        bool ok = mbar_wait(&S.q_full, nrow & 1, abort);
        for (int t = 0; t < T && ok; ++t) {
          const uint32_t gt = g0 + t, st = gt & 1, ph = (gt >> 1) & 1;
          if (!(ok = mbar_wait(&S.a_full[st], ph, abort))) break;
          if (!(ok = mbar_wait(&S.d_empty[st], ph ^ 1, abort))) break;
          tc_fence_after();
          const Desc2 ad = desc2(sdesc(sA + st * kABytes, 16, 1024)), qd = desc2(sdesc(sQ, 16, 1024));
          mma_e4m3_2<0>(tmem + 64 * st, ad, qd, idesc);
#pragma unroll
          for (int kk = 1; kk < 4; ++kk) mma_e4m3_2<1>(tmem + 64 * st, desc_at(ad, kk * 32), desc_at(qd, kk * 32), idesc);
          mma_commit(&S.d_full[st]);
          mma_commit(&S.a_free[st]);
          if (t + 2 < T) {   // reuse this stage for tile t + 2 once its MMAs have read it
            if (!(ok = mbar_wait(&S.a_free[st], ph, abort))) break;
            load_tile(gt + 2, t + 2);
          }
        }
        if (!ok) {
          // drain before the CTA exits: the TMA loads issued here and the MMAs
          for (uint32_t st = 0; st < 2 && st < issued; ++st) {
            const uint32_t last = st + 2 * ((issued - 1 - st) / 2);
            mbar_wait_own(&S.a_full[st], (last >> 1) & 1);
          }
          mbar_wait_own(&S.q_full, nrow & 1);
        }
      }
      __syncwarp();
    } else if (warp < 4) {
      // ---------------------------------------------------- epilogue (quadrant = warp)
      const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
      const float4* wq4 = reinterpret_cast<const float4*>(S.wq);
      for (int t = 0; t < T; ++t) {
        const uint32_t gt = g0 + t, st = gt & 1, ph = (gt >> 1) & 1;
        const int s = t * kKT + warp * 32 + lane;
        float sk = 0.f;
        bool key_ok = s <= pos;
        if (key_ok) {
          const int64_t row = cache_row(cm, seq, s, err);
          key_ok = row >= 0;
          if (key_ok) sk = __ldg(k_scale + row);
        }
        if (!mbar_wait_warp(&S.d_full[st], ph, abort)) break;
        tc_fence_after();
        const float acc = idx_epi::head_sum64(tmem + lane_base + 64 * st, wq4);
        if (s <= pos) slot[s] = key_ok ? acc * sk : -INFINITY;
        tc_fence_before();
        mbar_arrive(&S.d_empty[st]);
      }
    }
    g0 += T;
    ++nrow;
    tc_fence_before();
    __syncthreads();
    if (*abort) break;
    // ------------------------------------------------------ exact selection (all warps)
    const RowKeys rk{slot, n, true};
    radix_path<kFbThreads>(rk, k, idx + (int64_t)i * k, err, S.hist, S.cand, S.warp_tot, S.T);
    __syncthreads();
    if (tid == 0) S.row = next_row(fail_ctr, fail_rows);
    __syncthreads();
  }

  // every MMA issued here has completed before the tensor memory is freed
  if (warp == 4) {
    if (lane == 0) mma_commit(&S.fin);
    __syncwarp();
    mbar_wait_own(&S.fin, 0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
  if (tid == 0 && S.abort) flag_error(err, DSA_ERR_TIMEOUT);
}

int sm_count_fb() {
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

}  // namespace

int sel_fallback_grid(int num_q) { return std::max(1, std::min(num_q, sm_count_fb())); }

cudaError_t launch_sel_fallback(const QueryBatch& qb, const CacheMap& cm, const dsa_indexer_inputs& ix, int k,
                                int32_t* idx, float* slots, int64_t ld, int grid, uint32_t* fail_ctr,
                                const uint32_t* fail_rows, int* err, cudaStream_t stream) {
  CUtensorMap tm_q, tm_k;
  if (!make_tmap_rows128(&tm_q, ix.q, (uint64_t)qb.num_q * kHI, 128, kHI)) return cudaErrorInvalidValue;
  if (!make_tmap_rows128(&tm_k, ix.k, (uint64_t)cm.num_rows, 128, 64)) return cudaErrorInvalidValue;
  cudaError_t e =
      cudaFuncSetAttribute(sel_fallback_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc);
  if (e != cudaSuccess) return e;
  return launch_pdl(sel_fallback_kernel, dim3(grid), dim3(kFbThreads), kSmemAlloc, stream, tm_q, tm_k, qb, cm,
                    ix.q_scale, ix.w, ix.k_scale, k, idx, slots, ld, fail_ctr, fail_rows, err);
}

}  // namespace dsa
