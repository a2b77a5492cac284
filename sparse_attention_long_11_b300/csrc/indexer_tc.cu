// Lightning indexer on the 5th-generation tensor cores: an FP8 (e4m3) GEMM
// with the ReLU, weighted head sum and scales fused into the epilogue
// (DeepSeek-V3.2 summary card, "How DSA Works": the lightning indexer scores
// every key of a query cheaply in FP8; news article on DeepSeek-V3.2,
// sparse-attention section: a few low-precision heads on every token pair).
//
//   I[t,s] = sk[s] * sum_j (w[t,j] sq[t,j]) * ReLU(<q8[t,j,:], k8[s,:]>)
// (the positive scales move out of the ReLU).
//
// Layout: keys on M (128 TMEM lanes), (4 queries x 64 heads) on N = 256, so
// the head sum of one (key, query) pair lies in one thread's TMEM row and
// needs no cross-thread reduction.  K = 128 (4 MMAs of K = 32).  D is double
// buffered (2 x 256 of the 512 TMEM columns) so the epilogue of tile g
// overlaps the MMAs of tile g+1.
//
// Work item = (group of 4 consecutive query rows, key split).  When the four
// rows belong to one sequence (prefill chunks) they share every key tile:
// one pass with N = 256.  Otherwise (decode batches, chunk boundaries) each
// query makes its own pass over its own sequence with N = 64.  Key tiles are
// loaded by TMA: 2 boxes of 64 rows, so paged caches whose block size is a
// multiple of 64 are read block by block.
//
// Warps: 0 = TMA producer, 1 = TMEM owner + MMA issuer, 2 = setup,
// 4..11 = epilogue (warp 4+e reads TMEM lane quadrant e%4 and handles
// queries 2(e/4), 2(e/4)+1).  All waits are bounded (see tc.cuh).
#include <algorithm>

#include "launch.h"
#include "tc.cuh"
#include "tmap.h"

namespace dsa {
namespace {
using namespace tc;

constexpr int kQG = 4;                          // queries per group
constexpr int kHI = 64, kDI = 128;
constexpr int kKT = 128;                        // keys per tile
constexpr int kStagesA = 6;
constexpr uint32_t kBBytes = kQG * kHI * 128;   // 32 KB
constexpr uint32_t kABytes = kKT * 128;         // 16 KB
constexpr uint32_t kOffA = kBBytes;
constexpr uint32_t kSmemBytes = kOffA + kStagesA * kABytes;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;
constexpr int kThreads = 384;
constexpr int kEpiThreads = 256;

struct __align__(16) Shared {
  uint64_t a_full[kStagesA], a_empty[kStagesA], d_full[2], d_empty[2], b_full, fin;
  float wq[kQG][kHI];           // w * q_scale
  int seq[kQG], pos[kQG], active[kQG];
  int npass, uniform;
  int pass_q[kQG], pass_seq[kQG], pass_T[kQG], pass_maxpos[kQG];
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ bool wait_plain(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const long long t0 = clock64();
  while (!mbar_try_wait(a, parity))
    if (clock64() - t0 > kWaitLimitCycles) return false;
  return true;
}

__global__ void __launch_bounds__(kThreads, 1)
indexer_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  QueryBatch qb, CacheMap cm, const float* __restrict__ q_scale, const float* __restrict__ w,
                  const float* __restrict__ k_scale, float* __restrict__ scores, int64_t ld, int splits,
                  int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Shared S;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gi = blockIdx.x, z = blockIdx.y;
  volatile int* abort = &S.abort;
  const uint32_t sB = smem_u32(sm), sA = smem_u32(sm + kOffA);

  if (tid == 0) {
    for (int s = 0; s < kStagesA; ++s) {
      mbar_init(&S.a_full[s], 1);
      mbar_init(&S.a_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.d_full[b], 1);
      mbar_init(&S.d_empty[b], kEpiThreads);
    }
    mbar_init(&S.b_full, 1);
    mbar_init(&S.fin, 1);
    S.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == 2) {
    // group description and folded weights
    for (int e = lane; e < kQG * kHI; e += 32) {
      const int qq = e / kHI, j = e % kHI;
      const int r = gi * kQG + qq;
      float v = 0.f;
      if (r < qb.num_q) v = __ldg(w + (int64_t)r * kHI + j) * __ldg(q_scale + (int64_t)r * kHI + j);
      S.wq[qq][j] = v;
    }
    if (lane == 0) {
      int first_seq = -1, same = 1, nact = 0;
      for (int qq = 0; qq < kQG; ++qq) {
        const int r = gi * kQG + qq;
        int act = 0, sq = 0, ps = -1;
        if (r < qb.num_q) {
          sq = __ldg(qb.q_seq + r);
          ps = __ldg(qb.q_pos + r);
          act = ps >= 0 && ps < qb.max_kv && sq >= 0 && sq < cm.num_seqs;
          if (!act) flag_error(err, DSA_ERR_BOUNDS);
        }
        S.seq[qq] = sq;
        S.pos[qq] = ps;
        S.active[qq] = act;
        if (act) {
          if (first_seq < 0) first_seq = sq;
          else if (sq != first_seq) same = 0;
          ++nact;
        }
      }
      S.uniform = same && nact > 0;
      int np = 0;
      if (S.uniform) {
        int mp = -1;
        for (int qq = 0; qq < kQG; ++qq)
          if (S.active[qq]) mp = max(mp, S.pos[qq]);
        S.pass_q[0] = -1;
        S.pass_seq[0] = first_seq;
        S.pass_maxpos[0] = mp;
        S.pass_T[0] = mp / kKT + 1;
        np = 1;
      } else {
        for (int qq = 0; qq < kQG; ++qq) {
          if (!S.active[qq]) continue;
          S.pass_q[np] = qq;
          S.pass_seq[np] = S.seq[qq];
          S.pass_maxpos[np] = S.pos[qq];
          S.pass_T[np] = S.pos[qq] / kKT + 1;
          ++np;
        }
      }
      S.npass = np;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  const int npass = S.npass;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && npass > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      mbar_arrive_expect_tx(&S.b_full, kBBytes);
      tma_load_2d(sB, &tm_q, 0, gi * kQG * kHI, &S.b_full);
      uint32_t g = 0;
      for (int p = 0; p < npass && !*abort; ++p) {
        const int T = S.pass_T[p], seq = S.pass_seq[p], mp = S.pass_maxpos[p];
        const int t0 = (int)((int64_t)T * z / splits), t1 = (int)((int64_t)T * (z + 1) / splits);
        for (int t = t0; t < t1; ++t, ++g) {
          const int st = g % kStagesA;
          if (!mbar_wait(&S.a_empty[st], ((g / kStagesA) & 1) ^ 1, abort)) break;
          int64_t rows[2];
          uint32_t bytes = 0;
          for (int hh = 0; hh < 2; ++hh) {
            const int sh = t * kKT + 64 * hh;
            rows[hh] = -1;
            if (sh > mp) continue;
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
            if (rows[hh] >= 0)
              tma_load_2d(sA + st * kABytes + hh * 8192, &tm_k, 0, (int32_t)rows[hh], &S.a_full[st]);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (npass > 0 && mbar_wait(&S.b_full, 0, abort)) {
      uint32_t g = 0;
      for (int p = 0; p < npass && !*abort; ++p) {
        const bool uni = S.uniform != 0;
        const uint32_t idesc = idesc_e4m3(128, uni ? 256 : 64);
        const uint32_t boff = uni ? 0u : (uint32_t)S.pass_q[p] * (kHI * 128);
        const int T = S.pass_T[p];
        const int t0 = (int)((int64_t)T * z / splits), t1 = (int)((int64_t)T * (z + 1) / splits);
        bool ok = true;
        for (int t = t0; t < t1; ++t, ++g) {
          const int st = g % kStagesA, b = g & 1;
          if (!(ok = mbar_wait(&S.a_full[st], (g / kStagesA) & 1, abort))) break;
          if (!(ok = mbar_wait(&S.d_empty[b], ((g >> 1) & 1) ^ 1, abort))) break;
          tc_fence_after();
          if (lane == 0) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_e4m3(tmem + 256 * b, sdesc(sA + st * kABytes + kk * 32, 16, 1024),
                       sdesc(sB + boff + kk * 32, 16, 1024), idesc, kk > 0 ? 1u : 0u);
            mma_commit(&S.a_empty[st]);
            mma_commit(&S.d_full[b]);
          }
          __syncwarp();
        }
        if (!ok) break;
      }
    }
    if (lane == 0) mma_commit(&S.fin);
    __syncwarp();
    wait_plain(&S.fin, 0);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int e = warp - 4, qd = e & 3, qh = e >> 2;
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    uint32_t g = 0;
    for (int p = 0; p < npass && !*abort; ++p) {
      const bool uni = S.uniform != 0;
      const int seq = S.pass_seq[p];
      const int T = S.pass_T[p];
      const int t0 = (int)((int64_t)T * z / splits), t1 = (int)((int64_t)T * (z + 1) / splits);
      bool ok = true;
      for (int t = t0; t < t1; ++t, ++g) {
        const int b = g & 1;
        if (!(ok = mbar_wait(&S.d_full[b], (g >> 1) & 1, abort))) break;
        tc_fence_after();
        const int s = t * kKT + qd * 32 + lane;
        float sk = 0.f;
        bool key_ok = s <= S.pass_maxpos[p];
        if (key_ok) {
          const int64_t row = cache_row(cm, seq, s, err);
          key_ok = row >= 0;
          if (key_ok) sk = __ldg(k_scale + row);
        }
        for (int u = 0; u < 2; ++u) {
          const int qq = uni ? 2 * qh + u : S.pass_q[p];
          if (!uni && (qh != 0 || u != 0)) break;
          uint32_t r[4][16];
          const uint32_t col = 256 * b + (uni ? qq * 64 : 0);
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld16(tmem + lane_base + col + c * 16, r[c]);
          tmem_ld_wait();
          const float4* wq4 = reinterpret_cast<const float4*>(S.wq[qq]);
          float a0 = 0.f, a1 = 0.f;
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int j4 = 0; j4 < 4; ++j4) {
              const float4 wv = wq4[c * 4 + j4];
              a0 = fmaf(wv.x, fmaxf(__uint_as_float(r[c][4 * j4 + 0]), 0.f), a0);
              a1 = fmaf(wv.y, fmaxf(__uint_as_float(r[c][4 * j4 + 1]), 0.f), a1);
              a0 = fmaf(wv.z, fmaxf(__uint_as_float(r[c][4 * j4 + 2]), 0.f), a0);
              a1 = fmaf(wv.w, fmaxf(__uint_as_float(r[c][4 * j4 + 3]), 0.f), a1);
            }
          const int row_q = gi * kQG + qq;
          if (s < qb.max_kv && row_q < qb.num_q) {
            const bool live = S.active[qq] && key_ok && s <= S.pos[qq];
            scores[(int64_t)row_q * ld + s] = live ? (a0 + a1) * sk : -INFINITY;
          }
        }
        tc_fence_before();
        mbar_arrive(&S.d_empty[b]);
      }
      if (!ok) break;
    }
    // the last split also writes -inf from the end of the scanned tiles to max_kv
    if (z == splits - 1) {
      const int et = tid - 128;
      for (int qq = 0; qq < kQG; ++qq) {
        const int row_q = gi * kQG + qq;
        if (row_q >= qb.num_q) break;
        int from = 0;
        if (S.active[qq]) {
          int T = 0;
          for (int p = 0; p < npass; ++p)
            if (S.uniform || S.pass_q[p] == qq) T = S.pass_T[p];
          from = T * kKT;
        }
        for (int s = from + et; s < qb.max_kv; s += kEpiThreads) scores[(int64_t)row_q * ld + s] = -INFINITY;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (tid == 0 && S.abort) flag_error(err, DSA_ERR_TIMEOUT);
}

int sm_count_here() {
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

bool indexer_tc_supported(const CacheMap& cm, const dsa_indexer_inputs& ix) {
  if (ix.dtype != DSA_FP8_E4M3 || ix.heads != kHI || ix.dim != kDI) return false;
  if (cm.block_size != 0 && cm.block_size % 64 != 0) return false;
  return true;
}

cudaError_t launch_indexer_tc(const QueryBatch& qb, const CacheMap& cm, const dsa_indexer_inputs& ix, float* scores,
                              int64_t ld, int* err, cudaStream_t stream) {
  CUtensorMap tm_q, tm_k;
  if (!make_tmap_rows128(&tm_q, ix.q, (uint64_t)qb.num_q * kHI, 128, kQG * kHI)) return cudaErrorInvalidValue;
  if (!make_tmap_rows128(&tm_k, ix.k, (uint64_t)cm.num_rows, 128, 64)) return cudaErrorInvalidValue;
  const int groups = (qb.num_q + kQG - 1) / kQG;
  const int tiles = (qb.max_kv + kKT - 1) / kKT;
  int splits = (2 * sm_count_here() + groups - 1) / groups;
  splits = std::max(1, std::min(splits, std::max(1, tiles / 4)));
  cudaError_t e = cudaFuncSetAttribute(indexer_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc);
  if (e != cudaSuccess) return e;
  indexer_tc_kernel<<<dim3(groups, splits), kThreads, kSmemAlloc, stream>>>(tm_q, tm_k, qb, cm, ix.q_scale, ix.w,
                                                                             ix.k_scale, scores, ld, splits, err);
  return cudaGetLastError();
}

}  // namespace dsa
