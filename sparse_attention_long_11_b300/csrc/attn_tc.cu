// Sparse MQA attention on the 5th-generation tensor cores (tcgen05 + TMEM)
// for the DeepSeek-V3.2 latent shape: 128 query heads share one 576-wide bf16
// KV row per token (512 latent + 64 rope dims), the value is the first 512
// dims, and each query attends only to its selected positions (DeepSeek-V3.2
// summary card, "How DSA Works": full attention only on the selected tokens;
// news article on DeepSeek-V3.2, sparse-attention section: MQA / MLA on the
// sparse set).
//
// Design (B300: 148 SMs, 512 TMEM columns x 128 lanes per SM, 227 KB smem):
//   * The fp32 output of one query (128 heads x 512) fills a whole TMEM, so a
//     query runs on a CLUSTER OF TWO CTAs.  CTA c owns value dims
//     [256c, 256c+256): its TMEM holds O_c (256 columns) and two S buffers.
//   * The score contraction is split by dims: CTA c contracts its 256 latent
//     dims plus half of the 64 rope dims (288 of 576), so every KV byte is
//     gathered exactly once per query, by exactly one CTA.  The two partial
//     score tiles are exchanged through distributed shared memory and summed
//     (the same fp32 sum in both CTAs), so both run an identical online
//     softmax and scale their half of O consistently.
//   * Tiles of 64 selected keys.  Heads are the MMA's M (=128); per tile each
//     CTA issues 18 MMAs 128x64x16 for S and 4 MMAs 128x256x16 for P.V, with
//     V read MN-major straight out of the gathered K-major tile.
//   * Warp roles per CTA: warps 0-3 softmax/epilogue (thread = head = TMEM
//     lane), warps 4-7 gather (two groups of 64 threads alternate tiles,
//     16-byte cp.async per chunk, one row per thread), warp 8 TMEM owner and
//     MMA issuer.  Persistent: cluster j handles queries j, j+C, ...
//   * Lazy rescaling: the running max used for the exponent only moves when
//     a tile's max exceeds it by more than 8 (a factor 256), so O in TMEM is
//     rarely rewritten.
//   * Every wait is bounded; on expiry the CTA raises an abort flag, all roles
//     drain, the device error word reports DSA_ERR_TIMEOUT.
#include <algorithm>

#include "launch.h"
#include "tc.cuh"

namespace dsa {
namespace {
using namespace tc;

constexpr int kH = 128, kDqk = 576, kDv = 512;
constexpr int kNK = 64;                                   // keys per tile
constexpr uint32_t kQSlotBytes = 128 * 128;               // 128 heads x 128 B
constexpr uint32_t kKVSlotBytes = kNK * 128;              // 64 keys x 128 B
constexpr uint32_t kQBytes = 5 * kQSlotBytes;             // slots 0-3 latent, 4 rope (half used)
constexpr uint32_t kKVStageBytes = 5 * kKVSlotBytes;
constexpr uint32_t kXBytes = kH * kNK * 4;                // partial scores from the peer
constexpr uint32_t kPBytes = kH * 128;                    // 128 x 64 bf16 probabilities
constexpr uint32_t kOffKV = kQBytes;
constexpr uint32_t kOffX = kOffKV + 2 * kKVStageBytes;
constexpr uint32_t kOffP = kOffX + kXBytes;
constexpr uint32_t kSmemBytes = kOffP + kPBytes;          // 208 KB
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;        // + alignment slack
constexpr int kThreads = 288;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0, kTmemS = 256;              // S buffer b at kTmemS + 64 b
constexpr float kLn2 = 0.69314718055994530942f;

struct Bars {
  uint64_t kv_full[2], kv_empty[2], s_full[2], s_empty[2];
  uint64_t q_full, q_empty, p_full, pv_done, o_empty, x_full, x_empty, fin;
  uint32_t tmem_base;
  int abort;
};

// Tiles to process for one query: up to the last tile holding a valid entry
// (0 <= s <= pos).  Executed by a full warp; every role computes it the same way.
__device__ __forceinline__ int count_tiles(const int32_t* row, int k, int pos) {
  int last = -1;
  for (int j = threadIdx.x & 31; j < k; j += 32) {
    const int s = __ldg(row + j);
    if (s >= 0 && s <= pos) last = j;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
  return last < 0 ? 0 : last / kNK + 1;
}

__device__ __forceinline__ bool wait_fin(uint64_t* bar) {   // bounded, ignores the abort flag
  const uint32_t a = smem_u32(bar);
  const long long t0 = clock64();
  while (!mbar_try_wait(a, 0))
    if (clock64() - t0 > kWaitLimitCycles) return false;
  return true;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
attn_tc_kernel(QueryBatch qb, CacheMap cm, const __nv_bfloat16* __restrict__ q,
               const __nv_bfloat16* __restrict__ kv, const int32_t* __restrict__ idx, int k, float scale_log2,
               __nv_bfloat16* __restrict__ out, float* __restrict__ lse, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Bars B;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t crank = cluster_ctarank(), peer = crank ^ 1u;
  const int cluster = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  volatile int* abort = &B.abort;

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&B.kv_full[s], 64);
      mbar_init(&B.kv_empty[s], 1);
      mbar_init(&B.s_full[s], 1);
      mbar_init(&B.s_empty[s], 128);
    }
    mbar_init(&B.q_full, 128);
    mbar_init(&B.q_empty, 1);
    mbar_init(&B.p_full, 128);
    mbar_init(&B.pv_done, 1);
    mbar_init(&B.o_empty, 128);
    mbar_init(&B.x_full, 128);
    mbar_init(&B.x_empty, 128);
    mbar_init(&B.fin, 1);
    B.abort = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(&B.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // the peer's barriers exist before anyone arrives on them remotely
  tc_fence_after();
  const uint32_t tmem = B.tmem_base;
  const uint32_t sQ = smem_u32(sm), sKV = smem_u32(sm + kOffKV), sP = smem_u32(sm + kOffP);

  if (warp < 4) {
    // ------------------------------------------------------------ softmax / epilogue
    const int h = tid;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const uint32_t x_peer = mapa(smem_u32(sm + kOffX), peer);
    const uint32_t x_full_peer = mapa(smem_u32(&B.x_full), peer);
    const uint32_t x_empty_peer = mapa(smem_u32(&B.x_empty), peer);
    const float4* X4 = reinterpret_cast<const float4*>(sm + kOffX);
    uint32_t g = 0;
    for (int i = cluster; i < qb.num_q && !*abort; i += ncl) {
      const int pos = __ldg(qb.q_pos + i);
      const bool qok = pos >= 0 && pos < qb.max_kv;
      const int32_t* irow = idx + (int64_t)i * k;
      const int nt = qok ? count_tiles(irow, k, pos) : 0;
      __nv_bfloat16* orow = out + ((int64_t)i * kH + h) * kDv + crank * 256;
      if (nt == 0) {
        uint4* o4 = reinterpret_cast<uint4*>(orow);
#pragma unroll 4
        for (int c = 0; c < 32; ++c) o4[c] = make_uint4(0, 0, 0, 0);
        if (crank == 0) lse[(int64_t)i * kH + h] = -INFINITY;
        if (!qok && h == 0 && crank == 0) flag_error(err, DSA_ERR_BOUNDS);
        continue;
      }
      float m_use = -INFINITY, l = 0.f;
      bool ok = true;
      for (int t = 0; t < nt; ++t, ++g) {
        const int b = g & 1;
        const int e0 = t * kNK + lane, e1 = e0 + 32;
        const int s0 = e0 < k ? __ldg(irow + e0) : -1, s1 = e1 < k ? __ldg(irow + e1) : -1;
        const uint32_t v_lo = __ballot_sync(0xffffffffu, s0 >= 0 && s0 <= pos);
        const uint32_t v_hi = __ballot_sync(0xffffffffu, s1 >= 0 && s1 <= pos);

        if (!(ok = mbar_wait(&B.s_full[b], (g >> 1) & 1, abort))) break;
        tc_fence_after();
        float s[64];
        {
          uint32_t r[4][16];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld16(tmem + lane_base + kTmemS + b * 64 + c * 16, r[c]);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int j = 0; j < 16; ++j) s[c * 16 + j] = __uint_as_float(r[c][j]);
        }
        tc_fence_before();
        mbar_arrive(&B.s_empty[b]);

        // exchange partial scores with the peer CTA
        if (!(ok = mbar_wait<true>(&B.x_empty, (g & 1) ^ 1, abort))) break;
#pragma unroll
        for (int jq = 0; jq < 16; ++jq)
          st_cluster_v4(x_peer + (uint32_t)(jq * 128 + h) * 16u,
                        make_float4(s[4 * jq], s[4 * jq + 1], s[4 * jq + 2], s[4 * jq + 3]));
        mbar_arrive_remote(x_full_peer);
        if (!(ok = mbar_wait<true>(&B.x_full, g & 1, abort))) break;
#pragma unroll
        for (int jq = 0; jq < 16; ++jq) {
          const float4 v = X4[jq * 128 + h];
          s[4 * jq] += v.x; s[4 * jq + 1] += v.y; s[4 * jq + 2] += v.z; s[4 * jq + 3] += v.w;
        }
        mbar_arrive_remote(x_empty_peer);

        // online softmax in base 2
        float mt = -INFINITY;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const bool valid = ((j < 32 ? v_lo >> j : v_hi >> (j - 32)) & 1u) != 0;
          s[j] = valid ? s[j] * scale_log2 : -INFINITY;
          mt = fmaxf(mt, s[j]);
        }
        float alpha = 1.f;
        bool rescale = false;
        if (mt > m_use + 8.f) {
          alpha = exp2f(m_use - mt);
          m_use = mt;
          rescale = true;
        }
        uint32_t pk[32];
        float psum = 0.f;
#pragma unroll
        for (int j = 0; j < 64; j += 2) {
          const float p0 = m_use == -INFINITY ? 0.f : exp2f(s[j] - m_use);
          const float p1 = m_use == -INFINITY ? 0.f : exp2f(s[j + 1] - m_use);
          const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
          psum += __low2float(pb) + __high2float(pb);
          pk[j / 2] = *reinterpret_cast<const uint32_t*>(&pb);
        }
        l = l * alpha + psum;

        // P.V of the previous tile must be done before P and O are touched
        if (!(ok = mbar_wait(&B.pv_done, (g & 1) ^ 1, abort))) break;
        tc_fence_after();
        if (rescale && t > 0) {
#pragma unroll 1
          for (int c = 0; c < 256; c += 16) {
            uint32_t r[16];
            tmem_ld16(tmem + lane_base + kTmemO + c, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
            tmem_st16(tmem + lane_base + kTmemO + c, r);
          }
          tmem_st_wait();
        }
        uint8_t* prow = sm + kOffP;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
          *reinterpret_cast<uint4*>(prow + sw128_offset(h, cc)) =
              make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&B.p_full);
      }
      if (!ok) break;
      // epilogue: O row of this head, normalised, bf16
      if (!mbar_wait(&B.pv_done, (g - 1) & 1, abort)) break;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint4* o4 = reinterpret_cast<uint4*>(orow);
#pragma unroll 1
      for (int c = 0; c < 256; c += 16) {
        uint32_t r[16];
        tmem_ld16(tmem + lane_base + kTmemO + c, r);
        tmem_ld_wait();
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(r[2 * j]) * inv,
                                                         __uint_as_float(r[2 * j + 1]) * inv);
          w[j] = *reinterpret_cast<const uint32_t*>(&v);
        }
        o4[c / 8] = make_uint4(w[0], w[1], w[2], w[3]);
        o4[c / 8 + 1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
      if (crank == 0) lse[(int64_t)i * kH + h] = l > 0.f ? (m_use + log2f(l)) * kLn2 : -INFINITY;
      tc_fence_before();
      mbar_arrive(&B.o_empty);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ gather (cp.async)
    const int grp = (tid - 128) >> 6, p = (tid - 128) & 63;
    uint32_t g = 0, qv = 0;
    for (int i = cluster; i < qb.num_q && !*abort; i += ncl) {
      const int pos = __ldg(qb.q_pos + i);
      if (pos < 0 || pos >= qb.max_kv) continue;
      const int seq = __ldg(qb.q_seq + i);
      const int32_t* irow = idx + (int64_t)i * k;
      const int nt = count_tiles(irow, k, pos);
      if (nt == 0) continue;
      if (!mbar_wait(&B.q_empty, (qv & 1) ^ 1, abort)) break;
      {
        const int h = p + 64 * grp;
        const __nv_bfloat16* qrow = q + ((int64_t)i * kH + h) * kDqk;
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int cc = 0; cc < 8; ++cc)
            cp_async16(sQ + a * kQSlotBytes + sw128_offset(h, cc), qrow + crank * 256 + a * 64 + cc * 8, 16);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int c8 = 4 * crank + cc;
          cp_async16(sQ + 4 * kQSlotBytes + sw128_offset(h, c8), qrow + 512 + c8 * 8, 16);
        }
        cp_async_commit();
        cp_async_wait_all();
        fence_proxy_async_smem();
        mbar_arrive(&B.q_full);
      }
      bool ok = true;
      for (int t = 0; t < nt; ++t, ++g) {
        if ((int)(g & 1) != grp) continue;
        if (!(ok = mbar_wait(&B.kv_empty[grp], ((g >> 1) & 1) ^ 1, abort))) break;
        const int e = t * kNK + p;
        int64_t row = -1;
        if (e < k) {
          const int s = __ldg(irow + e);
          if (s >= 0 && s <= pos) row = cache_row(cm, seq, s, err);
          else if (s != -1) flag_error(err, DSA_ERR_BOUNDS);
        }
        const uint32_t sb = sKV + grp * kKVStageBytes;
        const __nv_bfloat16* src = row >= 0 ? kv + row * kDqk : kv;
        const uint32_t nb = row >= 0 ? 16u : 0u;
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int cc = 0; cc < 8; ++cc)
            cp_async16(sb + a * kKVSlotBytes + sw128_offset(p, cc), src + crank * 256 + a * 64 + cc * 8, nb);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int c8 = 4 * crank + cc;
          cp_async16(sb + 4 * kKVSlotBytes + sw128_offset(p, c8), src + 512 + c8 * 8, nb);
        }
        cp_async_commit();
        cp_async_wait_all();
        fence_proxy_async_smem();
        mbar_arrive(&B.kv_full[grp]);
      }
      if (!ok) break;
      ++qv;
    }
  } else {
    // ------------------------------------------------------------ MMA issue (warp 8, lane 0 issues)
    const uint32_t id_s = idesc_bf16(128, kNK, false);
    const uint32_t id_pv = idesc_bf16(128, 256, true);
    uint32_t g = 0, qv = 0;
    auto issue_pv = [&](uint32_t gp, int tp) -> bool {
      if (!mbar_wait(&B.p_full, gp & 1, abort)) return false;
      if (tp == 0 && !mbar_wait(&B.o_empty, (qv & 1) ^ 1, abort)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t skv = sKV + (gp & 1) * kKVStageBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16(tmem + kTmemO, sdesc(sP + kk * 32, 16, 1024), sdesc(skv + kk * 2048, kKVSlotBytes, 1024), id_pv,
                   (tp > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&B.pv_done);
        mma_commit(&B.kv_empty[gp & 1]);
      }
      __syncwarp();
      return true;
    };
    for (int i = cluster; i < qb.num_q && !*abort; i += ncl) {
      const int pos = __ldg(qb.q_pos + i);
      if (pos < 0 || pos >= qb.max_kv) continue;
      const int nt = count_tiles(idx + (int64_t)i * k, k, pos);
      if (nt == 0) continue;
      if (!mbar_wait(&B.q_full, qv & 1, abort)) break;
      bool ok = true;
      for (int t = 0; t < nt; ++t, ++g) {
        const uint32_t st = g & 1;
        if (!(ok = mbar_wait(&B.kv_full[st], (g >> 1) & 1, abort))) break;
        if (!(ok = mbar_wait(&B.s_empty[st], ((g >> 1) & 1) ^ 1, abort))) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t dS = tmem + kTmemS + 64 * st;
          const uint32_t skv = sKV + st * kKVStageBytes;
          uint32_t n = 0;
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk, ++n)
              mma_bf16(dS, sdesc(sQ + a * kQSlotBytes + kk * 32, 16, 1024),
                       sdesc(skv + a * kKVSlotBytes + kk * 32, 16, 1024), id_s, n > 0 ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const uint32_t ko = (2 * crank + kk) * 32;
            mma_bf16(dS, sdesc(sQ + 4 * kQSlotBytes + ko, 16, 1024), sdesc(skv + 4 * kKVSlotBytes + ko, 16, 1024),
                     id_s, 1u);
          }
          mma_commit(&B.s_full[st]);
          if (t == nt - 1) mma_commit(&B.q_empty);
        }
        __syncwarp();
        if (t > 0 && !(ok = issue_pv(g - 1, t - 1))) break;
      }
      if (!ok || !issue_pv(g - 1, nt - 1)) break;
      ++qv;
    }
    if (lane == 0) mma_commit(&B.fin);
    __syncwarp();
    wait_fin(&B.fin);   // every MMA issued by this CTA has completed
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();       // the peer no longer reads or writes our shared memory
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (tid == 0 && B.abort) flag_error(err, DSA_ERR_TIMEOUT);
}

int sm_count() {
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

cudaError_t launch_attn_tc(const QueryBatch& qb, const CacheMap& cm, const dsa_attn_inputs& at, const int32_t* idx,
                           int k, void* out, float* lse, int* err, cudaStream_t stream) {
  const int ncl = std::min(qb.num_q, sm_count() / 2);
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc);
  if (e != cudaSuccess) return e;
  const float scale_log2 = (float)((double)at.softmax_scale * 1.4426950408889634);
  attn_tc_kernel<<<2 * ncl, kThreads, kSmemAlloc, stream>>>(
      qb, cm, static_cast<const __nv_bfloat16*>(at.q), static_cast<const __nv_bfloat16*>(at.kv), idx, k, scale_log2,
      static_cast<__nv_bfloat16*>(out), lse, err);
  return cudaGetLastError();
}

}  // namespace dsa
