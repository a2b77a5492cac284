// Sparse MQA attention on the 5th-generation tensor cores (tcgen05 + TMEM)
// for the DeepSeek-V3.2 latent shape: 128 query heads share one 576-wide bf16
// KV row per token (512 latent + 64 rope dims), the value is the first 512
// dims, and each query attends only to its selected positions (DeepSeek-V3.2
// summary card, "How DSA Works": full attention only on the selected tokens;
// news article on DeepSeek-V3.2, sparse-attention section: MQA / MLA on the
// sparse set).
//
// Design (B300: 148 SMs, TMEM of 512 columns x 128 lanes per SM, 227 KB smem):
//   * The fp32 output of one query (128 heads x 512) fills a whole TMEM, so a
//     query runs on a CLUSTER OF TWO CTAs.  CTA c owns value dims
//     [256c, 256c+256): its TMEM holds O_c (256 columns), two S buffers
//     (2 x 64) and the query's 256 latent dims of this CTA (128 columns of
//     packed bf16), the A operand of the latent score MMAs.  Keeping Q out
//     of shared memory frees room for three KV stages and removes 64 KB of
//     operand reads per tile from the shared-memory bandwidth.
//   * The score contraction is split by dims: CTA c contracts latent dims
//     [256c, 256c+256) and rope dims [512+32c, 512+32c+32) (288 of 576), so
//     every KV byte is gathered exactly once per query, by one CTA.  The two
//     fp32 partial score tiles are exchanged through distributed shared
//     memory and summed in the same order in both CTAs, so both run the same
//     online softmax and scale their half of O consistently.  DSMEM moves
//     only ~15-19 B/clk per SM on B300, so the exchange runs on its own warps
//     with double-buffered receive tiles and overlaps the softmax and MMAs.
//   * Tiles of 64 selected keys, gathered with coalesced 16-byte cp.async
//     (a warp moves 512 contiguous bytes of one row per instruction) into
//     128B-swizzled latent slots and a 64B-swizzled rope half.  (TMA
//     tile::gather4 measured ~64 clk per 4-row instruction on B300, slower
//     than this path.)  Heads are the MMA's M (=128); per tile each CTA issues 18 MMAs
//     128x64x16 for S and 4 MMAs 128x256x16 for P.V, with V read MN-major
//     straight out of the gathered K-major latent slots.
//   * Warp roles per CTA: 0-3 softmax/epilogue (thread = head = TMEM lane),
//     4-7 score exchange, 8-13 gather (three groups of two warps, group j
//     fills KV stage j with the tiles g = j mod 3; at each query warps 8-11
//     write Q's latent part into TMEM and warp 8 loads the rope part with
//     TMA), 14 TMEM owner + MMA issuer.
//     Persistent: cluster j handles queries j, j+C, ...
//   * Lazy rescaling: the running max used for the exponent only moves when
//     a tile's max exceeds it by more than 8 (a factor 256).
//   * Every wait is bounded; on expiry the CTA raises an abort flag, all roles
//     drain, the device error word reports DSA_ERR_TIMEOUT.
#include <algorithm>

#include "launch.h"
#include "tc.cuh"
#include "tmap.h"

namespace dsa {
namespace {
using namespace tc;

constexpr int kH = 128, kDqk = 576, kDv = 512;
constexpr int kNK = 64;                                    // keys per tile
constexpr uint32_t kQRopeBytes = 128 * 64;                 // rope half: 128 heads x 64 B (SW64)
constexpr uint32_t kKVSlotBytes = kNK * 128;               // 64 keys x 128 B
constexpr uint32_t kKVRopeBytes = kNK * 64;                // 64 keys x 64 B
constexpr uint32_t kKVStageBytes = 4 * kKVSlotBytes + kKVRopeBytes;   // 36 KB
constexpr uint32_t kXBytes = kH * kNK * 4;                 // one partial score tile from the peer
constexpr uint32_t kPBytes = kH * 128;                     // 128 x 64 bf16 probabilities (SW128)
constexpr int kStages = 3;
constexpr uint32_t kOffQRope = 0;
constexpr uint32_t kOffKV = kOffQRope + kQRopeBytes;       // 8 KB
constexpr uint32_t kOffX = kOffKV + kStages * kKVStageBytes;   // 116 KB
constexpr uint32_t kOffP = kOffX + 2 * kXBytes;            // 180 KB: P[0], P[1]
constexpr uint32_t kSmemBytes = kOffP + 2 * kPBytes;       // 212 KB (P double buffered)
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;         // + alignment slack
constexpr int kThreads = 480;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0, kTmemS = 256, kTmemQ = 384;  // S buffer b at kTmemS + 64 b
constexpr float kLn2 = 0.69314718055994530942f;

// Optional per-tile timeline of the first CTA (build with -DDSA_ATTN_TRACE):
// SM clock stamps per role (0 softmax, 1 exchange, 2 producer, 3 MMA), tile
// and event, read back with dsa_attn_trace_read().
#ifdef DSA_ATTN_TRACE
__device__ long long g_attn_trace[4][512][8];
#define ATTN_TRACE(role, tile, ev, cond)                                                   \
  do {                                                                                    \
    if ((cond) && blockIdx.x == 0 && (tile) < 512) g_attn_trace[role][tile][ev] = clock64(); \
  } while (0)
#else
#define ATTN_TRACE(role, tile, ev, cond) \
  do {                                   \
  } while (0)
#endif

struct Bars {
  uint64_t kv_full[kStages], kv_empty[kStages], s_full[2], s_empty[2], xf[2], xe[2];
  uint64_t p_full[2], pv_done[2];
  uint64_t q_full, q_empty, o_empty, fin;
  uint32_t tmem_base;
  int abort;
};

// Tiles to process for one query: up to the last tile holding a valid entry
// (0 <= s <= pos).  With prefix_valid (rows written by the top-k stage:
// ascending, valid entries first) that is ceil(min(k, pos+1) / 64) without
// reading the row; otherwise a full warp scans it.  Every role computes it
// the same way.
__device__ __forceinline__ int count_tiles(const int32_t* row, int k, int pos, bool prefix_valid) {
  if (prefix_valid) return (min(k, pos + 1) + kNK - 1) / kNK;
  int last = -1;
#pragma unroll 8
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

// Own partial score row of this thread's head (64 fp32 from TMEM).
__device__ __forceinline__ void load_s(uint32_t taddr, float (&s)[64]) {
  uint32_t r[4][16];
#pragma unroll
  for (int c = 0; c < 4; ++c) tmem_ld16(taddr + c * 16, r[c]);
  tmem_ld_wait();
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int j = 0; j < 16; ++j) s[c * 16 + j] = __uint_as_float(r[c][j]);
}

struct QueryInfo {
  int pos, nt;
  bool ok;
};

__device__ __forceinline__ QueryInfo query_info(const QueryBatch& qb, const int32_t* idx, int k, int i,
                                                bool prefix_valid) {
  QueryInfo r;
  r.pos = __ldg(qb.q_pos + i);
  r.ok = r.pos >= 0 && r.pos < qb.max_kv;
  r.nt = r.ok ? count_tiles(idx + (int64_t)i * k, k, r.pos, prefix_valid) : 0;
  return r;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q_rope, const __nv_bfloat16* __restrict__ q,
               const __nv_bfloat16* __restrict__ kv, QueryBatch qb, CacheMap cm, const int32_t* __restrict__ idx, int k, int prefix_valid,
               float scale_log2, __nv_bfloat16* __restrict__ out, float* __restrict__ lse, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Bars B;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t crank = cluster_ctarank(), peer = crank ^ 1u;
  const int cluster = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  const bool pv = prefix_valid != 0;
  volatile int* abort = &B.abort;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&B.kv_full[s], 64);    // the 64 threads of one gather group
      mbar_init(&B.kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&B.s_full[s], 1);
      mbar_init(&B.s_empty[s], 256);   // the exchange warps and the softmax warps both read S
      mbar_init(&B.xf[s], 1);          // armed by our softmax thread 0; the peer's st.async credit the bytes
      mbar_init(&B.xe[s], 128);        // arrivals of the peer's softmax warps
    }
    mbar_init(&B.q_full, 129);       // 128 TMEM writers + the rope TMA (with its bytes)
    mbar_init(&B.q_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&B.p_full[s], 128);
      mbar_init(&B.pv_done[s], 1);
    }
    mbar_init(&B.o_empty, 128);
    mbar_init(&B.fin, 1);
    B.abort = 0;
    fence_mbar_init();
    mbar_arrive_expect_tx(&B.xf[0], kXBytes);   // arm the first phase of both receive tiles
    mbar_arrive_expect_tx(&B.xf[1], kXBytes);
  }
  if (warp == 14) {
    tmem_alloc(&B.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // the peer's barriers exist before anyone arrives on them remotely
  tc_fence_after();
  const uint32_t tmem = B.tmem_base;
  const uint32_t sQr = smem_u32(sm + kOffQRope), sKV = smem_u32(sm + kOffKV);
  const uint32_t sP = smem_u32(sm + kOffP);

  if (warp < 4) {
    // ------------------------------------------------------------ softmax / epilogue
    const int h = tid;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const uint32_t xe_peer[2] = {mapa(smem_u32(&B.xe[0]), peer), mapa(smem_u32(&B.xe[1]), peer)};
    uint32_t g = 0;
    for (int i = cluster; i < qb.num_q && !*abort; i += ncl) {
      const QueryInfo qi = query_info(qb, idx, k, i, pv);
      const int pos = qi.pos, nt = qi.nt;
      const int32_t* irow = idx + (int64_t)i * k;
      __nv_bfloat16* orow = out + ((int64_t)i * kH + h) * kDv + crank * 256;
      if (nt == 0) {
        uint4* o4 = reinterpret_cast<uint4*>(orow);
#pragma unroll 4
        for (int c = 0; c < 32; ++c) o4[c] = make_uint4(0, 0, 0, 0);
        if (crank == 0) lse[(int64_t)i * kH + h] = -INFINITY;
        if (!qi.ok && h == 0 && crank == 0) flag_error(err, DSA_ERR_BOUNDS);
        continue;
      }
      const int n_valid = min(k, pos + 1);
      float m_use = -INFINITY, l = 0.f;
      bool ok = true;
      for (int t = 0; t < nt; ++t, ++g) {
        const int b = g & 1;
        const uint32_t par = (g >> 1) & 1;
        int s0 = 0, s1 = 0;
        if (!pv) {   // loads issued early; their latency hides behind the waits below
          const int e0 = t * kNK + lane, e1 = e0 + 32;
          s0 = e0 < k ? __ldg(irow + e0) : -1;
          s1 = e1 < k ? __ldg(irow + e1) : -1;
        }
        ATTN_TRACE(0, g, 0, h == 0);
        if (!(ok = mbar_wait<true>(&B.xf[b], par, abort))) break;   // the peer's partial is in X[b]
        ATTN_TRACE(0, g, 1, h == 0);
        if (!(ok = mbar_wait(&B.s_full[b], par, abort))) break;
        ATTN_TRACE(0, g, 6, h == 0);
        tc_fence_after();
        float s[64];
        load_s(tmem + lane_base + kTmemS + b * 64, s);
        ATTN_TRACE(0, g, 7, h == 0);
        {
          const float4* X4 = reinterpret_cast<const float4*>(sm + kOffX + b * kXBytes);
#pragma unroll
          for (int jq = 0; jq < 16; ++jq) {
            const float4 v = X4[jq * 128 + h];
            // CTA 0's partial first, so both CTAs form the identical fp32 sum
            if (crank == 0) {
              s[4 * jq] += v.x; s[4 * jq + 1] += v.y; s[4 * jq + 2] += v.z; s[4 * jq + 3] += v.w;
            } else {
              s[4 * jq] = v.x + s[4 * jq]; s[4 * jq + 1] = v.y + s[4 * jq + 1];
              s[4 * jq + 2] = v.z + s[4 * jq + 2]; s[4 * jq + 3] = v.w + s[4 * jq + 3];
            }
          }
        }
        ATTN_TRACE(1, g, 4, h == 0 && s[0] != 12345.f);   // after the partial read (value dependency)
        tc_fence_before();
        mbar_arrive(&B.s_empty[b]);
        ATTN_TRACE(1, g, 5, h == 0);
        // X[b] consumed (the loads above have returned and their values are in
        // use): the peer may write its next tile there.  A release-ordered
        // remote arrive costs ~1.5k clk here; relaxed is enough.
        mbar_arrive_remote_relaxed(xe_peer[b]);
        if (h == 0) mbar_arrive_expect_tx(&B.xf[b], kXBytes);   // arm the next phase of this receive tile
        ATTN_TRACE(0, g, 2, h == 0);

        uint32_t v_lo, v_hi;
        if (pv) {
          const int rem = n_valid - t * kNK;   // the valid entries of this tile form a prefix
          v_lo = rem >= 32 ? 0xffffffffu : (rem <= 0 ? 0u : (1u << rem) - 1u);
          v_hi = rem >= 64 ? 0xffffffffu : (rem <= 32 ? 0u : (1u << (rem - 32)) - 1u);
        } else {
          v_lo = __ballot_sync(0xffffffffu, s0 >= 0 && s0 <= pos);
          v_hi = __ballot_sync(0xffffffffu, s1 >= 0 && s1 <= pos);
        }

        // online softmax in base 2: logits x = scale * log2(e) * S
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const bool valid = ((j < 32 ? v_lo >> j : v_hi >> (j - 32)) & 1u) != 0;
          s[j] = valid ? s[j] * scale_log2 : -INFINITY;
          m4[j & 3] = fmaxf(m4[j & 3], s[j]);
        }
        const float mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        float alpha = 1.f;
        bool rescale = false;
        if (mt > m_use + 8.f) {
          alpha = ex2_approx(m_use - mt);
          m_use = mt;
          rescale = true;
        }
        const float msub = m_use == -INFINITY ? 0.f : m_use;   // all p are 0 while nothing is valid
        uint32_t pk[32];
        float ps4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 64; j += 2) {
          const float p0 = ex2_approx(s[j] - msub);
          const float p1 = ex2_approx(s[j + 1] - msub);
          const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
          ps4[(j >> 1) & 3] += __low2float(pb) + __high2float(pb);
          pk[j / 2] = *reinterpret_cast<const uint32_t*>(&pb);
        }
        const float psum = (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
        l = l * alpha + psum;
        ATTN_TRACE(0, g, 3, h == 0);

        // P[b] is free once the P.V of tile g-2 is done; rescaling O also
        // needs the P.V of tile g-1 to be done
        if (!(ok = mbar_wait(&B.pv_done[b], par ^ 1, abort))) break;
        if (rescale && t > 0 && !(ok = mbar_wait(&B.pv_done[b ^ 1], ((g - 1) >> 1) & 1, abort))) break;
        ATTN_TRACE(0, g, 4, h == 0);
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
        uint8_t* prow = sm + kOffP + b * kPBytes;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
          *reinterpret_cast<uint4*>(prow + sw128_offset(h, cc)) =
              make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&B.p_full[b]);
        ATTN_TRACE(0, g, 5, h == 0);
      }
      if (!ok) break;
      // epilogue: O row of this head, normalised, bf16
      if (!mbar_wait(&B.pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, abort)) break;
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
    // ------------------------------------------------------------ score exchange
    const int h = ((warp & 3) << 5) | lane;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t x_peer = mapa(smem_u32(sm + kOffX), peer);
    const uint32_t xf_peer[2] = {mapa(smem_u32(&B.xf[0]), peer), mapa(smem_u32(&B.xf[1]), peer)};
    // (the peer arms its xf[b] with the tile's bytes; our st.async credit them)
    uint32_t g = 0;
    for (int i = cluster; i < qb.num_q && !*abort; i += ncl) {
      const QueryInfo qi = query_info(qb, idx, k, i, pv);
      bool ok = true;
      for (int t = 0; t < qi.nt; ++t, ++g) {
        const int b = g & 1;
        const uint32_t par = (g >> 1) & 1;
        ATTN_TRACE(1, g, 0, h == 0);
        if (!(ok = mbar_wait(&B.s_full[b], par, abort))) break;
        ATTN_TRACE(1, g, 1, h == 0);
        tc_fence_after();
        float s[64];
        load_s(tmem + lane_base + kTmemS + b * 64, s);
        tc_fence_before();
        mbar_arrive(&B.s_empty[b]);
        // the peer has consumed what we wrote into its X[b] two tiles ago
        if (!(ok = mbar_wait<true>(&B.xe[b], par ^ 1, abort))) break;
        ATTN_TRACE(1, g, 2, h == 0);
        const uint32_t dst = x_peer + b * kXBytes;
#pragma unroll
        for (int jq = 0; jq < 16; ++jq)
          st_async_v4(dst + (uint32_t)(jq * 128 + h) * 16u,
                      make_float4(s[4 * jq], s[4 * jq + 1], s[4 * jq + 2], s[4 * jq + 3]), xf_peer[b]);
        ATTN_TRACE(1, g, 3, h == 0);
      }
      if (!ok) break;
    }
  } else if (warp < 14) {
    // ------------------------------------------------------------ gather (cp.async) + Q (TMA)
    // Group grp (warps 8+2grp, 9+2grp) fills stage grp with the tiles g with
    // g % 3 == grp; warp wg of the group copies rows 32wg .. 32wg+31.
    const int grp = (warp - 8) >> 1, wg = (warp - 8) & 1;
    const bool q_writer = warp < 12;                         // warps 8-11 cover the four TMEM lane quadrants
    const int hq = ((warp & 3) << 5) | lane;                 // TMEM lane (head) this thread writes Q for
    const uint32_t q_lane = (uint32_t)((warp & 3) * 32) << 16;
    uint32_t g = 0, qv = 0;
    if (warp == 8 && lane == 0) tma_prefetch_desc(&tm_q_rope);
    for (int i = cluster; i < qb.num_q && !*abort; i += ncl) {
      const QueryInfo qi = query_info(qb, idx, k, i, pv);
      if (qi.nt == 0) continue;
      const int seq = __ldg(qb.q_seq + i);
      const int32_t* irow = idx + (int64_t)i * k;
      // Q of this query: every S MMA of the previous query has completed
      if (q_writer && !mbar_wait(&B.q_empty, (qv & 1) ^ 1, abort)) break;
      if (warp == 8 && lane == 0) {
        mbar_arrive_expect_tx(&B.q_full, kQRopeBytes);
        tma_load_2d(sQr, &tm_q_rope, 512 + 32 * crank, i * kH, &B.q_full);
        if (i + ncl < qb.num_q) tma_prefetch_2d(&tm_q_rope, 512 + 32 * crank, (i + ncl) * kH);
      }
      if (q_writer) {
        // latent dims [256c, 256c+256) of head hq -> TMEM columns kTmemQ .. kTmemQ+127
        const uint4* qrow = reinterpret_cast<const uint4*>(q + ((int64_t)i * kH + hq) * kDqk + crank * 256);
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < 128; c0 += 64) {
          uint4 v[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = __ldg(qrow + c0 / 4 + j);
          uint32_t r[4][16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            r[j >> 2][4 * (j & 3) + 0] = v[j].x;
            r[j >> 2][4 * (j & 3) + 1] = v[j].y;
            r[j >> 2][4 * (j & 3) + 2] = v[j].z;
            r[j >> 2][4 * (j & 3) + 3] = v[j].w;
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) tmem_st16(tmem + q_lane + kTmemQ + c0 + 16 * u, r[u]);
        }
        tmem_st_wait();
        // warm L2 with this thread's row of the next query this cluster handles
        if (i + ncl < qb.num_q) {
          const char* nrow = reinterpret_cast<const char*>(q + ((int64_t)(i + ncl) * kH + hq) * kDqk + crank * 256);
#pragma unroll
          for (int j = 0; j < 4; ++j) prefetch_l2(nrow + 128 * j);
        }
        tc_fence_before();
        mbar_arrive(&B.q_full);
      }
      bool ok = true;
      for (int t = 0; t < qi.nt; ++t, ++g) {
        if ((int)(g % kStages) != grp) continue;
        // row of this lane's entry (loaded before the wait so the latency overlaps it)
        const int e = t * kNK + 32 * wg + lane;
        int s_e = -1;
        if (e < k) s_e = __ldg(irow + e);
        ATTN_TRACE(2, g, 0, lane == 0 && wg == 0);
        const int st = g % kStages;
        if (!(ok = mbar_wait(&B.kv_empty[st], ((g / kStages) & 1) ^ 1, abort))) break;
        ATTN_TRACE(2, g, 1, lane == 0 && wg == 0);
        int row = -1;                                         // physical rows fit in 31 bits
        if (s_e >= 0 && s_e <= qi.pos) row = (int)cache_row(cm, seq, s_e, err);
        else if (s_e != -1) flag_error(err, DSA_ERR_BOUNDS);
        const uint32_t sb = sKV + st * kKVStageBytes;
        const __nv_bfloat16* lat = kv + crank * 256 + lane * 8;
        // one 32-bit broadcast per row; batches of 16 rows let the shuffles pipeline
#pragma unroll
        for (int b0 = 0; b0 < 32; b0 += 16) {
          int rr[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) rr[j] = __shfl_sync(0xffffffffu, row, b0 + j);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            cp_async16(sb + (lane >> 3) * kKVSlotBytes + sw128_offset(32 * wg + b0 + j, lane & 7),
                       rr[j] >= 0 ? lat + (int64_t)rr[j] * kDqk : kv, rr[j] >= 0 ? 16u : 0u);
        }
        {
          const __nv_bfloat16* rope = kv + 512 + 32 * crank + (lane & 3) * 8;
          int rr[4];
#pragma unroll
          for (int it = 0; it < 4; ++it) rr[it] = __shfl_sync(0xffffffffu, row, it * 8 + (lane >> 2));
#pragma unroll
          for (int it = 0; it < 4; ++it)   // rope halves: 8 rows x 4 chunks per instruction
            cp_async16(sb + 4 * kKVSlotBytes + sw64_offset(32 * wg + it * 8 + (lane >> 2), lane & 3),
                       rr[it] >= 0 ? rope + (int64_t)rr[it] * kDqk : kv, rr[it] >= 0 ? 16u : 0u);
        }
        cp_async_commit();
        cp_async_wait_all();
        fence_proxy_async_smem();
        mbar_arrive(&B.kv_full[st]);
        ATTN_TRACE(2, g, 2, lane == 0 && wg == 0);
      }
      if (!ok) break;
      ++qv;
    }
  } else {
    // ------------------------------------------------------------ MMA issue (warp 14, lane 0 issues)
    // Order per tile g: the score MMAs of g, then the P.V of g-1 as soon as
    // its P is ready (issuing score tiles further ahead was measured slower:
    // they queue in front of the P.V in the tensor pipe).
    const uint32_t id_s = idesc_bf16(128, kNK, false);
    const uint32_t id_pv = idesc_bf16(128, 256, true);
    uint32_t g = 0, qv = 0;
    auto issue_pv = [&](uint32_t gp, int tp) -> bool {
      ATTN_TRACE(3, gp, 3, lane == 0);
      if (!mbar_wait(&B.p_full[gp & 1], (gp >> 1) & 1, abort)) return false;
      ATTN_TRACE(3, gp, 4, lane == 0);
      if (tp == 0 && !mbar_wait(&B.o_empty, (qv & 1) ^ 1, abort)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t skv = sKV + (gp % kStages) * kKVStageBytes;
        const uint32_t sp = sP + (gp & 1) * kPBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16(tmem + kTmemO, sdesc(sp + kk * 32, 16, 1024), sdesc(skv + kk * 2048, kKVSlotBytes, 1024), id_pv,
                   (tp > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&B.pv_done[gp & 1]);
        mma_commit(&B.kv_empty[gp % kStages]);
      }
      __syncwarp();
      return true;
    };
    for (int i = cluster; i < qb.num_q && !*abort; i += ncl) {
      const QueryInfo qi = query_info(qb, idx, k, i, pv);
      const int nt = qi.nt;
      if (nt == 0) continue;
      if (!mbar_wait(&B.q_full, qv & 1, abort)) break;
      bool ok = true;
      for (int t = 0; t < nt; ++t, ++g) {
        const uint32_t st = g % kStages, sb = g & 1;
        ATTN_TRACE(3, g, 0, lane == 0);
        if (!(ok = mbar_wait(&B.kv_full[st], (g / kStages) & 1, abort))) break;
        ATTN_TRACE(3, g, 1, lane == 0);
        if (!(ok = mbar_wait(&B.s_empty[sb], ((g >> 1) & 1) ^ 1, abort))) break;
        ATTN_TRACE(3, g, 2, lane == 0);
        tc_fence_after();
        if (lane == 0) {
          const uint32_t dS = tmem + kTmemS + 64 * sb;
          const uint32_t skv = sKV + st * kKVStageBytes;
          uint32_t n = 0;
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk, ++n)
              mma_bf16_ts(dS, tmem + kTmemQ + a * 32 + kk * 8, sdesc(skv + a * kKVSlotBytes + kk * 32, 16, 1024),
                          id_s, n > 0 ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
            mma_bf16(dS, sdesc_sw64(sQr + kk * 32, 512), sdesc_sw64(skv + 4 * kKVSlotBytes + kk * 32, 512), id_s,
                     1u);
          mma_commit(&B.s_full[sb]);
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
  if (warp == 14) {
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

#ifdef DSA_ATTN_TRACE
extern "C" __attribute__((visibility("default"))) int dsa_attn_trace_read(long long* out) {
  return (int)cudaMemcpyFromSymbol(out, g_attn_trace, sizeof(g_attn_trace));
}
#endif

cudaError_t launch_attn_tc(const QueryBatch& qb, const CacheMap& cm, const dsa_attn_inputs& at, const int32_t* idx,
                           int k, bool prefix_valid, void* out, float* lse, int* err, cudaStream_t stream) {
  CUtensorMap q_rope;
  const uint64_t qrows = (uint64_t)qb.num_q * kH;
  if (!make_tmap_bf16(&q_rope, at.q, qrows, kDqk, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  const int ncl = std::min(qb.num_q, sm_count() / 2);
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc);
  if (e != cudaSuccess) return e;
  const float scale_log2 = (float)((double)at.softmax_scale * 1.4426950408889634);
  attn_tc_kernel<<<2 * ncl, kThreads, kSmemAlloc, stream>>>(q_rope, static_cast<const __nv_bfloat16*>(at.q),
                                                             static_cast<const __nv_bfloat16*>(at.kv),
                                                             qb, cm, idx, k,
                                                             prefix_valid ? 1 : 0, scale_log2,
                                                             static_cast<__nv_bfloat16*>(out), lse, err);
  return cudaGetLastError();
}

}  // namespace dsa
