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
//     of shared memory frees room for four KV stages and removes 64 KB of
//     operand reads per tile from the shared-memory bandwidth.
//   * The score contraction is split by dims: CTA c contracts latent dims
//     [256c, 256c+256) and rope dims [512+32c, 512+32c+32) (288 of 576), so
//     every KV byte is gathered exactly once per query, by one CTA.  The two
//     partial logit tiles (raw dots, as fp16, or as 16-bit fixed point over
//     each head's range where a warp's partials are large) are exchanged:
//     16-bit codes halve the distributed-shared-memory traffic, which moves
//     only ~15 B/clk per SM each way.  Each CTA adds the peer's partial to
//     its own fp32 one and runs the online softmax for its half of O.  The
//     receive tiles are double buffered, so the exchange of tile g overlaps
//     the MMAs of tile g+1.
//   * Tiles of 64 selected keys, gathered with coalesced 16-byte cp.async
//     (a warp moves 512 contiguous bytes of one row per instruction) into
//     128B-swizzled latent slots and a 64B-swizzled rope half.  (TMA
//     tile::gather4 measured ~64 clk per 4-row instruction on B300, slower
//     than this path.)  Heads are the MMA's M (=128); per tile each CTA issues 18 MMAs
//     128x64x16 for S and 4 MMAs 128x256x16 for P.V, with V read MN-major
//     straight out of the gathered K-major latent slots.  An S buffer is
//     released as soon as its tile's scores are loaded (P goes through
//     shared memory), so score MMAs run ahead of the softmax.
//   * Warp roles per CTA: 0-7 exchange + softmax + epilogue in two groups
//     that take alternate tiles (thread = head = TMEM lane), so that one
//     group computes while the other waits for the peer's partial logits,
//     8-13 gather (three groups of two warps, group j
//     fills the tiles g = j mod 3 into KV stage g mod 4; at each query warps 8-11
//     write Q's latent part into TMEM and warp 8 loads the rope part with
//     TMA), 14 TMEM owner + score MMA issuer, 15 P.V MMA issuer.
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
constexpr uint32_t kXCodeBytes = kH * kNK * 2;             // one partial logit tile from the peer: 16-bit codes
constexpr uint32_t kXBytes = kXCodeBytes + kH * 8;         // ... plus each head's (step, lo) pair
constexpr int kStages = 4;
constexpr uint32_t kOffQRope = 0;
constexpr uint32_t kOffKV = kOffQRope + kQRopeBytes;       // 8 KB
constexpr uint32_t kOffX = kOffKV + kStages * kKVStageBytes;   // 152 KB
constexpr uint32_t kPBytes = kH * 128;                     // 128 x 64 bf16 probabilities (SW128)
constexpr uint32_t kOffP = kOffX + 2 * kXBytes;            // 186 KB: P[0], P[1] (1024-aligned)
constexpr uint32_t kSmemBytes = kOffP + 2 * kPBytes;       // 218 KB
static_assert(kOffP % 1024 == 0, "P tiles are 128B-swizzled MMA operands");
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;         // + alignment slack
constexpr int kGatherWarp0 = 8;
constexpr int kGatherGroups = 3;                           // of two warps; group j gathers the tiles g = j mod 3
constexpr int kMmaWarp = kGatherWarp0 + 2 * kGatherGroups; // 14: TMEM owner, score MMAs; 15: P.V MMAs
constexpr int kThreads = (kMmaWarp + 2) * 32;              // 512: at most 4 warps per SM sub-partition
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0, kTmemS = 256, kTmemQ = 384;  // S buffer b at kTmemS + 64 b
constexpr float kLn2 = 0.69314718055994530942f;

struct Bars {
  uint64_t kv_full[kStages], kv_empty[kStages], s_full[2], xf[2], xe[2];
  uint64_t s_empty[2], p_full[2], pv_done[2], mdone[2];
  uint64_t q_full, q_rope, q_empty, o_empty, qend, fin[2];
  uint64_t ostg_full[2], ostg_free[2];   // [group] O staging (in the group's P buffer) written / read by the TMA
  float mpub[2][128];           // [group][head] running maximum after the group's latest tile
  float lsum[2][2][128];        // [query parity][group][head] the groups' sums at the end of a query
  float lrsum[2][2][128];       // ... the same sums of the bf16-rounded probabilities the MMA used
  float mseen[2][2][128];       // ... and the maxima they are relative to
  float mdep;                   // write-only: orders the consumed-X arrive after the X loads (below)
  uint32_t tmem_base;
  int abort;
};

// Tiles to process for one query: up to the last tile holding a valid entry
// (0 <= s <= pos).  With prefix_valid (rows written by the top-k stage:
// ascending, valid entries first) that is ceil(min(k, pos+1) / 64) without
// reading the row; otherwise a full warp searches the row from its end in
// blocks of 256 entries, so a row whose last block holds a valid entry (any
// full selection) costs one round of loads.  Every role computes it the
// same way (the search out of line: inlined into every role it costs
// registers there).
__device__ __noinline__ int search_tiles(const int32_t* row, int k, int pos) {
  const int lane = threadIdx.x & 31;
  int last = -1;
  for (int b = (k - 1) / 256 * 256; b >= 0 && last < 0; b -= 256) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = b + 32 * u + lane;
      if (j < k) {
        const int s = __ldg(row + j);
        if (s >= 0 && s <= pos) last = j;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
  }
  return last < 0 ? 0 : last / kNK + 1;
}
__device__ __forceinline__ int count_tiles(const int32_t* row, int k, int pos, bool prefix_valid) {
  return prefix_valid ? (min(k, pos + 1) + kNK - 1) / kNK : search_tiles(row, k, pos);
}

struct QueryInfo {
  int pos, nt;
  bool ok;
};

__device__ __forceinline__ QueryInfo query_info(const QueryBatch& qb, const int32_t* idx, int k, int i, int pos,
                                                bool prefix_valid) {
  QueryInfo r;
  r.pos = pos;
  r.ok = r.pos >= 0 && r.pos < qb.max_kv;
  r.nt = r.ok ? count_tiles(idx + (int64_t)i * k, k, r.pos, prefix_valid) : 0;
  return r;
}

// The position (or sequence) of query n, or 0 past the batch: the loops
// below load each value one query ahead, so the load's latency (under the
// memory traffic of a query boundary) is off the boundary's path.
__device__ __forceinline__ int ahead_ld(const int32_t* v, int n, int num_q) { return n < num_q ? __ldg(v + n) : 0; }

// Eight e4m3 codes (memory order) -> the eight bf16 values
// bf16(s * code): each code widened exactly (e4m3 -> f16 -> f32), the
// product taken in fp32, then rounded once to nearest even.
__device__ __forceinline__ uint4 e4m3x8_scaled_bf16(uint2 c, float s) {
  uint32_t h[4];
  asm("{\n .reg .b16 l0, h0, l1, h1;\n mov.b32 {l0, h0}, %4;\n mov.b32 {l1, h1}, %5;\n"
      " cvt.rn.f16x2.e4m3x2 %0, l0;\n cvt.rn.f16x2.e4m3x2 %1, h0;\n"
      " cvt.rn.f16x2.e4m3x2 %2, l1;\n cvt.rn.f16x2.e4m3x2 %3, h1;\n}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(c.x), "r"(c.y));
  const uint64_t ss = f2(s, s);
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 v = f16x2_to_f32x2(h[j]);             // (lower code, upper code)
    const float2 p = f2_split(mul2(f2(v.x, v.y), ss));
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o[j]) : "f"(p.y), "f"(p.x));   // upper half = second code
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Reductions over one head's 64 logits of a tile: four independent chains of
// three-input min / max (eight steps each) and a final combine, so the
// result is ready soon after the last input without holding many temporaries.
template <bool kAbs, bool kMin>
__device__ __forceinline__ float tree64(const float (&x)[64]) {
  auto in = [&](int j) { return kAbs ? fabsf(x[j]) : x[j]; };
  auto op = [](float p, float q, float r) { return kMin ? min3(p, q, r) : max3(p, q, r); };
  float c[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) c[q] = in(16 * q);
#pragma unroll
  for (int j = 1; j < 15; j += 2)
#pragma unroll
    for (int q = 0; q < 4; ++q) c[q] = op(c[q], in(16 * q + j), in(16 * q + j + 1));
#pragma unroll
  for (int q = 0; q < 4; ++q) c[q] = kMin ? fminf(c[q], in(16 * q + 15)) : fmaxf(c[q], in(16 * q + 15));
  return op(op(c[0], c[1], c[2]), c[3], c[3]);
}
__device__ __forceinline__ float abs_max64(const float (&x)[64]) { return tree64<true, false>(x); }
__device__ __forceinline__ float max64(const float (&x)[64]) { return tree64<false, false>(x); }
__device__ __forceinline__ void min_max64(const float (&x)[64], float& lo, float& hi) {
  lo = tree64<false, true>(x);
  hi = tree64<false, false>(x);
}

// Adds the peer's partial logits of head h (row h of the received tile: 64
// 16-bit codes, fp16 or fixed point with the head's (step, lo) in sc) to
// this CTA's own x.
template <bool kFixed>
__device__ __forceinline__ void add_peer(float (&x)[64], const uint4* X4, int h, float2 sc) {
  const uint64_t st2 = f2(sc.x, sc.x), lo2 = f2(sc.y, sc.y), m23 = f2(-8388608.f, -8388608.f);
#pragma unroll
  for (int jq = 0; jq < 8; ++jq) {
    const uint4 v = X4[jq * 128 + h];
    const uint32_t pw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      uint64_t pv2;
      if (kFixed) {
        // each 16-bit code u as the float 2^23 + u, less 2^23 (exact), then lo + u step
        const uint64_t u2 = add2(f2(__uint_as_float(prmt(pw[e], 0x4B000000u, 0x7410u)),
                                    __uint_as_float(prmt(pw[e], 0x4B000000u, 0x7432u))),
                                 m23);
        pv2 = fma2(u2, st2, lo2);
      } else {
        const float2 pf = f16x2_to_f32x2(pw[e]);
        pv2 = f2(pf.x, pf.y);
      }
      const int j = 8 * jq + 2 * e;
      const float2 sum = f2_split(add2(f2(x[j], x[j + 1]), pv2));
      x[j] = sum.x;
      x[j + 1] = sum.y;
    }
  }
}

// P = 2^(x scale_log2 - msub) for one head's 64 logits, as bf16 pairs in pk;
// ls = the sum of the fp32 probabilities and, with kRounded, lrs = the sum of
// the bf16-rounded ones (else lrs = ls).
template <bool kRounded>
__device__ __forceinline__ void probabilities(const float (&x)[64], float scale_log2, float msub, uint32_t (&pk)[32],
                                              float& ls, float& lrs) {
  uint64_t ps2[2] = {0ull, 0ull}, pr2[2] = {0ull, 0ull};
  const uint64_t sl2 = f2(scale_log2, scale_log2), nm2 = f2(-msub, -msub);
#pragma unroll
  for (int j = 0; j < 64; j += 2) {
    const float2 d = f2_split(fma2(f2(x[j], x[j + 1]), sl2, nm2));
    const float p0 = ex2_approx(d.x);
    const float p1 = ex2_approx(d.y);
    const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
    ps2[(j >> 1) & 1] = add2(ps2[(j >> 1) & 1], f2(p0, p1));
    pk[j / 2] = *reinterpret_cast<const uint32_t*>(&pb);
    if (kRounded)
      pr2[(j >> 1) & 1] =
          add2(pr2[(j >> 1) & 1], f2(__uint_as_float(pk[j / 2] << 16), __uint_as_float(pk[j / 2] & 0xffff0000u)));
  }
  const float2 a = f2_split(ps2[0]), b = f2_split(ps2[1]);
  ls = (a.x + a.y) + (b.x + b.y);
  if (kRounded) {
    const float2 c = f2_split(pr2[0]), d = f2_split(pr2[1]);
    lrs = (c.x + c.y) + (d.x + d.y);
  } else {
    lrs = ls;
  }
}

// kFp8Kv: the latent cache holds e4m3 codes and per-row scales (kv_scale);
// the gather dequantises each row into the same bf16 shared-memory tiles.
template <bool kFp8Kv>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q_rope, const __grid_constant__ CUtensorMap tm_o,
               const __nv_bfloat16* __restrict__ q,
               const void* __restrict__ kv_raw, const float* __restrict__ kv_scale, QueryBatch qb, CacheMap cm, const int32_t* __restrict__ idx, int k, int prefix_valid,
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
      mbar_init(&B.xf[s], 1);          // armed by our thread 0; the peer's st.async credit the bytes
      mbar_init(&B.xe[s], 128);        // arrivals of the peer's softmax group of this parity
    }
    mbar_init(&B.q_full, 128);       // the 128 TMEM writers of Q's latent part
    mbar_init(&B.q_rope, 1);         // the rope TMA (with its bytes)
    mbar_init(&B.q_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&B.p_full[s], 128);
      mbar_init(&B.pv_done[s], 1);
      mbar_init(&B.mdone[s], 128);
      mbar_init(&B.s_empty[s], 128);   // the softmax group of this parity has loaded S
    }
    mbar_init(&B.o_empty, 256);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&B.ostg_full[s], 128);
      mbar_init(&B.ostg_free[s], 1);
    }
    mbar_init(&B.qend, 256);
    mbar_init(&B.fin[0], 1);
    mbar_init(&B.fin[1], 1);
    B.abort = 0;
    fence_mbar_init();
    mbar_arrive_expect_tx(&B.xf[0], kXBytes);   // arm the first phase of both receive tiles
    mbar_arrive_expect_tx(&B.xf[1], kXBytes);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&B.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // the peer's barriers exist before anyone arrives on them remotely
  tc_fence_after();
  pdl_wait();      // the set-up above ran while the stream's previous kernel finished
  pdl_release();
  const uint32_t tmem = B.tmem_base;
  const uint32_t sQr = smem_u32(sm + kOffQRope), sKV = smem_u32(sm + kOffKV), sP = smem_u32(sm + kOffP);

  if (warp < 8) {
    // ------------------------------------------------------------ exchange, softmax, epilogue
    // Two groups of four warps take alternate tiles (group b the tiles g with
    // g % 2 == b, which use S/P buffer b and receive tile X[b]); in a group,
    // thread = head = TMEM lane, over all 64 keys.  While one group waits for
    // the peer's partial logits of its tile, the other computes.  The running
    // maximum passes from tile to tile (so from group to group) through
    // shared memory; each group keeps its own running sum, relative to the
    // maximum it last saw, and the two sums meet at the end of the query.
    // The S buffer is released as soon as the group has loaded it, so the
    // score MMAs of later tiles do not wait for this tile's P.V; P (bf16)
    // goes to shared memory, the A operand of the P.V MMA.
    const int grp = warp >> 2, q4 = warp & 3;
    const int h = (q4 << 5) | lane;
    const int gtid = tid & 127;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const uint32_t tS = tmem + lane_base + kTmemS + grp * 64;   // this group's S / P buffer
    const uint32_t x_peer = mapa(smem_u32(sm + kOffX + grp * kXBytes), peer);
    const uint32_t xf_peer = mapa(smem_u32(&B.xf[grp]), peer);
    const uint32_t xe_peer = mapa(smem_u32(&B.xe[grp]), peer);
    const uint4* X4 = reinterpret_cast<const uint4*>(sm + kOffX + grp * kXBytes);
    const float2* XS = reinterpret_cast<const float2*>(sm + kOffX + grp * kXBytes + kXCodeBytes);
    uint32_t g = 0, qv = 0;   // tiles and queries (with tiles) so far, counted alike by both groups
    int pos_next = ahead_ld(qb.q_pos, cluster, qb.num_q);
    for (int i = cluster; i < qb.num_q && !*abort; i += ncl) {
      const int pos_i = pos_next;
      const QueryInfo qi = query_info(qb, idx, k, i, pos_i, pv);
      const int pos = qi.pos, nt = qi.nt;
      const int32_t* irow = idx + (int64_t)i * k;
      __nv_bfloat16* orow = out + ((int64_t)i * kH + h) * kDv + crank * 256 + grp * 128;
      if (nt == 0) {
        uint4* o4 = reinterpret_cast<uint4*>(orow);
#pragma unroll 4
        for (int c = 0; c < 16; ++c) o4[c] = make_uint4(0, 0, 0, 0);
        if (crank == 0 && grp == 0) lse[(int64_t)i * kH + h] = -INFINITY;
        if (!qi.ok && h == 0 && crank == 0 && grp == 0) flag_error(err, DSA_ERR_BOUNDS);
        pos_next = ahead_ld(qb.q_pos, i + ncl, qb.num_q);
        continue;
      }
      const int n_valid = min(k, pos + 1);
      float m_seen = -INFINITY, l = 0.f, lr = 0.f;   // the maximum this group last used, its sums relative to it
      bool ok = true;
      const uint32_t g0 = g;
      for (int t = ((g0 & 1u) == (uint32_t)grp) ? 0 : 1; t < nt; t += 2) {
        const uint32_t gt = g0 + t;
        const uint32_t par = (gt >> 1) & 1;
        int s_e0 = 0, s_e1 = 0;
        if (!pv) {   // this lane's entries (keys lane, lane+32 of the tile), loaded early
          const int e0 = t * kNK + lane, e1 = e0 + 32;
          s_e0 = e0 < k ? __ldg(irow + e0) : -1;
          s_e1 = e1 < k ? __ldg(irow + e1) : -1;
        }
        if (!(ok = mbar_wait_warp(&B.s_full[grp], par, abort))) break;
        tc_fence_after();
        // own partial logits, raw dots (the scale to base-2 units is applied
        // in the exponent); the peer gets them as fp16 or, where they are
        // large, as 16-bit fixed point (R20)
        float x[64];
        {
          uint32_t r[4][16];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld16(tS + c * 16, r[c]);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 64; ++j) x[j] = __uint_as_float(r[j >> 4][j & 15]);
        }
        tc_fence_before();
        mbar_arrive(&B.s_empty[grp]);   // S(gt+2) may be computed into this buffer
        // own partial -> the peer's X[grp], once the peer has consumed what we wrote there two tiles ago
        if (!(ok = mbar_wait_warp<true>(&B.xe[grp], par ^ 1, abort))) break;
        bool precise;   // this warp sent fixed point (warp-uniform)
        {
          // fp16 carries a partial within 2^-11 of its size: a logit error
          // under 0.004 base-2 units while |x| stays below 8 of them.  A warp
          // with any larger partial sends 16-bit fixed point over each head's
          // range instead: codes u = round((x - lo) / step), 0..65534, step =
          // (hi - lo) / 65534, read back as lo + u step within about half a step.
          precise = __any_sync(0xffffffffu, abs_max64(x) * scale_log2 > 8.f);
          float step = -1.f, lo = 0.f;   // a negative step marks fp16 codes
          if (precise) {
            float hi;
            min_max64(x, lo, hi);
            const float range = hi - lo;
            const float inv = range > 0.f ? __fdividef(65534.f, range) : 0.f;
            step = range * (1.f / 65534.f);
            const uint64_t nlo2 = f2(-lo, -lo), inv2 = f2(inv, inv), mag2 = f2(12582912.f, 12582912.f);
#pragma unroll
            for (int jq = 0; jq < 8; ++jq) {
              uint32_t cw[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                // (x - lo) * inv + 1.5 * 2^23: the low 16 bits of the float are the rounded code
                const int j = 8 * jq + 2 * e;
                const float2 y = f2_split(fma2(add2(f2(x[j], x[j + 1]), nlo2), inv2, mag2));
                cw[e] = prmt(__float_as_uint(y.x), __float_as_uint(y.y), 0x5410u);
              }
              st_async_v4_b32(x_peer + (uint32_t)(jq * 128 + h) * 16u, make_uint4(cw[0], cw[1], cw[2], cw[3]),
                              xf_peer);
            }
          } else {
#pragma unroll
            for (int jq = 0; jq < 8; ++jq) {
              const int j = 8 * jq;
              st_async_v4_b32(x_peer + (uint32_t)(jq * 128 + h) * 16u,
                              make_uint4(f16x2_sat(x[j], x[j + 1]), f16x2_sat(x[j + 2], x[j + 3]),
                                         f16x2_sat(x[j + 4], x[j + 5]), f16x2_sat(x[j + 6], x[j + 7])),
                              xf_peer);
            }
          }
          st_async_v2_f32(x_peer + kXCodeBytes + (uint32_t)h * 8u, step, lo, xf_peer);
        }
        if (!(ok = mbar_wait_warp<true>(&B.xf[grp], par, abort))) break;   // the peer's partial is in X[grp]
        // arm the next phase: the peer writes X[grp] again only after all of
        // this group has read it and said so (below)
        if (gtid == 0) mbar_arrive_expect_tx(&B.xf[grp], kXBytes);
        uint32_t vm_lo, vm_hi;
        if (pv) {
          const int rem = n_valid - t * kNK;   // the valid entries of this tile form a prefix
          vm_lo = rem >= 32 ? 0xffffffffu : (rem <= 0 ? 0u : (1u << rem) - 1u);
          vm_hi = rem >= 64 ? 0xffffffffu : (rem <= 32 ? 0u : (1u << (rem - 32)) - 1u);
        } else {
          vm_lo = __ballot_sync(0xffffffffu, s_e0 >= 0 && s_e0 <= pos);
          vm_hi = __ballot_sync(0xffffffffu, s_e1 >= 0 && s_e1 <= pos);
        }
        // x = own (fp32) + peer (fp16 or fixed point), raw dots.  The two CTAs'
        // logits differ by the rounding of one partial; each CTA's half of O
        // stays consistent with its own P and sum, which is all the
        // normalisation needs.
        const float2 sc = XS[h];              // the peer's (step, lo) for this head
        const bool peer_fixed = sc.x >= 0.f;  // warp-uniform: the peer's warp for these heads voted
        if (peer_fixed) add_peer<true>(x, X4, h, sc);
        else add_peer<false>(x, X4, h, sc);
        if ((vm_lo & vm_hi) != 0xffffffffu) {   // rare: a tile with invalid entries
#pragma unroll
          for (int j = 0; j < 64; ++j)
            if (!(((j < 32 ? vm_lo : vm_hi) >> (j & 31)) & 1u)) x[j] = -INFINITY;
        }
        const float mt = max64(x) * scale_log2;   // base-2 units
        // X[grp] consumed: the store below needs mt, which depends on every
        // value loaded from X, and instructions issue in order, so the relaxed
        // arrive after it follows those loads (a release-ordered remote arrive
        // costs ~1.5k clk)
        *reinterpret_cast<volatile float*>(&B.mdep) = mt;
        mbar_arrive_remote_relaxed(xe_peer);
        // the running maximum after tile gt-1 (waiting also at a query's first
        // tile keeps the two groups within one tile of each other)
        float m_prev = -INFINITY;
        if (gt > 0) {
          if (!(ok = mbar_wait_warp(&B.mdone[grp ^ 1], ((gt - 1) >> 1) & 1, abort))) break;
          if (t > 0) m_prev = B.mpub[grp ^ 1][h];
        }
        // lazy rescaling: the maximum used only moves when exceeded by more than 8 (a factor 256)
        const float m_use = mt > m_prev + 8.f ? mt : m_prev;
        B.mpub[grp][h] = m_use;
        mbar_arrive(&B.mdone[grp]);
        if (m_use != m_seen) {   // this group's sums follow the maximum
          const float a = ex2_approx(m_seen - m_use);
          l *= a;
          lr *= a;
          m_seen = m_use;
        }
        const float msub = m_use == -INFINITY ? 0.f : m_use;   // all p are 0 while nothing is valid
        uint32_t pk[32];
        // the sum of the fp32 probabilities (for LSE), and the one that
        // normalises O.  Where large partials travelled as fixed point (a
        // peaked softmax) the latter sums the bf16-rounded probabilities the
        // P.V MMA multiplies, so that O is an exact convex combination of the
        // V rows with the rounded weights; elsewhere it is the fp32 sum.
        float ls, lrs;
        if (__any_sync(0xffffffffu, precise || peer_fixed)) probabilities<true>(x, scale_log2, msub, pk, ls, lrs);
        else probabilities<false>(x, scale_log2, msub, pk, ls, lrs);
        l += ls;
        lr += lrs;
        // The heads of a warp decide separately whether their maximum moved,
        // but the TMEM loads and stores are warp-collective: the warp rescales
        // when any of its heads needs it, the others by exactly 1.
        const bool rescale = t > 0 && m_use != m_prev;
        if (__any_sync(0xffffffffu, rescale)) {
          // O holds the P.V of tiles < gt relative to m_prev; that of tile gt-1 must be complete
          if (!(ok = mbar_wait_warp(&B.pv_done[grp ^ 1], ((gt - 1) >> 1) & 1, abort))) break;
          tc_fence_after();
          const float alpha = rescale ? ex2_approx(m_prev - m_use) : 1.f;
#pragma unroll 1
          for (int c = 0; c < 256; c += 16) {
            uint32_t r[16];
            tmem_ld16(tmem + lane_base + kTmemO + c, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
            tmem_st16(tmem + lane_base + kTmemO + c, r);
          }
        }
        // P -> shared memory (SW128, row = head); P[grp] is free once the
        // P.V of tile gt-2 has completed
        if (!(ok = mbar_wait_warp(&B.pv_done[grp], par ^ 1, abort))) break;
        {
          uint8_t* prow = sm + kOffP + grp * kPBytes;
#pragma unroll
          for (int cc = 0; cc < 8; ++cc)
            *reinterpret_cast<uint4*>(prow + sw128_offset(h, cc)) =
                make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&B.p_full[grp]);
      }
      g = g0 + nt;
      if (!ok) break;
      pos_next = ahead_ld(qb.q_pos, i + ncl, qb.num_q);   // the next query's position, during this epilogue
      // epilogue: the two groups' sums relative to the final maximum; each
      // group normalises and stores half of this CTA's O columns
      const int qb2 = qv & 1;
      B.lsum[qb2][grp][h] = l;
      B.lrsum[qb2][grp][h] = lr;
      B.mseen[qb2][grp][h] = m_seen;
      mbar_arrive(&B.qend);
      if (!mbar_wait_warp(&B.qend, qb2, abort)) break;
      const float ma = B.mseen[qb2][0][h], mb = B.mseen[qb2][1][h];
      const float mf = fmaxf(ma, mb);
      const float fa = mf == -INFINITY ? 0.f : ex2_approx(ma - mf), fb = mf == -INFINITY ? 0.f : ex2_approx(mb - mf);
      const float lt = B.lsum[qb2][0][h] * fa + B.lsum[qb2][1][h] * fb;      // for LSE
      const float ltr = B.lrsum[qb2][0][h] * fa + B.lrsum[qb2][1][h] * fb;   // for O
      if (!mbar_wait_warp(&B.pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, abort)) break;
      tc_fence_after();
      const float inv = ltr > 0.f ? 1.f / ltr : 0.f;
      // O leaves through the TMA: every P.V of the query has completed, so the
      // group's P buffer is free and stages the group's 128 columns as two
      // boxes of 64 (128 heads x 128 B, 128-byte swizzle); the rows of a
      // box are stored as whole lines instead of one 16-byte piece per head.
      uint8_t* stg = sm + kOffP + grp * kPBytes;
      constexpr int kEpiLoads = kFp8Kv ? 1 : 2;   // 16-column TMEM loads per wait (registers allowing)
      bool eok = true;
#pragma unroll 1
      for (int b = 0; b < 2 && eok; ++b) {
#pragma unroll 1
        for (int c = 0; c < 64; c += 16 * kEpiLoads) {
          uint32_t r2[kEpiLoads][16];
#pragma unroll
          for (int u = 0; u < kEpiLoads; ++u) tmem_ld16(tmem + lane_base + kTmemO + grp * 128 + 64 * b + c + 16 * u, r2[u]);
          tmem_ld_wait();
          auto r = [&](int j) { return r2[j >> 4][j & 15]; };
#pragma unroll
          for (int q = 0; q < 2 * kEpiLoads; ++q) {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(r(8 * q + 2 * j)) * inv,
                                                             __uint_as_float(r(8 * q + 2 * j + 1)) * inv);
              w[j] = *reinterpret_cast<const uint32_t*>(&v);
            }
            *reinterpret_cast<uint4*>(stg + sw128_offset(h, c / 8 + q)) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&B.ostg_full[grp]);
        if (gtid == 0) {
          if ((eok = mbar_wait(&B.ostg_full[grp], b, abort))) {
            tma_store_2d(&tm_o, smem_u32(stg), crank * 256 + grp * 128 + 64 * b, i * kH);
            bulk_commit();
            bulk_wait_read();   // the staging may be written again
            mbar_arrive(&B.ostg_free[grp]);
          }
        }
        eok = mbar_wait_warp(&B.ostg_free[grp], b, abort);
      }
      if (!eok) break;
      if (crank == 0 && grp == 0) lse[(int64_t)i * kH + h] = lt > 0.f ? (mf + log2f(lt)) * kLn2 : -INFINITY;
      tc_fence_before();
      mbar_arrive(&B.o_empty);
      ++qv;
    }
    if (gtid == 0) bulk_wait_all();   // this group's O stores have completed before the CTA may exit
  } else if (warp < kMmaWarp) {
    // ------------------------------------------------------------ gather (cp.async) + Q (TMA)
    // Group grp (warps 8+2grp, 9+2grp) fills stage grp with the tiles g with
    // g % 3 == grp; warp wg of the group copies rows 32wg .. 32wg+31.
    const int grp = (warp - kGatherWarp0) >> 1, wg = (warp - kGatherWarp0) & 1;
    const bool q_writer = warp < 12;                         // warps 8-11 cover the four TMEM lane quadrants
    const int hq = ((warp & 3) << 5) | lane;                 // TMEM lane (head) this thread writes Q for
    const uint32_t q_lane = (uint32_t)((warp & 3) * 32) << 16;
    uint32_t g = 0, qv = 0, n_rope = 0;   // n_rope: rope TMA loads issued (warp 8, lane 0)
    if (warp == 8 && lane == 0) tma_prefetch_desc(&tm_q_rope);
    // bf16 rows: this lane's entry s_e of tile gt -> 16-byte cp.async pieces
    // of the warp's 32 rows in stage st (latent half, then rope quarter)
    auto issue_bf16 = [&](int s_e, int qpos, int seq, int st) {
      int row = -1;                                         // physical rows fit in 31 bits
      if (s_e >= 0 && s_e <= qpos) row = (int)cache_row(cm, seq, s_e, err);
      else if (s_e != -1) flag_error(err, DSA_ERR_BOUNDS);
      const uint32_t sb = sKV + st * kKVStageBytes;
      const __nv_bfloat16* kv = static_cast<const __nv_bfloat16*>(kv_raw);
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
    };
    int pos_next = ahead_ld(qb.q_pos, cluster, qb.num_q), seq_next = ahead_ld(qb.q_seq, cluster, qb.num_q);
    for (int i = cluster; i < qb.num_q && !*abort; i += ncl) {
      const int pos_i = pos_next, seq = seq_next;
      pos_next = ahead_ld(qb.q_pos, i + ncl, qb.num_q);
      seq_next = ahead_ld(qb.q_seq, i + ncl, qb.num_q);
      const QueryInfo qi = query_info(qb, idx, k, i, pos_i, pv);
      if (qi.nt == 0) continue;
      const int32_t* irow = idx + (int64_t)i * k;
      // Q of this query: every S MMA of the previous query has completed
      if (q_writer && !mbar_wait_warp(&B.q_empty, (qv & 1) ^ 1, abort)) break;
      // A Q writer's first tile of this query, when its stage is free by now
      // (the previous query's last P.V MMAs have mostly completed): its
      // copies go out before Q is written and land meanwhile, instead of
      // after it (the query's first tiles wait on both).
      int t_pre = -1;
      if (!kFp8Kv && q_writer) {
        const int t1 = (grp - (int)(g % kGatherGroups) + kGatherGroups) % kGatherGroups;
        if (t1 < qi.nt) {
          const uint32_t g1 = g + t1;
          const int st1 = g1 % kStages;
          const bool free1 = __shfl_sync(0xffffffffu, lane == 0 ? (int)mbar_test(&B.kv_empty[st1], ((g1 / kStages) & 1) ^ 1) : 0, 0) != 0;
          if (free1) {
            const int e = t1 * kNK + 32 * wg + lane;
            const int s_e = e < k ? __ldg(irow + e) : -1;
            issue_bf16(s_e, qi.pos, seq, st1);
            t_pre = t1;
          }
        }
      }
      if (warp == 8 && lane == 0) {
        mbar_arrive_expect_tx(&B.q_rope, kQRopeBytes);
        tma_load_2d(sQr, &tm_q_rope, 512 + 32 * crank, i * kH, &B.q_rope);
        ++n_rope;
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
        if ((int)(g % kGatherGroups) != grp) continue;
        if (t == t_pre) {
          cp_async_wait_all();
          fence_proxy_async_smem();
          mbar_arrive(&B.kv_full[g % kStages]);
          continue;
        }
        // row of this lane's entry (loaded before the wait so the latency overlaps it)
        const int e = t * kNK + 32 * wg + lane;
        int s_e = -1;
        if (e < k) s_e = __ldg(irow + e);
        const int st = g % kStages;
        if constexpr (kFp8Kv) {
          // FP8 rows go through registers (8 codes = 8 bytes per lane and row
          // in, 16 bytes of bf16 out, into the same swizzled slots the bf16
          // path fills), so their loads may start before the stage is free:
          // the first two batches of 8 rows are in flight during the wait,
          // and after it each batch is converted while the next one loads.
          int row = -1;
          if (s_e >= 0 && s_e <= qi.pos) row = (int)cache_row(cm, seq, s_e, err);
          else if (s_e != -1) flag_error(err, DSA_ERR_BOUNDS);
          const uint8_t* kv8 = static_cast<const uint8_t*>(kv_raw);
          const float srow = row >= 0 ? __ldg(kv_scale + row) : 0.f;
          const uint8_t* lat8 = kv8 + crank * 256 + lane * 8;
          const uint8_t* rope8 = kv8 + 512 + 32 * crank + (lane & 3) * 8;
          auto load8 = [&](int b0, uint2 (&c)[8]) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int r = __shfl_sync(0xffffffffu, row, b0 + j);
              c[j] = r >= 0 ? __ldg(reinterpret_cast<const uint2*>(lat8 + (int64_t)r * kDqk)) : make_uint2(0, 0);
            }
          };
          uint8_t* sbp = sm + kOffKV + st * kKVStageBytes;
          auto store8 = [&](int b0, const uint2 (&c)[8]) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float sj = __shfl_sync(0xffffffffu, srow, b0 + j);
              *reinterpret_cast<uint4*>(sbp + (lane >> 3) * kKVSlotBytes + sw128_offset(32 * wg + b0 + j, lane & 7)) =
                  e4m3x8_scaled_bf16(c[j], sj);
            }
          };
          uint2 ca[8], cb[8], cr[4];
          load8(0, ca);
          load8(8, cb);
          if (!(ok = mbar_wait_warp(&B.kv_empty[st], ((g / kStages) & 1) ^ 1, abort))) break;
          store8(0, ca);
          load8(16, ca);
          store8(8, cb);
          load8(24, cb);
          store8(16, ca);
#pragma unroll
          for (int it = 0; it < 4; ++it) {   // rope: 8 rows x 4 lanes of 8 codes per step
            const int r = __shfl_sync(0xffffffffu, row, it * 8 + (lane >> 2));
            cr[it] = r >= 0 ? __ldg(reinterpret_cast<const uint2*>(rope8 + (int64_t)r * kDqk)) : make_uint2(0, 0);
          }
          store8(24, cb);
#pragma unroll
          for (int it = 0; it < 4; ++it) {
            const float sj = __shfl_sync(0xffffffffu, srow, it * 8 + (lane >> 2));
            *reinterpret_cast<uint4*>(sbp + 4 * kKVSlotBytes + sw64_offset(32 * wg + it * 8 + (lane >> 2), lane & 3)) =
                e4m3x8_scaled_bf16(cr[it], sj);
          }
          fence_proxy_async_smem();
          mbar_arrive(&B.kv_full[st]);
          continue;
        }
        if (!(ok = mbar_wait_warp(&B.kv_empty[st], ((g / kStages) & 1) ^ 1, abort))) break;
        issue_bf16(s_e, qi.pos, seq, st);
        cp_async_wait_all();
        fence_proxy_async_smem();
        mbar_arrive(&B.kv_full[st]);
      }
      if (!ok) break;
      ++qv;
    }
    // copies issued before an abort, and the last rope TMA issued here, have
    // landed before the CTA may exit
    cp_async_wait_all();
    if (warp == 8 && lane == 0 && n_rope > 0) mbar_wait_own(&B.q_rope, (n_rope - 1) & 1);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ score MMA issue (lane 0)
    // S(g) goes into buffer g % 2 once the softmax group has loaded S(g-2)
    // from it.  The tensor core accepts only a couple of MMAs ahead, so a
    // second issuing warp lets the P.V MMAs slot in between the score MMAs
    // instead of waiting behind them.
    const uint32_t id_s = idesc_bf16(128, kNK, false);
    uint32_t g = 0, qv = 0;
    int pos_next = ahead_ld(qb.q_pos, cluster, qb.num_q);
    for (int i = cluster; i < qb.num_q && !*abort; i += ncl) {
      const int pos_i = pos_next;
      pos_next = ahead_ld(qb.q_pos, i + ncl, qb.num_q);
      const QueryInfo qi = query_info(qb, idx, k, i, pos_i, pv);
      const int nt = qi.nt;
      if (nt == 0) continue;
      if (!mbar_wait_warp(&B.q_full, qv & 1, abort) || !mbar_wait_warp(&B.q_rope, qv & 1, abort)) break;
      bool ok = true;
      for (int t = 0; t < nt; ++t, ++g) {
        const uint32_t st = g % kStages, sb = g & 1;
        if (!(ok = mbar_wait_warp(&B.kv_full[st], (g / kStages) & 1, abort))) break;
        if (!(ok = mbar_wait_warp(&B.s_empty[sb], ((g >> 1) & 1) ^ 1, abort))) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t dS = tmem + kTmemS + 64 * sb;
          const uint32_t skv = sKV + st * kKVStageBytes;
          // one descriptor per operand and tile; each MMA offsets its low word
          const Desc2 kd = desc2(sdesc(skv, 16, 1024));
          const Desc2 rq = desc2(sdesc_sw64(sQr, 512)), rk = desc2(sdesc_sw64(skv + 4 * kKVSlotBytes, 512));
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t aq = tmem + kTmemQ + a * 32 + kk * 8;
              const Desc2 b = desc_at(kd, a * kKVSlotBytes + kk * 32);
              if (a == 0 && kk == 0) mma_bf16_ts2<0>(dS, aq, b, id_s);
              else mma_bf16_ts2<1>(dS, aq, b, id_s);
            }
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) mma_bf16_2<1>(dS, desc_at(rq, kk * 32), desc_at(rk, kk * 32), id_s);
          mma_commit(&B.s_full[sb]);
          if (t == nt - 1) mma_commit(&B.q_empty);
        }
        __syncwarp();
      }
      if (!ok) break;
      ++qv;
    }
    if (lane == 0) mma_commit(&B.fin[0]);
    __syncwarp();
    mbar_wait_own(&B.fin[0], 0);   // every MMA issued by this warp has completed
  } else {
    // ------------------------------------------------------------ P.V MMA issue (warp 15, lane 0)
    const uint32_t id_pv = idesc_bf16(128, 256, true);
    uint32_t g = 0, qv = 0;
    int pos_next = ahead_ld(qb.q_pos, cluster, qb.num_q);
    for (int i = cluster; i < qb.num_q && !*abort; i += ncl) {
      const int pos_i = pos_next;
      pos_next = ahead_ld(qb.q_pos, i + ncl, qb.num_q);
      const QueryInfo qi = query_info(qb, idx, k, i, pos_i, pv);
      const int nt = qi.nt;
      if (nt == 0) continue;
      bool ok = true;
      for (int t = 0; t < nt; ++t, ++g) {
        if (!(ok = mbar_wait_warp(&B.p_full[g & 1], (g >> 1) & 1, abort))) break;
        // the epilogue of the previous query has read O
        if (t == 0 && !(ok = mbar_wait_warp(&B.o_empty, (qv & 1) ^ 1, abort))) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t skv = sKV + (g % kStages) * kKVStageBytes;
          const uint32_t sp = sP + (g & 1) * kPBytes;
          const Desc2 pd = desc2(sdesc(sp, 16, 1024)), vd = desc2(sdesc(skv, kKVSlotBytes, 1024));
          mma_bf16_2(tmem + kTmemO, pd, vd, id_pv, t > 0 ? 1u : 0u);
#pragma unroll
          for (int kk = 1; kk < 4; ++kk) mma_bf16_2<1>(tmem + kTmemO, desc_at(pd, kk * 32), desc_at(vd, kk * 2048), id_pv);
          mma_commit(&B.pv_done[g & 1]);
          mma_commit(&B.kv_empty[g % kStages]);
        }
        __syncwarp();
      }
      if (!ok) break;
      ++qv;
    }
    if (lane == 0) mma_commit(&B.fin[1]);
    __syncwarp();
    mbar_wait_own(&B.fin[1], 0);   // every MMA issued by this warp has completed
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();       // the peer no longer reads or writes our shared memory
  if (warp == kMmaWarp) {
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

// A whole FP8 latent cache as bf16: each thread converts groups of eight
// codes of one row with the gather's own conversion (e4m3x8_scaled_bf16),
// so the copy holds exactly the values the FP8 gather stages.  Groups are
// strided over the grid; loads and stores are contiguous across a warp.
__global__ void __launch_bounds__(256) kv_dequant_kernel(const uint8_t* __restrict__ kv8,
                                                         const float* __restrict__ kv_scale, int64_t num_rows,
                                                         __nv_bfloat16* __restrict__ out) {
  constexpr int kGroups = kDqk / 8;   // 72 groups of eight codes a row
  const int64_t n = num_rows * kGroups;
  for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < n; g += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = g / kGroups;
    const uint2 c = __ldg(reinterpret_cast<const uint2*>(kv8) + g);
    reinterpret_cast<uint4*>(out)[g] = e4m3x8_scaled_bf16(c, __ldg(kv_scale + r));
  }
}

}  // namespace

cudaError_t launch_kv_dequant(const void* kv, const float* kv_scale, int64_t num_rows, void* out,
                              cudaStream_t stream) {
  if (num_rows <= 0) return cudaSuccess;
  const int64_t groups = num_rows * (kDqk / 8);
  const int64_t blocks = std::min<int64_t>((groups + 255) / 256, (int64_t)sm_count() * 8);
  kv_dequant_kernel<<<(unsigned)blocks, 256, 0, stream>>>(static_cast<const uint8_t*>(kv), kv_scale, num_rows,
                                                          static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

cudaError_t launch_attn_tc(const QueryBatch& qb, const CacheMap& cm, const dsa_attn_inputs& at, const int32_t* idx,
                           int k, bool prefix_valid, void* out, float* lse, int* err, cudaStream_t stream) {
  CUtensorMap q_rope, o_map;
  const uint64_t qrows = (uint64_t)qb.num_q * kH;
  if (!make_tmap_bf16(&q_rope, at.q, qrows, kDqk, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&o_map, out, qrows, kDv, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
  const int ncl = std::min(qb.num_q, sm_count() / 2);
  const bool fp8 = at.dtype == DSA_FP8_E4M3;
  auto kern = fp8 ? attn_tc_kernel<true> : attn_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc);
  if (e != cudaSuccess) return e;
  const float scale_log2 = (float)((double)at.softmax_scale * 1.4426950408889634);
  return launch_pdl(kern, dim3(2 * ncl), dim3(kThreads), kSmemAlloc, stream, q_rope, o_map,
                    static_cast<const __nv_bfloat16*>(at.q), at.kv, fp8 ? at.kv_scale : nullptr, qb, cm, idx, k,
                    prefix_valid ? 1 : 0, scale_log2, static_cast<__nv_bfloat16*>(out), lse, err);
}

}  // namespace dsa
