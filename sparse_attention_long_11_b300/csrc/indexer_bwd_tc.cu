// Indexer training step on the 5th-generation tensor cores (FP8 indexer
// operands, 64 heads x 128): the alignment loss KL(p || softmax(I)) over a
// query's candidate entries and its gradients (news article on DeepSeek-V3.2,
// continued-pre-training section: the indexer learns from a Kullback-Leibler
// loss against the main attention's distribution, over all keys in the dense
// warm-up and over the selected entries in the sparse phase).
//
// Same quantities as the CUDA-core kernel (indexer_bwd.cu); with the code
// dots x_je = <q8_j, k8_e>, m_je = [x_je > 0] and the dequantising scales:
//   I_e  = sum_j w_j sq_j sk_e ReLU(x_je),  pi = softmax(I),  g_e = pi_e - p_e
//   dq_j = w_j sum_e g_e m_je sk_e k8_e                  = w_j D[:, j]
//   dw_j = sum_e g_e m_je sq_j sk_e x_je = sq_j <q8_j, D[:, j]>
//   dk_e = sum_j (g_e w_j m_je sq_j) q8_j
// with D = K8^T G, G_ej = g_e m_je sk_e.  The identity for dw is exact: the
// only rounding it adds is that of G, as in dq.
//
// One CTA (four warps, thread = entry of a 128-entry tile = TMEM lane) per
// query, two passes over the query's entries:
//   pass 1  gather the tile's key rows, decode them to fp16 (exact for e4m3),
//           X = K Q^T on the tensor cores (kind::f16, M = 128 entries,
//           N = 64 heads, K = 128 dims, fp32 accumulate: each product is
//           exact, the sum is an fp32 sum); per entry its I and the 64-bit
//           head mask, a dot within 1e-5 |q_j| |k_e| of zero re-decided in
//           fp64 from the fp16 rows already in shared memory (exact for e4m3
//           products; the fp32 sum errs by less than 127 2^-24 |q_j| |k_e|);
//   then    pi, g, the loss; power-of-two scales that put G and B = g w m sq
//           in fp16's normal range;
//   pass 2  gather the tile again; write G and B (fp16, scaled) and run
//           D += K^T G (M = 128 dims, N = 64 heads, K = 128 entries, both
//           operands read MN-major from the rows just written) and
//           dK = B Q8 (M = 128 entries, N = 128 dims, K = 64 heads); the dK
//           rows are added to dk with vector atomics.
//   end     dq and dw from D (TMEM lane = dim).
// Operands of the gradient contractions are rounded once to fp16 (2^-11
// relative), well inside the 1e-3 tolerance of each sum's magnitude.
#include <algorithm>
#include <cmath>

#include "launch.h"
#include "tc.cuh"

namespace dsa {
namespace {
using namespace tc;

constexpr int kThreads = 128;
constexpr int kHI = 64, kDI = 128, kTile = 128;
constexpr uint32_t kQHalf = kHI * 128;        // 64 heads x 64 dims (fp16), one 128B-swizzled half
constexpr uint32_t kKHalf = kTile * 128;      // 128 entries x 64 dims (fp16)
constexpr uint32_t kOffQ = 0;                 // Q: two halves (dims 0-63, 64-127)
constexpr uint32_t kOffK = kOffQ + 2 * kQHalf;    // key tile: two halves
constexpr uint32_t kOffG = kOffK + 2 * kKHalf;    // G: 128 entries x 64 heads (fp16)
constexpr uint32_t kOffB = kOffG + kTile * 128;   // B: 128 entries x 64 heads (fp16)
constexpr uint32_t kOffArr = kOffB + kTile * 128; // per entry: I then g (fp32), mask (u64)
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kTmemX = 0, kTmemD = 64, kTmemK = 128;

// fp16 instruction descriptor: D fp32, A and B fp16, M x N, majors as given.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// Four e4m3 codes (one 32-bit word, memory order) -> two f16x2 words.
__device__ __forceinline__ uint2 e4m3x4_to_f16(uint32_t c) {
  uint2 r;
  asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n cvt.rn.f16x2.e4m3x2 %0, lo;\n cvt.rn.f16x2.e4m3x2 %1, hi;\n}"
      : "=r"(r.x), "=r"(r.y)
      : "r"(c));
  return r;
}
__device__ __forceinline__ float f16_lo(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v & 0xFFFF))); }
__device__ __forceinline__ float f16_hi(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v >> 16))); }
__device__ __forceinline__ uint32_t f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

constexpr int kPend = 4;   // near-zero dots an entry may defer per tile (more are decided inline)

struct BwdShared {
  uint64_t mma;
  uint8_t npend[kThreads];          // per entry of the tile: deferred exact decisions
  uint8_t pend_j[kThreads][kPend];  // ... their heads, ascending
  float pend_x[kThreads][kPend];    // the exact dots (rounded to fp32)
  float qn[kHI], wv[kHI], sqv[kHI];
  alignas(16) float wsq[kHI];   // w_j sq_j
  float qn_max;                 // the largest code norm |q8_j|
  float red[kThreads / 32];
  float dwp[kThreads / 32][kHI];
  float skst[2][kThreads];      // each entry's key scale, copied with its tile's rows
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ float block_reduce(float v, float* red, bool is_max) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float u = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, u) : v + u;
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = red[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) t = is_max ? fmaxf(t, red[w]) : t + red[w];
  return t;
}

// 2^e with e the exponent that puts v (> 0) just below 2^14.
__device__ __forceinline__ float fp16_scale(float v) {
  if (!(v > 0.f) || !isfinite(v)) return 1.f;
  int e;
  frexpf(v, &e);   // v < 2^e
  return ldexpf(1.f, 14 - e);
}

// Four consecutive fp16 values, dims d0 .. d0+3 (d0 a multiple of 4), of row
// r of a tile held as two 128B-swizzled halves of 64 dims, `half` bytes apart.
__device__ __forceinline__ uint2 f16x4_at(const uint8_t* tile, uint32_t half, int r, int d0) {
  return *reinterpret_cast<const uint2*>(tile + (d0 >> 6) * half + sw128_offset(r, (d0 & 63) >> 3) + 2 * (d0 & 7));
}

// The exact dot of row kr of the decoded key tile at sk (fp16, decoded
// exactly from the row's e4m3 codes) with head j of the query (fp16 rows in
// the 128B-swizzled halves at sq) in fp64: every product of two e4m3 values
// and every partial sum is exact in fp64 (the sum of 128 products between
// 2^-18 and 448^2 needs at most 43 bits), so any order gives the same value.
// Here one warp computes it: lane l takes dims 4l .. 4l+3 and a butterfly
// adds the lanes' sums.  Called by a whole warp.
__device__ __forceinline__ double exact_code_dot_warp(const uint8_t* sk, int kr, const uint8_t* sq, int j, int lane) {
  const int d0 = 4 * lane;
  const uint2 f = f16x4_at(sk, kKHalf, kr, d0), g = f16x4_at(sq, kQHalf, j, d0);
  double acc = (double)f16_lo(f.x) * (double)f16_lo(g.x);
  acc = fma((double)f16_hi(f.x), (double)f16_hi(g.x), acc);
  acc = fma((double)f16_lo(f.y), (double)f16_lo(g.y), acc);
  acc = fma((double)f16_hi(f.y), (double)f16_hi(g.y), acc);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  return acc;
}

// The same dot by one thread (an entry with more than kPend near-zero dots in
// a tile: rare); kept out of line.
__device__ __noinline__ double exact_code_dot(const uint8_t* sk, int kr, const uint8_t* sq, int j) {
  double acc = 0.0;
  for (int d0 = 0; d0 < kDI; d0 += 4) {
    const uint2 f = f16x4_at(sk, kKHalf, kr, d0), g = f16x4_at(sq, kQHalf, j, d0);
    acc = fma((double)f16_lo(f.x), (double)f16_lo(g.x), acc);
    acc = fma((double)f16_hi(f.x), (double)f16_hi(g.x), acc);
    acc = fma((double)f16_lo(f.y), (double)f16_lo(g.y), acc);
    acc = fma((double)f16_hi(f.y), (double)f16_hi(g.y), acc);
  }
  return acc;
}

__global__ void __launch_bounds__(kThreads, 2)
indexer_kl_bwd_tc_kernel(QueryBatch qb, CacheMap cm, const uint8_t* __restrict__ q8, const float* __restrict__ q_scale,
                         const float* __restrict__ w, const uint8_t* __restrict__ k8, const float* __restrict__ k_scale,
                         const int32_t* __restrict__ idx, int kk, const float* __restrict__ p,
                         float* __restrict__ loss, float* __restrict__ grad_scores, float* __restrict__ dw,
                         float* __restrict__ dq, float* __restrict__ dk, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ BwdShared S;
  float* Ie = reinterpret_cast<float*>(sm + kOffArr);                        // [kk] I, then g
  uint64_t* msk = reinterpret_cast<uint64_t*>(sm + kOffArr + ((4 * kk + 15) & ~15));   // [kk]
  const int t = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort = &S.abort;
  const uint32_t sQ = smem_u32(sm + kOffQ), sK = smem_u32(sm + kOffK), sG = smem_u32(sm + kOffG),
                 sB = smem_u32(sm + kOffB);

  const int pos = __ldg(qb.q_pos + t), seq = __ldg(qb.q_seq + t);
  if (pos < 0 || pos >= qb.max_kv) {
    if (tid == 0) {
      flag_error(err, DSA_ERR_BOUNDS);
      loss[t] = 0.f;
    }
    for (int j = tid; j < kHI; j += kThreads) dw[(int64_t)t * kHI + j] = 0.f;
    for (int e = tid; e < kHI * kDI; e += kThreads) dq[(int64_t)t * kHI * kDI + e] = 0.f;
    if (grad_scores)
      for (int e = tid; e < kk; e += kThreads) grad_scores[(int64_t)t * kk + e] = 0.f;
    return;
  }
  const int32_t* irow = idx + (int64_t)t * kk;
  const float* prow = p + (int64_t)t * kk;

  if (tid == 0) {
    mbar_init(&S.mma, 1);
    S.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&S.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  // ---- the query: Q8 as fp16 (thread = head, half), code norms, weights, scales
  {
    const int j = tid >> 1, h = tid & 1;
    const uint4* src = reinterpret_cast<const uint4*>(q8 + ((int64_t)t * kHI + j) * kDI + 64 * h);
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {   // 16 codes -> two 16-byte chunks of fp16
      const uint4 v = __ldg(src + c);
      const uint32_t cw[4] = {v.x, v.y, v.z, v.w};
      uint32_t hw[8];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint2 f = e4m3x4_to_f16(cw[q]);
        hw[2 * q] = f.x;
        hw[2 * q + 1] = f.y;
        const float a = f16_lo(f.x), b = f16_hi(f.x), c2 = f16_lo(f.y), d = f16_hi(f.y);
        ss = fmaf(a, a, fmaf(b, b, fmaf(c2, c2, fmaf(d, d, ss))));
      }
      *reinterpret_cast<uint4*>(sm + kOffQ + h * kQHalf + sw128_offset(j, 2 * c)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4*>(sm + kOffQ + h * kQHalf + sw128_offset(j, 2 * c + 1)) =
          make_uint4(hw[4], hw[5], hw[6], hw[7]);
    }
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    const float qnj = sqrtf(ss);
    if (h == 0) {
      S.qn[j] = qnj;
      S.wv[j] = __ldg(w + (int64_t)t * kHI + j);
      S.sqv[j] = __ldg(q_scale + (int64_t)t * kHI + j);
      S.wsq[j] = S.wv[j] * S.sqv[j];
    }
    float qm = qnj;   // the largest head norm (all 128 threads hold one of the 64, twice)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) qm = fmaxf(qm, __shfl_xor_sync(0xffffffffu, qm, o));
    if (lane == 0) S.red[warp] = qm;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  const float qn_max = fmaxf(fmaxf(S.red[0], S.red[1]), fmaxf(S.red[2], S.red[3]));
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  uint32_t nmma = 0;   // MMA commits waited on (barrier phase)
  bool ok = true;

  // The key rows of a tile reach shared memory in two steps, so that a
  // tile's loads are in flight while the previous tile computes:
  //   locate  this thread's entry e0 + tid: its physical row (-1: padding)
  //           and key scale;
  //   stage   cp.async of the warp's 32 rows of e4m3 codes into a staging
  //           tile (128 B a row, 16-byte chunk c of row r at c ^ (r & 7);
  //           lane l copies chunk l % 8 of row l / 8 + 4i, so each copy
  //           instruction writes four whole rows);
  //   decode  once the warp's copies have landed: this thread's row, decoded
  //           to fp16 (exact for e4m3) into row tid of the key tile, and its
  //           code norm.
  // The entry indices are loaded one tile ahead of locate (ld_idx), so
  // that locate, which the next tile's copies wait on, starts from a value
  // already in a register.
  auto ld_idx = [&](int e0) { return e0 + tid < kk ? __ldg(irow + e0 + tid) : -1; };
  // locate also starts the copy of the entry's key scale into skst[buf][tid]
  // (zero for padding); it joins the tile's copy group, which stage commits.
  auto locate = [&](int s, int& row_out, int buf) {
    int64_t row = -1;
    if (s >= 0 && s <= pos) row = cache_row(cm, seq, s, err);
    else if (s != -1) flag_error(err, DSA_ERR_BOUNDS);
    row_out = (int)row;
    cp_async4(smem_u32(&S.skst[buf][tid]), row >= 0 ? k_scale + row : k_scale, row >= 0 ? 4u : 0u);
  };
  auto stage = [&](uint32_t stg, int row) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rl = 4 * i + (lane >> 3), c = lane & 7, r = warp * 32 + rl;
      const int src = __shfl_sync(0xffffffffu, row, rl);
      cp_async16(stg + r * 128 + ((c ^ (r & 7)) << 4), k8 + (int64_t)(src >= 0 ? src : 0) * kDI + c * 16,
                 src >= 0 ? 16u : 0u);
    }
    cp_async_commit();
  };
  auto decode = [&](const uint8_t* stg, float& kn_out) {
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 v = *reinterpret_cast<const uint4*>(stg + tid * 128 + ((c ^ (tid & 7)) << 4));
      const uint32_t cw[4] = {v.x, v.y, v.z, v.w};
      uint32_t hw[8];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint2 f = e4m3x4_to_f16(cw[q]);
        hw[2 * q] = f.x;
        hw[2 * q + 1] = f.y;
        const float a = f16_lo(f.x), b = f16_hi(f.x), c2 = f16_lo(f.y), d = f16_hi(f.y);
        ss = fmaf(a, a, fmaf(b, b, fmaf(c2, c2, fmaf(d, d, ss))));
      }
      // 16 codes -> fp16 chunks 2(c%4), 2(c%4)+1 of half c/4
      const uint32_t base = kOffK + (c >> 2) * kKHalf;
      *reinterpret_cast<uint4*>(sm + base + sw128_offset(tid, 2 * (c & 3))) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4*>(sm + base + sw128_offset(tid, 2 * (c & 3) + 1)) = make_uint4(hw[4], hw[5], hw[6], hw[7]);
    }
    kn_out = sqrtf(ss);
  };
  // One thread issues `fn`'s MMAs and commits; every thread waits for them.
  auto mma_round = [&](auto fn) -> bool {
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      fn();
      mma_commit(&S.mma);
    }
    const bool r = mbar_wait_warp(&S.mma, nmma & 1, abort);
    ++nmma;
    tc_fence_after();
    return r;
  };

  // ---------------------------------------------------------------- pass 1
  // staging tiles: G's and B's space, free until pass 2, alternately
  float smax = 0.f;   // largest key scale among valid entries (this thread)
  int row_n = -1;
  int s_n = -1;   // the next tile's entry index (this thread's)
  if (kk > 0) {
    locate(ld_idx(0), row_n, 0);
    stage(sG, row_n);
    s_n = ld_idx(kTile);
  }
  for (int e0 = 0, it = 0; e0 < kk && ok; e0 += kTile, ++it) {
    const int row = row_n;
    if (e0 + kTile < kk) {   // the next tile's rows, in flight while this one computes
      const int s1 = s_n;
      s_n = ld_idx(e0 + 2 * kTile);
      locate(s1, row_n, (it + 1) & 1);
      stage((it & 1) ? sG : sB, row_n);
      cp_async_wait_group1();
    } else {
      cp_async_wait_all();
    }
    __syncwarp();
    const float sk = S.skst[it & 1][tid];
    float kn;
    decode(sm + ((it & 1) ? kOffB : kOffG), kn);
    if (row >= 0) smax = fmaxf(smax, sk);
    ok = mma_round([&] {
      const Desc2 kd = desc2(sdesc(sK, 16, 1024)), qd = desc2(sdesc(sQ, 16, 1024));
      constexpr uint32_t id = idesc_f16(128, kHI, false, false);
      mma_bf16_2<0>(tmem + kTmemX, kd, qd, id);
#pragma unroll
      for (int s = 1; s < 8; ++s)   // K = 128 dims in steps of 16
        mma_bf16_2<1>(tmem + kTmemX, desc_at(kd, (s >> 2) * kKHalf + (s & 3) * 32),
                      desc_at(qd, (s >> 2) * kQHalf + (s & 3) * 32), id);
    });
    if (!ok) break;
    const int e = e0 + tid;
    uint64_t m = 0ull;
    float iv = 0.f;   // sum_j w_j sq_j ReLU(x_j); times sk at the end
    int np = 0;       // near-zero dots deferred to the warps' exact pass below
    const float kb = row >= 0 ? 1e-5f * kn : -1.f;   // |x_j| <= kb |q8_j| is near zero
    const float4* wsq4 = reinterpret_cast<const float4*>(S.wsq);
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {   // 16 heads at a time, straight from TMEM
      uint32_t r[16];
      tmem_ld16(tmem + lane_base + kTmemX + 16 * c, r);
      tmem_ld_wait();
      // screen: the smallest |x| of the 16 against the largest bound any of them has
      float amin = fabsf(__uint_as_float(r[0]));
#pragma unroll
      for (int u = 1; u < 15; u += 2)
        amin = min3(amin, fabsf(__uint_as_float(r[u])), fabsf(__uint_as_float(r[u + 1])));
      amin = fminf(amin, fabsf(__uint_as_float(r[15])));
      const bool near = amin <= kb * qn_max;
      if (!near) {
        // no dot of the 16 lies within its bound: every sign is the fp32
        // dot's (straight-line code, the same sums as the loop below)
        uint32_t mc = 0u;
#pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) {
          const float4 wq = wsq4[4 * c + u4];
          const float wj[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const float xv = __uint_as_float(r[4 * u4 + v]);
            if (xv > 0.f) {
              mc |= 1u << (4 * u4 + v);
              iv = fmaf(wj[v], xv, iv);
            }
          }
        }
        m |= (uint64_t)mc << (16 * c);
        continue;
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {   // rare: the exact test of each head's bound
        const int j = 16 * c + u;
        float xv = __uint_as_float(r[u]);
        bool posv = xv > 0.f;
        const float bound = kb * S.qn[j];
        if (bound > 0.f && fabsf(xv) <= bound) {   // near zero: decide the sign exactly
          if (np < kPend) {
            S.pend_j[tid][np++] = (uint8_t)j;
            continue;
          }
          const double exact = exact_code_dot(sm + kOffK, tid, sm + kOffQ, j);
          posv = exact > 0.0;
          xv = (float)exact;
        }
        if (posv) {
          m |= 1ull << j;
          iv = fmaf(S.wsq[j], xv, iv);
        }
      }
    }
    // the deferred dots: each warp decides its own entries' (a warp per dot)
    S.npend[tid] = (uint8_t)np;
    __syncwarp();
    for (uint32_t pm = __ballot_sync(0xffffffffu, np > 0); pm; pm &= pm - 1) {
      const int et = warp * 32 + __ffs(pm) - 1, n = S.npend[et];
      for (int q = 0; q < n; ++q) {
        const double ex = exact_code_dot_warp(sm + kOffK, et, sm + kOffQ, S.pend_j[et][q], lane);
        if (lane == 0) S.pend_x[et][q] = ex > 0.0 ? (float)ex : 0.f;
      }
    }
    __syncwarp();
    for (int q = 0; q < np; ++q) {   // heads ascending
      const float xv = S.pend_x[tid][q];
      if (xv > 0.f) {
        const int j = S.pend_j[tid][q];
        m |= 1ull << j;
        iv = fmaf(S.wsq[j], xv, iv);
      }
    }
    if (e < kk) {
      Ie[e] = row >= 0 ? iv * sk : -INFINITY;
      msk[e] = row >= 0 ? m : 0ull;
    }
    tc_fence_before();
    __syncthreads();   // the key tile and X are rewritten by the next tile
  }

  // ---------------------------------------------------------------- pi, g, loss, scales
  float lmax = -INFINITY;
  for (int e = tid; e < kk; e += kThreads) lmax = fmaxf(lmax, Ie[e]);
  const float M = block_reduce(lmax, S.red, true);
  float zp = 0.f;
  if (M != -INFINITY)
    for (int e = tid; e < kk; e += kThreads) zp += Ie[e] == -INFINITY ? 0.f : __expf(Ie[e] - M);
  const float Z = block_reduce(zp, S.red, false);
  const float logZ = logf(Z);
  float lpart = 0.f, gmax = 0.f;
  // the targets come from global memory: eight loads in flight per thread,
  // then the eight entries in the same order as one at a time
  constexpr int kPB = 8;
  for (int e8 = tid; e8 < kk; e8 += kPB * kThreads) {
    float pv[kPB];
#pragma unroll
    for (int u = 0; u < kPB; ++u) {
      const int e = e8 + u * kThreads;
      pv[u] = e < kk ? __ldg(prow + e) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kPB; ++u) {
      const int e = e8 + u * kThreads;
      if (e >= kk) break;
      const float iv = Ie[e];
      float g = 0.f;
      if (iv != -INFINITY) {
        const float lpi = iv - M - logZ;
        const float pe = pv[u];
        g = __expf(lpi) - pe;
        if (pe > 0.f) lpart += pe * (logf(pe) - lpi);
      }
      Ie[e] = g;
      gmax = fmaxf(gmax, fabsf(g));
      if (grad_scores) grad_scores[(int64_t)t * kk + e] = g;
    }
  }
  const float lsum = block_reduce(lpart, S.red, false);
  if (tid == 0) loss[t] = M == -INFINITY ? 0.f : lsum;
  gmax = block_reduce(gmax, S.red, true);
  smax = block_reduce(smax, S.red, true);
  float wsmax = 0.f;
  for (int j = tid; j < kHI; j += kThreads) wsmax = fmaxf(wsmax, fabsf(S.wv[j] * S.sqv[j]));
  wsmax = block_reduce(wsmax, S.red, true);
  const float scG = fp16_scale(gmax * smax), scB = fp16_scale(gmax * wsmax);   // G, B scaled below 2^14
  __syncthreads();
  if (ok && kk > 0) {   // pass 2's first tile
    locate(ld_idx(0), row_n, 0);
    stage(sG, row_n);
    s_n = ld_idx(kTile);
  }

  // ---------------------------------------------------------------- pass 2
  // one staging tile in G's space: each thread reads its staged row before
  // it writes its G row over the same 128 bytes; the next tile is staged
  // once this tile's MMAs have read G
  for (int e0 = 0; e0 < kk && ok; e0 += kTile) {
    const int row = row_n;
    cp_async_wait_all();
    __syncwarp();
    const float sk = S.skst[0][tid];
    float kn;
    decode(sm + kOffG, kn);
    const int e = e0 + tid;
    const uint64_t m = e < kk ? msk[e] : 0ull;
    const float ge = e < kk ? Ie[e] : 0.f;
    {   // this entry's rows of G (g m sk) and B (g w m sq), scaled, as fp16
      const float gs = ge * sk * scG;
      const float gb = ge * scB;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t hg[4], hb[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int j = 8 * c + 2 * q;
          const bool m0 = (m >> j) & 1ull, m1 = (m >> (j + 1)) & 1ull;
          hg[q] = f16x2(m0 ? gs : 0.f, m1 ? gs : 0.f);
          hb[q] = f16x2(m0 ? gb * S.wsq[j] : 0.f, m1 ? gb * S.wsq[j + 1] : 0.f);
        }
        *reinterpret_cast<uint4*>(sm + kOffG + sw128_offset(tid, c)) = make_uint4(hg[0], hg[1], hg[2], hg[3]);
        *reinterpret_cast<uint4*>(sm + kOffB + sw128_offset(tid, c)) = make_uint4(hb[0], hb[1], hb[2], hb[3]);
      }
    }
    const bool first = e0 == 0;
    ok = mma_round([&] {
      // D[d][j] += sum_e K[e][d] G[e][j]: A = the key tile read MN-major (128 dims
      // in two 64-dim blocks), B = G MN-major; 8 steps of 16 entries
      const Desc2 kd = desc2(sdesc(sK, kKHalf, 1024)), gd = desc2(sdesc(sG, 8192, 1024));
      constexpr uint32_t idD = idesc_f16(128, kHI, true, true), idK = idesc_f16(128, kDI, false, true);
      mma_bf16_2(tmem + kTmemD, kd, gd, idD, first ? 0u : 1u);
#pragma unroll
      for (int s = 1; s < 8; ++s) mma_bf16_2<1>(tmem + kTmemD, desc_at(kd, s * 2048), desc_at(gd, s * 2048), idD);
      // dK[e][d] = sum_j B[e][j] Q[j][d]: A = B K-major, B = Q read MN-major
      // (128 dims in two 64-dim blocks); 4 steps of 16 heads
      const Desc2 bd = desc2(sdesc(sB, 16, 1024)), qm = desc2(sdesc(sQ, kQHalf, 1024));
      mma_bf16_2<0>(tmem + kTmemK, bd, qm, idK);
#pragma unroll
      for (int s = 1; s < 4; ++s) mma_bf16_2<1>(tmem + kTmemK, desc_at(bd, s * 32), desc_at(qm, s * 2048), idK);
    });
    if (!ok) break;
    if (e0 + kTile < kk) {   // G has been read: stage the next tile there while dk is written
      const int s1 = s_n;
      s_n = ld_idx(e0 + 2 * kTile);
      locate(s1, row_n, 0);
      stage(sG, row_n);
    }
    {   // dk of the warp's 32 entries' key rows.  The TMEM loads give each
        // lane its own entry's dims; the warp's rows of B (free: the MMAs
        // that read them have completed) transpose 32 dims at a time, so that
        // each vector atomic instruction covers four whole 128-byte row pieces
        // instead of one 16-byte piece of 32 rows.
      const bool add = row >= 0 && m != 0ull && ge != 0.f;
      const float inv = 1.f / scB;
      uint8_t* tw = sm + kOffB + warp * 32 * 128;   // this warp's 32 rows x 128 B
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r2[2][16];
        tmem_ld16(tmem + lane_base + kTmemK + 32 * c, r2[0]);
        tmem_ld16(tmem + lane_base + kTmemK + 32 * c + 16, r2[1]);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t* v = &r2[q >> 2][4 * (q & 3)];
          *reinterpret_cast<float4*>(tw + sw128_offset(lane, q)) =
              make_float4(__uint_as_float(v[0]) * inv, __uint_as_float(v[1]) * inv, __uint_as_float(v[2]) * inv,
                          __uint_as_float(v[3]) * inv);
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {   // entries 4i .. 4i+3 of the warp, 8 lanes x 16 B each
          const int er = 4 * i + (lane >> 3);
          const int rr = __shfl_sync(0xffffffffu, row, er);
          const bool ad = __shfl_sync(0xffffffffu, add, er);
          const float4 v = *reinterpret_cast<const float4*>(tw + sw128_offset(er, lane & 7));
          if (ad) atomicAdd(reinterpret_cast<float4*>(dk + (int64_t)rr * kDI + 32 * c + 4 * (lane & 7)), v);
        }
        __syncwarp();
      }
    }
    tc_fence_before();
    __syncthreads();
  }

  // ---------------------------------------------------------------- dq, dw (thread = dim)
  if (ok) {
    const int d = tid;
    const float inv = 1.f / scG;
    const bool any = kk > 0 && M != -INFINITY;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t r[16];
      tmem_ld16(tmem + lane_base + kTmemD + 16 * c, r);
      tmem_ld_wait();
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int j = 16 * c + u;
        const float Dv = any ? __uint_as_float(r[u]) * inv : 0.f;
        dq[((int64_t)t * kHI + j) * kDI + d] = S.wv[j] * Dv;
        // q8[j][d] (fp16, exact) times D[d][j]: this thread's term of dw_j
        const uint32_t qw = *reinterpret_cast<const uint32_t*>(
            sm + kOffQ + (d >> 6) * kQHalf + sw128_offset(j, (d & 63) >> 3) + 2 * (d & 6));
        const float qv = (d & 1) ? f16_hi(qw) : f16_lo(qw);
        float v = qv * Dv;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) S.dwp[warp][j] = v;
      }
    }
    __syncthreads();
    if (tid < kHI) {
      const float s = (S.dwp[0][tid] + S.dwp[1][tid]) + (S.dwp[2][tid] + S.dwp[3][tid]);
      dw[(int64_t)t * kHI + tid] = S.sqv[tid] * s;
    }
  }

  cp_async_wait_all();   // no copy into this CTA's shared memory is left in flight (an abort leaves early)
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (tid == 0 && S.abort) flag_error(err, DSA_ERR_TIMEOUT);
}

}  // namespace

bool indexer_kl_bwd_tc_supported(const dsa_indexer_inputs& ix) {
  return ix.dtype == DSA_FP8_E4M3 && ix.heads == kHI && ix.dim == kDI;
}

cudaError_t launch_indexer_kl_bwd_tc(const QueryBatch& qb, const CacheMap& cm, const dsa_indexer_inputs& ix,
                                     const int32_t* idx, int k, const float* p, float* loss, float* grad_scores,
                                     float* dw, float* dq, float* dk, int* err, cudaStream_t stream) {
  const size_t smem = kOffArr + ((4 * (size_t)k + 15) & ~size_t(15)) + 8 * (size_t)k + 1024;
  cudaError_t e = cudaFuncSetAttribute(indexer_kl_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  indexer_kl_bwd_tc_kernel<<<qb.num_q, kThreads, smem, stream>>>(
      qb, cm, static_cast<const uint8_t*>(ix.q), ix.q_scale, ix.w, static_cast<const uint8_t*>(ix.k), ix.k_scale, idx,
      k, p, loss, grad_scores, dw, dq, dk, err);
  return cudaGetLastError();
}

}  // namespace dsa
