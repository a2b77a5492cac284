// Indexer training step: the alignment loss of the lightning indexer and its
// gradients (news article on DeepSeek-V3.2, continued-pre-training section:
// the indexer learns from a Kullback-Leibler loss against the main
// attention's distribution -- over all keys in the dense warm-up, over the
// selected entries only in the sparse phase, where that loss is the
// indexer's only source of gradient).
//
// For query t with candidate entries S (the valid entries of its idx row),
// a target distribution p over them, the dequantised operands
// q_j = sq_j * q8_j and k_s = sk_s * k8_s, and x_js = <q_j, k_s>:
//   I_s  = sum_j w_j ReLU(x_js),   pi = softmax_S(I)
//   loss = sum_s p_s (log p_s - log pi_s),   g_s = pi_s - p_s
//   dw_j = sum_s g_s ReLU(x_js)
//   dq_j = w_j sum_s g_s [x_js > 0] k_s
//   dk_s += g_s sum_j w_j [x_js > 0] q_j          (scattered over key rows)
//
// CUDA cores, one 256-thread block per query, candidates in tiles of 64:
//   pass 1  per tile: the 64 x 64 head-key dots (each thread a 4 x 4 block),
//           I of the tile, the head masks [x > 0] as one 64-bit word per
//           entry, and dw's two sums (exp-weighted with a running maximum,
//           and p-weighted) -- so dw needs no second look at x;
//   then    pi, g and the loss over all entries;
//   pass 2  per tile: dq from the masks and g, and dk (vector atomics),
//           register-blocked 8 ways (a 16-byte shared load costs the same
//           four wavefronts whether or not the lanes share its address).
// The mask decides which terms exist, so it must not depend on rounding:
// a dot whose fp32 value lies within its rounding bound of zero
// (|x| <= 1e-5 |q_j| |k_s|, against a bound of 127 * 2^-24 |q_j| |k_s|) is
// recomputed in fp64, which is exact for products of e4m3 codes.
#include <cfloat>

#include "launch.h"

namespace dsa {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 64;    // candidate entries per tile
constexpr int kHeads = 64;   // head slots (heads beyond H_I have w = 0)

template <int DIM>
struct Smem {
  static constexpr int LD = DIM + 4;   // padded row: conflict-free float4 reads across rows
  static size_t bytes(int kk) {
    return sizeof(float) * (2 * kHeads * LD) + sizeof(float) * kk + sizeof(uint64_t) * kk;
  }
};

// Row `row` of the key cache, decoded (unscaled) into a shared row; threads
// cover 16-code (FP8) or 4-float (F32) pieces.
template <bool FP8, int DIM>
__device__ __forceinline__ void load_keys(const void* k, const int64_t* rows, float* kt) {
  constexpr int LD = Smem<DIM>::LD;
  if constexpr (FP8) {
    constexpr int C = DIM / 16;
    for (int c = threadIdx.x; c < kTile * C; c += kThreads) {
      const int r = c / C, ch = c % C;
      float* dst = kt + r * LD + ch * 16;
      const int64_t row = rows[r];
      if (row < 0) {
#pragma unroll
        for (int e = 0; e < 16; ++e) dst[e] = 0.f;
        continue;
      }
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(k) + row * DIM) + ch);
      const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 a = fp8x2_e4m3_to_float2((uint16_t)(wd[q] & 0xFFFF));
        const float2 b = fp8x2_e4m3_to_float2((uint16_t)(wd[q] >> 16));
        dst[4 * q] = a.x;
        dst[4 * q + 1] = a.y;
        dst[4 * q + 2] = b.x;
        dst[4 * q + 3] = b.y;
      }
    }
  } else {
    constexpr int C = DIM / 4;
    for (int c = threadIdx.x; c < kTile * C; c += kThreads) {
      const int r = c / C, ch = c % C;
      const int64_t row = rows[r];
      const float4 v = row < 0 ? make_float4(0.f, 0.f, 0.f, 0.f)
                               : __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(k) + row * DIM) + ch);
      *reinterpret_cast<float4*>(kt + r * LD + 4 * ch) = v;
    }
  }
}

// Euclidean norms of 64 shared rows (4 threads a row).
template <int DIM>
__device__ __forceinline__ void row_norms(const float* rows, float* out) {
  constexpr int LD = Smem<DIM>::LD;
  const int r = threadIdx.x >> 2, part = threadIdx.x & 3;
  float s = 0.f;
#pragma unroll 8
  for (int d = part * (DIM / 4); d < (part + 1) * (DIM / 4); ++d) s = fmaf(rows[r * LD + d], rows[r * LD + d], s);
  s += __shfl_xor_sync(0xffffffffu, s, 1);
  s += __shfl_xor_sync(0xffffffffu, s, 2);
  if (part == 0) out[r] = sqrtf(s);
}

__device__ __forceinline__ float block_sum(float v, float* scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) t += scratch[w];
  return t;
}

__device__ __forceinline__ float block_max(float v, float* scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = -INFINITY;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) t = fmaxf(t, scratch[w]);
  return t;
}

template <bool FP8, int DIM>
__global__ void __launch_bounds__(kThreads, 2)
indexer_kl_bwd_kernel(QueryBatch qb, CacheMap cm, int heads, const void* __restrict__ q,
                      const float* __restrict__ q_scale, const float* __restrict__ w, const void* __restrict__ k,
                      const float* __restrict__ k_scale, const int32_t* __restrict__ idx, int kk,
                      const float* __restrict__ p, float* __restrict__ loss, float* __restrict__ grad_scores,
                      float* __restrict__ dw, float* __restrict__ dq, float* __restrict__ dk, int* err) {
  constexpr int LD = Smem<DIM>::LD;
  extern __shared__ __align__(16) float sm[];
  float* qs = sm;                                                     // [64][LD] decoded q rows
  float* kt = qs + kHeads * LD;                                       // [64][LD] decoded key tile
  float* Ie = kt + kTile * LD;                                        // [kk] I, then g
  uint64_t* msk = reinterpret_cast<uint64_t*>(Ie + ((kk + 1) & ~1));  // [kk] head masks
  __shared__ float qn[kHeads], wv[kHeads], sqv[kHeads], kn[kTile], ksc[kTile], ps[kTile];
  __shared__ int64_t krow[kTile];
  __shared__ float red[kThreads / 32][kTile];
  __shared__ float scratch[kThreads / 32];

  const int t = blockIdx.x, tid = threadIdx.x;
  const int pos = __ldg(qb.q_pos + t), seq = __ldg(qb.q_seq + t);
  const bool qok = pos >= 0 && pos < qb.max_kv;
  if (!qok) {
    if (tid == 0) {
      flag_error(err, DSA_ERR_BOUNDS);
      loss[t] = 0.f;
    }
    for (int j = tid; j < heads; j += kThreads) dw[(int64_t)t * heads + j] = 0.f;
    for (int e = tid; e < heads * DIM; e += kThreads) dq[(int64_t)t * heads * DIM + e] = 0.f;
    if (grad_scores)
      for (int e = tid; e < kk; e += kThreads) grad_scores[(int64_t)t * kk + e] = 0.f;
    return;
  }
  const int32_t* irow = idx + (int64_t)t * kk;
  const float* prow = p + (int64_t)t * kk;

  // ---- the query's heads, decoded (unscaled), and their weights and scales
  for (int e = tid; e < kHeads * DIM; e += kThreads) {
    const int j = e / DIM, d = e % DIM;
    float v = 0.f;
    if (j < heads) {
      if constexpr (FP8) {
        const uint8_t c = __ldg(static_cast<const uint8_t*>(q) + ((int64_t)t * heads + j) * DIM + d);
        v = fp8x2_e4m3_to_float2((uint16_t)c).x;
      } else {
        v = __ldg(static_cast<const float*>(q) + ((int64_t)t * heads + j) * DIM + d);
      }
    }
    qs[j * LD + d] = v;
  }
  if (tid < kHeads) {
    wv[tid] = tid < heads ? __ldg(w + (int64_t)t * heads + tid) : 0.f;
    sqv[tid] = tid < heads && q_scale ? __ldg(q_scale + (int64_t)t * heads + tid) : 1.f;
  }
  for (int e = tid; e < kk; e += kThreads) msk[e] = 0ull;
  __syncthreads();
  row_norms<DIM>(qs, qn);

  // pass 1: thread (jg, kg) takes heads 4jg .. 4jg+3 and the tile's entries
  // kg, kg+16, kg+32, kg+48 (rows 16 apart fall in different shared-memory
  // banks, so a warp's 16 key-row reads do not collide)
  const int jg = tid >> 4, kg = tid & 15;
  const int h0 = 4 * jg;
  auto U = [&](int b) { return kg + 16 * b; };
  float A[4] = {0.f, 0.f, 0.f, 0.f}, B[4] = {0.f, 0.f, 0.f, 0.f};
  float M = -INFINITY, Z = 0.f;             // running maximum of I and sum of exp(I - M)

  auto tile_rows = [&](int e0) {
    if (tid < kTile) {
      const int e = e0 + tid;
      int64_t row = -1;
      float sc = 0.f;
      if (e < kk) {
        const int s = __ldg(irow + e);
        if (s >= 0 && s <= pos) {
          row = cache_row(cm, seq, s, err);
          if (row >= 0) sc = k_scale ? __ldg(k_scale + row) : 1.f;
        } else if (s != -1) {
          flag_error(err, DSA_ERR_BOUNDS);
        }
      }
      krow[tid] = row;
      ksc[tid] = sc;
    }
  };

  // ---------------------------------------------------------------- pass 1
  for (int e0 = 0; e0 < kk; e0 += kTile) {
    tile_rows(e0);
    if (tid < kTile) ps[tid] = (e0 + tid < kk) ? __ldg(prow + e0 + tid) : 0.f;
    __syncthreads();
    load_keys<FP8, DIM>(k, krow, kt);
    __syncthreads();
    row_norms<DIM>(kt, kn);
    float x[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) x[a][b] = 0.f;
#pragma unroll 4
    for (int d = 0; d < DIM; d += 4) {
      float4 qv[4], kv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) qv[a] = *reinterpret_cast<const float4*>(qs + (h0 + a) * LD + d);
#pragma unroll
      for (int b = 0; b < 4; ++b) kv[b] = *reinterpret_cast<const float4*>(kt + U(b) * LD + d);
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          x[a][b] = fmaf(qv[a].x, kv[b].x, x[a][b]);
          x[a][b] = fmaf(qv[a].y, kv[b].y, x[a][b]);
          x[a][b] = fmaf(qv[a].z, kv[b].z, x[a][b]);
          x[a][b] = fmaf(qv[a].w, kv[b].w, x[a][b]);
        }
    }
    __syncthreads();   // kn written
    float r[4][4], ipart[4] = {0.f, 0.f, 0.f, 0.f};
    uint32_t nib[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        float xv = x[a][b];
        const float bound = 1e-5f * qn[h0 + a] * kn[U(b)];
        bool posv = xv > 0.f;
        if (bound > 0.f && fabsf(xv) <= bound) {   // near zero: decide the sign exactly
          // four independent fp64 chains; every partial sum of e4m3
          // products is exact in fp64, so the order does not matter
          double acc[4] = {0.0, 0.0, 0.0, 0.0};
          const float* qa = qs + (h0 + a) * LD;
          const float* kb = kt + U(b) * LD;
          for (int d = 0; d < DIM; d += 4)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[c] = fma((double)qa[d + c], (double)kb[d + c], acc[c]);
          const double tot = (acc[0] + acc[1]) + (acc[2] + acc[3]);
          posv = tot > 0.0;
          xv = (float)tot;
        }
        r[a][b] = posv ? xv * sqv[h0 + a] * ksc[U(b)] : 0.f;
        if (posv) nib[b] |= 1u << a;
        ipart[b] = fmaf(wv[h0 + a], r[a][b], ipart[b]);
      }
    // I of the tile: sum over the 16 head groups (two per warp, then the warps)
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      ipart[b] += __shfl_xor_sync(0xffffffffu, ipart[b], 16);
      nib[b] |= __shfl_xor_sync(0xffffffffu, nib[b], 16) << 4;
    }
    if ((tid & 31) < 16) {
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        red[tid >> 5][U(b)] = ipart[b];
        if (nib[b] && e0 + U(b) < kk)
          atomicOr(reinterpret_cast<unsigned long long*>(msk + e0 + U(b)),
                   (unsigned long long)nib[b] << (8 * (tid >> 5)));
      }
    }
    __syncthreads();
    float iv = -INFINITY;
    if (tid < kTile) {
      if (krow[tid] >= 0) {
        iv = 0.f;
#pragma unroll
        for (int wq = 0; wq < kThreads / 32; ++wq) iv += red[wq][tid];
      }
      if (e0 + tid < kk) Ie[e0 + tid] = iv;
      red[0][tid] = iv;   // read back below (after the max)
    }
    const float tmax = block_max(tid < kTile ? iv : -INFINITY, scratch);
    const float Mn = fmaxf(M, tmax);
    if (Mn != -INFINITY) {
      const float alpha = M == -INFINITY ? 0.f : __expf(M - Mn);
      float ex[4], pb[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const float ib = red[0][U(b)];
        ex[b] = ib == -INFINITY ? 0.f : __expf(ib - Mn);
        pb[b] = krow[U(b)] >= 0 ? ps[U(b)] : 0.f;
      }
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        A[a] *= alpha;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          A[a] = fmaf(ex[b], r[a][b], A[a]);
          B[a] = fmaf(pb[b], r[a][b], B[a]);
        }
      }
      const float zt = block_sum(tid < kTile && iv != -INFINITY ? __expf(iv - Mn) : 0.f, scratch);
      Z = Z * alpha + zt;
      M = Mn;
    }
    __syncthreads();   // kt, red and ps are rewritten by the next tile
  }

  // ---------------------------------------------------------------- pi, g, loss, dw
  const float logZ = logf(Z);
  float lpart = 0.f;
  for (int e = tid; e < kk; e += kThreads) {
    const float iv = Ie[e];
    float g = 0.f;
    if (iv != -INFINITY) {
      const float lpi = iv - M - logZ;
      const float pe = __ldg(prow + e);
      g = __expf(lpi) - pe;
      if (pe > 0.f) lpart += pe * (logf(pe) - lpi);
    }
    Ie[e] = g;
    if (grad_scores) grad_scores[(int64_t)t * kk + e] = g;
  }
  const float lsum = block_sum(lpart, scratch);
  if (tid == 0) loss[t] = M == -INFINITY ? 0.f : lsum;
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    float av = A[a], bv = B[a];
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
      av += __shfl_xor_sync(0xffffffffu, av, o);
      bv += __shfl_xor_sync(0xffffffffu, bv, o);
    }
    if (kg == 0 && h0 + a < heads) dw[(int64_t)t * heads + h0 + a] = M == -INFINITY ? 0.f : av / Z - bv;
  }
  __syncthreads();

  // ---------------------------------------------------------------- pass 2: dq and dk
  // Register-blocked so that one shared-memory load feeds 8 FMAs per lane:
  //   dq: warp w owns heads 8w .. 8w+7, lane l the dims DL*l .. DL*l+DL-1;
  //       per entry it loads its DL key values and the entry's mask word;
  //   dk: warp w owns the tile's entries 8w .. 8w+7 (their masks held in
  //       registers), lane l the same dims; per head it loads DL values of q.
  constexpr int DL = DIM / 32;
  const int warp = tid >> 5, lane = tid & 31;
  float accq[8][DL];
#pragma unroll
  for (int h = 0; h < 8; ++h)
#pragma unroll
    for (int c = 0; c < DL; ++c) accq[h][c] = 0.f;
  for (int e0 = 0; e0 < kk; e0 += kTile) {
    tile_rows(e0);
    __syncthreads();
    load_keys<FP8, DIM>(k, krow, kt);
    __syncthreads();
    const int nu = min(kTile, kk - e0);
    // dq_j += g_s sk_s [x_js > 0] k8_s
    for (int u = 0; u < nu; ++u) {
      const uint32_t bits = (uint32_t)(msk[e0 + u] >> (8 * warp)) & 0xFFu;
      if (!bits) continue;                                   // warp-uniform
      const float gs = Ie[e0 + u] * ksc[u];
      float kv[DL];
#pragma unroll
      for (int c = 0; c < DL; ++c) kv[c] = kt[u * LD + DL * lane + c];
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const float cf = (bits >> h) & 1u ? gs : 0.f;
#pragma unroll
        for (int c = 0; c < DL; ++c) accq[h][c] = fmaf(cf, kv[c], accq[h][c]);
      }
    }
    // dk_s += g_s sum_j w_j sq_j [x_js > 0] q8_j
    {
      uint64_t mk[8];
      uint64_t any = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int u = 8 * warp + e;
        mk[e] = (u < nu && krow[u] >= 0) ? msk[e0 + u] : 0ull;
        any |= mk[e];
      }
      if (any) {                                             // warp-uniform
        float acck[8][DL];
#pragma unroll
        for (int e = 0; e < 8; ++e)
#pragma unroll
          for (int c = 0; c < DL; ++c) acck[e][c] = 0.f;
        for (int j = 0; j < kHeads; ++j) {
          const float cj = wv[j] * sqv[j];
          float qv[DL];
#pragma unroll
          for (int c = 0; c < DL; ++c) qv[c] = qs[j * LD + DL * lane + c];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float cf = (mk[e] >> j) & 1ull ? cj : 0.f;
#pragma unroll
            for (int c = 0; c < DL; ++c) acck[e][c] = fmaf(cf, qv[c], acck[e][c]);
          }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (!mk[e]) continue;
          const int u = 8 * warp + e;
          const float gs = Ie[e0 + u];
          float* dst = dk + krow[u] * DIM + DL * lane;
          if constexpr (DL == 4)
            atomicAdd(reinterpret_cast<float4*>(dst),
                      make_float4(gs * acck[e][0], gs * acck[e][1], gs * acck[e][2], gs * acck[e][3]));
          else if constexpr (DL == 2)
            atomicAdd(reinterpret_cast<float2*>(dst), make_float2(gs * acck[e][0], gs * acck[e][1]));
          else
            atomicAdd(dst, gs * acck[e][0]);
        }
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    const int j = 8 * warp + h;
    if (j >= heads) continue;
    float* dst = dq + ((int64_t)t * heads + j) * DIM + DL * lane;
    const float wj = wv[j];
#pragma unroll
    for (int c = 0; c < DL; ++c) dst[c] = wj * accq[h][c];
  }
}

template <bool FP8, int DIM>
cudaError_t launch_t(const QueryBatch& qb, const CacheMap& cm, const dsa_indexer_inputs& ix, const int32_t* idx,
                     int kk, const float* p, float* loss, float* grad_scores, float* dw, float* dq, float* dk,
                     int* err, cudaStream_t stream) {
  const size_t smem = Smem<DIM>::bytes(kk) + 8;
  auto kern = indexer_kl_bwd_kernel<FP8, DIM>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<qb.num_q, kThreads, smem, stream>>>(qb, cm, ix.heads, ix.q, ix.q_scale, ix.w, ix.k, ix.k_scale, idx, kk,
                                             p, loss, grad_scores, dw, dq, dk, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_indexer_kl_bwd(const QueryBatch& qb, const CacheMap& cm, const dsa_indexer_inputs& ix,
                                  const int32_t* idx, int k, const float* p, float* loss, float* grad_scores,
                                  float* dw, float* dq, float* dk, int* err, cudaStream_t stream) {
  if (indexer_kl_bwd_tc_supported(ix))
    return launch_indexer_kl_bwd_tc(qb, cm, ix, idx, k, p, loss, grad_scores, dw, dq, dk, err, stream);
  const bool fp8 = ix.dtype == DSA_FP8_E4M3;
  switch (ix.dim) {
    case 32:
      return fp8 ? launch_t<true, 32>(qb, cm, ix, idx, k, p, loss, grad_scores, dw, dq, dk, err, stream)
                 : launch_t<false, 32>(qb, cm, ix, idx, k, p, loss, grad_scores, dw, dq, dk, err, stream);
    case 64:
      return fp8 ? launch_t<true, 64>(qb, cm, ix, idx, k, p, loss, grad_scores, dw, dq, dk, err, stream)
                 : launch_t<false, 64>(qb, cm, ix, idx, k, p, loss, grad_scores, dw, dq, dk, err, stream);
    default:
      return fp8 ? launch_t<true, 128>(qb, cm, ix, idx, k, p, loss, grad_scores, dw, dq, dk, err, stream)
                 : launch_t<false, 128>(qb, cm, ix, idx, k, p, loss, grad_scores, dw, dq, dk, err, stream);
  }
}

}  // namespace dsa
