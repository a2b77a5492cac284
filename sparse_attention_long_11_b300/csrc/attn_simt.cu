// Sparse MQA attention on CUDA cores (every dtype/shape the ABI accepts).
//
// O[t,h,:] = sum_{s in sel(t)} softmax_s(scale * <q[t,h,:], kv[s,:]>) kv[s,:d_v]
// over the selected positions only (DeepSeek-V3.2 summary card, "How DSA
// Works": full attention computed only on the selected tokens; news article
// on DeepSeek-V3.2: multi-query / latent attention over the sparse set, all
// heads sharing one KV row).
//
// One block = one query x 8 heads (one warp per head).  The selected rows
// are gathered 32 at a time into shared memory (fp32, padded rows); lane j
// of a warp scores row j, the warp keeps an online softmax (running max m,
// running sum l) and each lane accumulates d_v/32 output columns.
#include "launch.h"

namespace dsa {
namespace {

constexpr int kThreads = 256;
constexpr int kHeadsPerBlock = 8;
constexpr int kTile = 32;
constexpr int kMaxCols = 16;   // d_v / 32 <= 16

template <typename T>
__device__ __forceinline__ void load4(const T* p, float* dst);
template <>
__device__ __forceinline__ void load4<float>(const float* p, float* dst) {
  float4 v = __ldg(reinterpret_cast<const float4*>(p));
  dst[0] = v.x; dst[1] = v.y; dst[2] = v.z; dst[3] = v.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16* p, float* dst) {
  uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
  dst[0] = __uint_as_float(v.x << 16); dst[1] = __uint_as_float(v.x & 0xFFFF0000u);
  dst[2] = __uint_as_float(v.y << 16); dst[3] = __uint_as_float(v.y & 0xFFFF0000u);
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
attn_simt_kernel(QueryBatch qb, CacheMap cm, int H, int d_qk, int d_v, const T* __restrict__ q,
                 const T* __restrict__ kv, const int32_t* __restrict__ idx, int k, float scale,
                 T* __restrict__ out, float* __restrict__ lse, int* err) {
  extern __shared__ float4 smem4[];
  const int ld = d_qk + 1;                                 // odd stride: conflict-free column reads
  float* q_s = reinterpret_cast<float*>(smem4);            // [8][d_qk]
  float* kv_s = q_s + kHeadsPerBlock * d_qk;               // [32][ld]
  float* p_s = kv_s + kTile * ld;                          // [8][32]
  int64_t* rows_s = reinterpret_cast<int64_t*>(p_s + kHeadsPerBlock * kTile + 2);  // [32]
  rows_s = reinterpret_cast<int64_t*>((reinterpret_cast<uintptr_t>(rows_s) + 7) & ~uintptr_t(7));

  const int i = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.y * kHeadsPerBlock + warp;
  const int pos = __ldg(qb.q_pos + i);
  const int seq = __ldg(qb.q_seq + i);
  const bool qok = pos >= 0 && pos < qb.max_kv;
  if (!qok && tid == 0 && blockIdx.y == 0) flag_error(err, DSA_ERR_BOUNDS);

  const T* qp = q + ((int64_t)i * H + blockIdx.y * kHeadsPerBlock) * d_qk;
  for (int e = tid * 4; e < kHeadsPerBlock * d_qk; e += kThreads * 4) load4<T>(qp + e, q_s + e);

  float o[kMaxCols];
#pragma unroll
  for (int c = 0; c < kMaxCols; ++c) o[c] = 0.f;
  float m = -INFINITY, l = 0.f;
  const int ncols = d_v / 32 + (lane < d_v % 32 ? 1 : 0);

  for (int t0 = 0; t0 < k; t0 += kTile) {
    if (tid < kTile) {
      int64_t row = -1;
      if (qok && t0 + tid < k) {
        const int s = __ldg(idx + (int64_t)i * k + t0 + tid);
        if (s >= 0 && s <= pos) row = cache_row(cm, seq, s, err);
        else if (s != -1) flag_error(err, DSA_ERR_BOUNDS);
      }
      rows_s[tid] = row;
    }
    __syncthreads();
    for (int e = tid * 4; e < kTile * d_qk; e += kThreads * 4) {
      const int r = e / d_qk, d = e - r * d_qk;
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      const int64_t row = rows_s[r];
      if (row >= 0) load4<T>(kv + row * d_qk + d, v);
      float* dst = kv_s + r * ld + d;
      dst[0] = v[0]; dst[1] = v[1]; dst[2] = v[2]; dst[3] = v[3];
    }
    __syncthreads();
    float sc = -INFINITY;
    if (rows_s[lane] >= 0) {
      const float* qh = q_s + warp * d_qk;
      const float* kr = kv_s + lane * ld;
      float a0 = 0.f, a1 = 0.f;
      for (int d = 0; d < d_qk; d += 2) {
        a0 = fmaf(qh[d], kr[d], a0);
        a1 = fmaf(qh[d + 1], kr[d + 1], a1);
      }
      sc = (a0 + a1) * scale;
    }
    float tmax = sc;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
    const float m_new = fmaxf(m, tmax);
    float alpha, p;
    if (m_new == -INFINITY) {           // nothing selected so far
      alpha = 1.f;
      p = 0.f;
    } else {
      alpha = expf(m - m_new);          // m = -inf -> 0
      p = expf(sc - m_new);             // sc = -inf -> 0
    }
    float psum = p;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
    l = l * alpha + psum;
    m = m_new;
    p_s[warp * kTile + lane] = p;
    __syncwarp();
#pragma unroll
    for (int c = 0; c < kMaxCols; ++c) {
      if (c < ncols) {
        const int d = lane + 32 * c;
        float acc = o[c] * alpha;
        for (int j = 0; j < kTile; ++j) acc = fmaf(p_s[warp * kTile + j], kv_s[j * ld + d], acc);
        o[c] = acc;
      }
    }
    __syncthreads();
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  T* op = out + ((int64_t)i * H + h) * d_v;
#pragma unroll
  for (int c = 0; c < kMaxCols; ++c) {
    if (c < ncols) {
      const float v = o[c] * inv;
      if constexpr (sizeof(T) == 2) op[lane + 32 * c] = __float2bfloat16_rn(v);
      else op[lane + 32 * c] = v;
    }
  }
  if (lane == 0) lse[(int64_t)i * H + h] = l > 0.f ? m + logf(l) : -INFINITY;
}

template <typename T>
cudaError_t launch_t(const QueryBatch& qb, const CacheMap& cm, const dsa_attn_inputs& at,
                     const int32_t* idx, int k, void* out, float* lse, int* err, cudaStream_t stream) {
  size_t smem = sizeof(float) * ((size_t)kHeadsPerBlock * at.d_qk + (size_t)kTile * (at.d_qk + 1) +
                                 kHeadsPerBlock * kTile + 4) + sizeof(int64_t) * (kTile + 1);
  auto kern = attn_simt_kernel<T>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(qb.num_q, at.heads / kHeadsPerBlock);
  kern<<<grid, kThreads, smem, stream>>>(qb, cm, at.heads, at.d_qk, at.d_v, static_cast<const T*>(at.q),
                                         static_cast<const T*>(at.kv), idx, k, at.softmax_scale,
                                         static_cast<T*>(out), lse, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_simt(const QueryBatch& qb, const CacheMap& cm, const dsa_attn_inputs& at,
                             const int32_t* idx, int k, void* out, float* lse, int* err,
                             cudaStream_t stream) {
  if (at.dtype == DSA_BF16) return launch_t<__nv_bfloat16>(qb, cm, at, idx, k, out, lse, err, stream);
  return launch_t<float>(qb, cm, at, idx, k, out, lse, err, stream);
}

}  // namespace dsa
