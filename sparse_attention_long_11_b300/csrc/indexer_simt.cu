// Lightning indexer on CUDA cores (every dtype/shape the ABI accepts).
//
// Computes I[t,s] = sum_j w[t,j] * ReLU(sq[t,j] * sk[s] * <q_I[t,j,:], k_I[s,:]>)
// for keys s <= t (DeepSeek-V3.2 summary card, "How DSA Works": the
// lightning indexer scores each query against all keys; news article on
// DeepSeek-V3.2, sparse-attention section: a few low-precision heads on
// every token pair).  Because sq, sk > 0, ReLU(sq*sk*x) = sq*sk*ReLU(x): the
// query scale is folded into the head weight and the key scale is applied
// after the head sum.
//
// One block = one query x 128 consecutive keys, one thread per key.  The
// query's heads sit decoded in shared memory (broadcast reads); the key row
// sits decoded in registers.
#include "launch.h"

namespace dsa {
namespace {

constexpr int kKeysPerBlock = 128;

template <bool FP8, int DIM>
__device__ __forceinline__ void load_key(const void* k, int64_t row, float (&kr)[DIM]) {
  if constexpr (FP8) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(k) + row * DIM);
#pragma unroll
    for (int c = 0; c < DIM / 16; ++c) {
      uint4 v = __ldg(p + c);
      uint32_t wds[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float2 a = fp8x2_e4m3_to_float2((uint16_t)(wds[q] & 0xFFFF));
        float2 b = fp8x2_e4m3_to_float2((uint16_t)(wds[q] >> 16));
        kr[c * 16 + q * 4 + 0] = a.x;
        kr[c * 16 + q * 4 + 1] = a.y;
        kr[c * 16 + q * 4 + 2] = b.x;
        kr[c * 16 + q * 4 + 3] = b.y;
      }
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(k) + row * DIM);
#pragma unroll
    for (int c = 0; c < DIM / 4; ++c) {
      float4 v = __ldg(p + c);
      kr[4 * c] = v.x; kr[4 * c + 1] = v.y; kr[4 * c + 2] = v.z; kr[4 * c + 3] = v.w;
    }
  }
}

template <bool FP8, int DIM>
__global__ void __launch_bounds__(kKeysPerBlock)
indexer_simt_kernel(QueryBatch qb, CacheMap cm, int heads, const void* __restrict__ q,
                    const float* __restrict__ q_scale, const float* __restrict__ w,
                    const void* __restrict__ k, const float* __restrict__ k_scale,
                    float* __restrict__ scores, int64_t ld, int* err) {
  extern __shared__ float4 smem4[];
  float* q_s = reinterpret_cast<float*>(smem4);   // [heads][DIM]
  float* wq_s = q_s + heads * DIM;                // [heads]: w * sq

  const int i = blockIdx.x;
  const int s = blockIdx.y * kKeysPerBlock + threadIdx.x;
  const int pos = __ldg(qb.q_pos + i);
  const int seq = __ldg(qb.q_seq + i);
  const bool qok = pos >= 0 && pos < qb.max_kv;
  if (!qok && blockIdx.y == 0 && threadIdx.x == 0) flag_error(err, DSA_ERR_BOUNDS);
  float* out = scores + (int64_t)i * ld;

  if (!qok || (int)(blockIdx.y * kKeysPerBlock) > pos) {   // whole tile masked
    if (s < qb.max_kv) out[s] = -INFINITY;
    return;
  }
  const int64_t qoff = (int64_t)i * heads * DIM;
  if constexpr (FP8) {
    const uint16_t* qp = reinterpret_cast<const uint16_t*>(static_cast<const uint8_t*>(q) + qoff);
    for (int e = threadIdx.x; e < heads * DIM / 2; e += kKeysPerBlock) {
      float2 v = fp8x2_e4m3_to_float2(__ldg(qp + e));
      q_s[2 * e] = v.x;
      q_s[2 * e + 1] = v.y;
    }
  } else {
    const float* qp = static_cast<const float*>(q) + qoff;
    for (int e = threadIdx.x; e < heads * DIM; e += kKeysPerBlock) q_s[e] = __ldg(qp + e);
  }
  for (int h = threadIdx.x; h < heads; h += kKeysPerBlock)
    wq_s[h] = __ldg(w + (int64_t)i * heads + h) * (FP8 ? __ldg(q_scale + (int64_t)i * heads + h) : 1.0f);
  __syncthreads();

  if (s >= qb.max_kv) return;
  if (s > pos) {
    out[s] = -INFINITY;
    return;
  }
  const int64_t row = cache_row(cm, seq, s, err);
  if (row < 0) {
    out[s] = -INFINITY;
    return;
  }
  float kr[DIM];
  load_key<FP8, DIM>(k, row, kr);
  float acc = 0.f;
  for (int h = 0; h < heads; ++h) {
    const float4* qh = reinterpret_cast<const float4*>(q_s + h * DIM);
    float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
#pragma unroll
    for (int c = 0; c < DIM / 4; ++c) {
      float4 qv = qh[c];
      d0 = fmaf(qv.x, kr[4 * c], d0);
      d1 = fmaf(qv.y, kr[4 * c + 1], d1);
      d2 = fmaf(qv.z, kr[4 * c + 2], d2);
      d3 = fmaf(qv.w, kr[4 * c + 3], d3);
    }
    acc = fmaf(wq_s[h], fmaxf((d0 + d1) + (d2 + d3), 0.f), acc);
  }
  if constexpr (FP8) acc *= __ldg(k_scale + row);
  out[s] = acc;
}

template <bool FP8, int DIM>
cudaError_t launch_t(const QueryBatch& qb, const CacheMap& cm, const dsa_indexer_inputs& ix,
                     float* scores, int64_t ld, int* err, cudaStream_t stream) {
  size_t smem = (size_t)ix.heads * DIM * sizeof(float) + (size_t)ix.heads * sizeof(float);
  auto kern = indexer_simt_kernel<FP8, DIM>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(qb.num_q, (qb.max_kv + kKeysPerBlock - 1) / kKeysPerBlock);
  kern<<<grid, kKeysPerBlock, smem, stream>>>(qb, cm, ix.heads, ix.q, ix.q_scale, ix.w, ix.k, ix.k_scale,
                                              scores, ld, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_indexer_simt(const QueryBatch& qb, const CacheMap& cm, const dsa_indexer_inputs& ix,
                                float* scores, int64_t ld, int* err, cudaStream_t stream) {
  const bool fp8 = ix.dtype == DSA_FP8_E4M3;
  switch (ix.dim) {
    case 32: return fp8 ? launch_t<true, 32>(qb, cm, ix, scores, ld, err, stream)
                        : launch_t<false, 32>(qb, cm, ix, scores, ld, err, stream);
    case 64: return fp8 ? launch_t<true, 64>(qb, cm, ix, scores, ld, err, stream)
                        : launch_t<false, 64>(qb, cm, ix, scores, ld, err, stream);
    default: return fp8 ? launch_t<true, 128>(qb, cm, ix, scores, ld, err, stream)
                        : launch_t<false, 128>(qb, cm, ix, scores, ld, err, stream);
  }
}

}  // namespace dsa
