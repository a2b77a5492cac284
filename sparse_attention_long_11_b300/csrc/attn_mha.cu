// Sparse attention in the per-head (non-absorbed) form: the prefill
// attention mode.  Susan Zhang's thread on the DeepSeek-V3.2 write-up names
// separate attention modes for disaggregated prefill and decode; the decode
// mode is the latent MQA of attn_tc.cu (one shared 576-wide row per key),
// this one gives every head its own key and value rows:
//   O[t,h,:] = sum_{s in sel(t)} softmax_s(scale * (<q_n[t,h], k_n[s,h]> + <q_r[t,h], k_r[s]>)) v[s,h,:]
// with k_n [rows, H, 128] and v [rows, H, 128] per head and k_r [rows, 64]
// shared by all heads (the rope part), bf16.
//
// A selected pair moves 128 heads x (128 + 128) x 2 + 64 x 2 = 65,664 bytes
// of rows, against 1,152 for the latent row, and every query gathers its own
// keys, so the mode is bound by the gathers, not by a contraction: one warp
// per (query, head); lane l holds dims 4l..4l+3 of the head's key and value
// and dims 2l, 2l+1 of the rope part, so each gathered row is one coalesced
// 256-byte (128-byte for the rope) warp load.  Loads of 8 selected keys are
// issued before their dot products; the softmax is online and exact (fp32,
// exp2f), the output bf16.
#include <cmath>

#include "launch.h"

namespace dsa {
namespace {

constexpr int kWarpsPerBlock = 8;   // heads per block
constexpr int kDn = 128, kDr = 64, kDv = 128;
constexpr int kBatch = 8;           // selected keys whose loads are in flight together

__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
attn_mha_kernel(QueryBatch qb, CacheMap cm, int H, const __nv_bfloat16* __restrict__ q,
                const __nv_bfloat16* __restrict__ kn, const __nv_bfloat16* __restrict__ kr,
                const __nv_bfloat16* __restrict__ v, const int32_t* __restrict__ idx, int k, float scale_log2,
                __nv_bfloat16* __restrict__ out, float* __restrict__ lse, int* err) {
  const int i = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * kWarpsPerBlock + warp;
  const int pos = __ldg(qb.q_pos + i), seq = __ldg(qb.q_seq + i);
  uint2* orow = reinterpret_cast<uint2*>(out + ((int64_t)i * H + h) * kDv) + lane;
  if (pos < 0 || pos >= qb.max_kv) {
    if (lane == 0 && h == 0) flag_error(err, DSA_ERR_BOUNDS);
    *orow = make_uint2(0u, 0u);
    if (lane == 0) lse[(int64_t)i * H + h] = -INFINITY;
    return;
  }
  // this lane's query dims, in base-2 logit units
  const __nv_bfloat16* qrow = q + ((int64_t)i * H + h) * (kDn + kDr);
  const uint2 qa = __ldg(reinterpret_cast<const uint2*>(qrow) + lane);
  const uint32_t qb2 = __ldg(reinterpret_cast<const uint32_t*>(qrow + kDn) + lane);
  const float2 q01 = bf16x2_to_f2(qa.x), q23 = bf16x2_to_f2(qa.y), qr = bf16x2_to_f2(qb2);
  const float qn[4] = {q01.x * scale_log2, q01.y * scale_log2, q23.x * scale_log2, q23.y * scale_log2};
  const float qr0 = qr.x * scale_log2, qr1 = qr.y * scale_log2;

  float m = -INFINITY, l = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
  const int32_t* irow = idx + (int64_t)i * k;
  for (int e0 = 0; e0 < k; e0 += 32) {
    // the physical row of this lane's entry (-1: padding or out of range)
    int row = -1;
    if (e0 + lane < k) {
      const int s = __ldg(irow + e0 + lane);
      if (s >= 0 && s <= pos) row = (int)cache_row(cm, seq, s, err);
      else if (s != -1) flag_error(err, DSA_ERR_BOUNDS);
    }
#pragma unroll 1
    for (int b = 0; b < 32; b += kBatch) {
      uint2 kv4[kBatch], vv4[kBatch];
      uint32_t kr2[kBatch];
      int rw[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        rw[u] = __shfl_sync(0xffffffffu, row, b + u);
        if (rw[u] >= 0) {
          kv4[u] = __ldg(reinterpret_cast<const uint2*>(kn + ((int64_t)rw[u] * H + h) * kDn) + lane);
          vv4[u] = __ldg(reinterpret_cast<const uint2*>(v + ((int64_t)rw[u] * H + h) * kDv) + lane);
          kr2[u] = __ldg(reinterpret_cast<const uint32_t*>(kr + (int64_t)rw[u] * kDr) + lane);
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (rw[u] < 0) continue;   // warp-uniform (a broadcast row)
        const float2 k01 = bf16x2_to_f2(kv4[u].x), k23 = bf16x2_to_f2(kv4[u].y), kr01 = bf16x2_to_f2(kr2[u]);
        float x = qn[0] * k01.x;
        x = fmaf(qn[1], k01.y, x);
        x = fmaf(qn[2], k23.x, x);
        x = fmaf(qn[3], k23.y, x);
        x = fmaf(qr0, kr01.x, x);
        x = fmaf(qr1, kr01.y, x);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        if (x > m) {   // the maximum moves: rescale what has been summed
          const float a = exp2f(m - x);
          l *= a;
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[c] *= a;
          m = x;
        }
        const float p = exp2f(x - m);
        l += p;
        const float2 v01 = bf16x2_to_f2(vv4[u].x), v23 = bf16x2_to_f2(vv4[u].y);
        acc[0] = fmaf(p, v01.x, acc[0]);
        acc[1] = fmaf(p, v01.y, acc[1]);
        acc[2] = fmaf(p, v23.x, acc[2]);
        acc[3] = fmaf(p, v23.y, acc[3]);
      }
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const __nv_bfloat162 o01 = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
  const __nv_bfloat162 o23 = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
  *orow = make_uint2(*reinterpret_cast<const uint32_t*>(&o01), *reinterpret_cast<const uint32_t*>(&o23));
  if (lane == 0) lse[(int64_t)i * H + h] = l > 0.f ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
}

}  // namespace

cudaError_t launch_attn_mha(const QueryBatch& qb, const CacheMap& cm, int heads, const void* q, const void* k_nope,
                            const void* k_rope, const void* v, float softmax_scale, const int32_t* idx, int k,
                            void* out, float* lse, int* err, cudaStream_t stream) {
  const dim3 grid(qb.num_q, heads / kWarpsPerBlock);
  const float scale_log2 = (float)((double)softmax_scale * 1.4426950408889634);
  attn_mha_kernel<<<grid, kWarpsPerBlock * 32, 0, stream>>>(
      qb, cm, heads, static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k_nope),
      static_cast<const __nv_bfloat16*>(k_rope), static_cast<const __nv_bfloat16*>(v), idx, k, scale_log2,
      static_cast<__nv_bfloat16*>(out), lse, err);
  return cudaGetLastError();
}

}  // namespace dsa
