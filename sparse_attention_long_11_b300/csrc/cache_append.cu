// Appending new tokens to the two caches the hot path reads: the indexer key
// cache (FP8 e4m3 rows with one fp32 scale each) and the latent KV cache
// (bf16 rows).  The keys are the "cheap FP8 relevance scores" operands of the
// DeepSeek-V3.2 summary card ("How DSA Works"); each new key row is encoded
// once, when its token is written: scale = amax(|row|) / 448 (1 for an
// all-zero row), codes = e4m3(row / scale) rounded to nearest (ties to even)
// and saturated to +-448, scale and division in fp32.
//
// One warp per token: lane l holds elements 4l .. 4l+3 of the 128-wide key,
// the row's amax is a warp reduction, the codes of a lane are one 32-bit
// store, and the warp copies the 1152-byte latent row with 16-byte moves --
// or, for an FP8 latent cache, encodes it like the key (two passes over the
// row in 8-element chunks: the amax, then the codes).
// Positions map to physical rows through the cache descriptor (paged or
// contiguous); a position outside it is skipped and flagged.
#include "launch.h"

namespace dsa {
namespace {

constexpr int kWarps = 4;   // tokens per block

// Four floats -> four e4m3 codes in memory order (byte 0 = a).  The
// conversion rounds to nearest, ties to even, and saturates to +-448.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));   // upper byte = b, lower = a
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ void bf16x8(uint4 v, float (&x)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    x[2 * j] = __uint_as_float(w[j] << 16);
    x[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
  }
}

__global__ void __launch_bounds__(kWarps * 32)
cache_append_kernel(CacheMap cm, int num_tok, const int32_t* __restrict__ tok_seq, const int32_t* __restrict__ tok_pos,
                    int k_is_bf16, const void* __restrict__ k_new, uint8_t* __restrict__ k_cache,
                    float* __restrict__ k_scale, const uint4* __restrict__ kv_new, void* __restrict__ kv_cache,
                    float* __restrict__ kv_scale, int d_qk, int* err) {
  const int lane = threadIdx.x & 31;
  const int i = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (i >= num_tok) return;
  const int seq = __ldg(tok_seq + i), pos = __ldg(tok_pos + i);
  if (cm.block_size == 0 && cm.seq_stride > 0 && pos >= cm.seq_stride) {   // would run into the next sequence
    if (lane == 0) flag_error(err, DSA_ERR_BOUNDS);
    return;
  }
  const int64_t row = cache_row(cm, seq, pos, lane == 0 ? err : nullptr);
  if (row < 0) return;

  float x[4];
  if (k_is_bf16) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(k_new) + (int64_t)i * 128) + lane);
    x[0] = __uint_as_float(v.x << 16);
    x[1] = __uint_as_float(v.x & 0xffff0000u);
    x[2] = __uint_as_float(v.y << 16);
    x[3] = __uint_as_float(v.y & 0xffff0000u);
  } else {
    const float4 v = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(k_new) + (int64_t)i * 128) + lane);
    x[0] = v.x;
    x[1] = v.y;
    x[2] = v.z;
    x[3] = v.w;
  }
  const float amax = warp_max(fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3]))));
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  reinterpret_cast<uint32_t*>(k_cache + row * 128)[lane] =
      e4m3x4(__fdiv_rn(x[0], scale), __fdiv_rn(x[1], scale), __fdiv_rn(x[2], scale), __fdiv_rn(x[3], scale));
  if (lane == 0) k_scale[row] = scale;
  if (!kv_new) return;
  const int vec = d_qk / 8;                      // 16-byte chunks of 8 bf16 values
  const uint4* src = kv_new + (int64_t)i * vec;
  if (!kv_scale) {
    uint4* dst = static_cast<uint4*>(kv_cache) + row * vec;
    for (int c = lane; c < vec; c += 32) dst[c] = __ldg(src + c);
    return;
  }
  float vmax = 0.f;
  for (int c = lane; c < vec; c += 32) {
    float y[8];
    bf16x8(__ldg(src + c), y);
#pragma unroll
    for (int j = 0; j < 8; ++j) vmax = fmaxf(vmax, fabsf(y[j]));
  }
  vmax = warp_max(vmax);
  const float vs = vmax > 0.f ? __fdiv_rn(vmax, 448.f) : 1.f;
  uint2* dst = reinterpret_cast<uint2*>(static_cast<uint8_t*>(kv_cache) + row * d_qk);
  for (int c = lane; c < vec; c += 32) {
    float y[8];
    bf16x8(__ldg(src + c), y);
    dst[c] = make_uint2(e4m3x4(__fdiv_rn(y[0], vs), __fdiv_rn(y[1], vs), __fdiv_rn(y[2], vs), __fdiv_rn(y[3], vs)),
                        e4m3x4(__fdiv_rn(y[4], vs), __fdiv_rn(y[5], vs), __fdiv_rn(y[6], vs), __fdiv_rn(y[7], vs)));
  }
  if (lane == 0) kv_scale[row] = vs;
}

}  // namespace

cudaError_t launch_cache_append(const CacheMap& cm, int num_tok, const int32_t* tok_seq, const int32_t* tok_pos,
                                bool k_is_bf16, const void* k_new, uint8_t* k_cache, float* k_scale,
                                const void* kv_new, void* kv_cache, float* kv_scale, int d_qk, int* err,
                                cudaStream_t stream) {
  const int blocks = (num_tok + kWarps - 1) / kWarps;
  cache_append_kernel<<<blocks, kWarps * 32, 0, stream>>>(
      cm, num_tok, tok_seq, tok_pos, k_is_bf16 ? 1 : 0, k_new, k_cache, k_scale,
      static_cast<const uint4*>(kv_new), kv_cache, kv_scale, d_qk, err);
  return cudaGetLastError();
}

}  // namespace dsa
