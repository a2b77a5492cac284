// Shared device-side helpers of the DSA kernels: the cache row map, the
// sticky device error word, order-preserving score keys.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "dsa.h"

namespace dsa {

// Cache row map handed to kernels by value (mirrors dsa_cache_desc).
struct CacheMap {
  int32_t num_seqs;
  int32_t block_size;   // 0 = contiguous
  int32_t max_blocks;
  int32_t pad_;
  int64_t num_rows;
  int64_t seq_stride;
  const int32_t* block_table;
};

// Query batch handed to kernels by value (mirrors dsa_query_desc).
struct QueryBatch {
  const int32_t* q_seq;
  const int32_t* q_pos;
  int32_t num_q;
  int32_t max_kv;
};

// Sticky error word: the first failing check wins; later ones are dropped.
__device__ __forceinline__ void flag_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// Physical row of (seq, pos), or -1 (and DSA_ERR_BOUNDS flagged) when any part
// of the map is out of range.  Never dereferences an out-of-range pointer.
// Programmatic dependent launch.  A kernel launched with programmatic
// stream serialization may start while the previous kernel in the stream is
// still running: pdl_wait() returns once that kernel has completed and its
// memory operations are visible (immediately when there is no such
// dependency), and pdl_release() lets the next kernel in the stream start
// its own set-up early.  Work before pdl_wait() touches no memory another
// kernel of the stream writes or reads.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ int64_t cache_row(const CacheMap& c, int seq, int pos, int* err) {
  if (seq < 0 || seq >= c.num_seqs || pos < 0) {
    flag_error(err, DSA_ERR_BOUNDS);
    return -1;
  }
  int64_t row;
  if (c.block_size == 0) {
    row = (int64_t)seq * c.seq_stride + pos;
  } else {
    int blk = pos / c.block_size;
    if (blk >= c.max_blocks) {
      flag_error(err, DSA_ERR_BOUNDS);
      return -1;
    }
    int phys = __ldg(c.block_table + (int64_t)seq * c.max_blocks + blk);
    if (phys < 0) {
      flag_error(err, DSA_ERR_BOUNDS);
      return -1;
    }
    row = (int64_t)phys * c.block_size + (pos - blk * c.block_size);
  }
  if (row >= c.num_rows) {
    flag_error(err, DSA_ERR_BOUNDS);
    return -1;
  }
  return row;
}

// Order-preserving unsigned key of a float score: larger score <-> larger
// key.  -0 is first mapped to +0 so that the two compare equal.
__device__ __forceinline__ uint32_t score_key(float x) {
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The score a key stands for (the inverse of score_key; -0 comes back as +0).
__device__ __forceinline__ float key_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// 64-bit selection key of a (score, position) pair: the score's key in the
// high word, the complement of the position in the low word.  Larger means
// selected first: higher score, then lower position; the keys of one row
// are all distinct, so "the k largest keys" is a unique set.
__device__ __forceinline__ uint64_t composite_key(float x, int pos) {
  return ((uint64_t)score_key(x) << 32) | (uint64_t)(0xffffffffu - (uint32_t)pos);
}
__device__ __forceinline__ int composite_pos(uint64_t c) { return (int)(0xffffffffu - (uint32_t)c); }

__device__ __forceinline__ float2 fp8x2_e4m3_to_float2(uint16_t v) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)v, __NV_E4M3);
  return __half22float2(*reinterpret_cast<__half2*>(&h));
}

}  // namespace dsa
