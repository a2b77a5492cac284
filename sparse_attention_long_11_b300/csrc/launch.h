// Internal host-side launchers of the DSA kernels (not part of the C ABI).
// Each enqueues one kernel on `stream` and returns the launch status.
#pragma once

#include <cuda_runtime.h>
#include "common.cuh"

namespace dsa {

// Lightning indexer, CUDA-core version: any supported dtype/shape.
cudaError_t launch_indexer_simt(const QueryBatch& qb, const CacheMap& cm, const dsa_indexer_inputs& ix,
                                float* scores, int64_t ld, int* err, cudaStream_t stream);

// Per-row exact top-k (radix select + ordered compaction).
cudaError_t launch_topk(const QueryBatch& qb, const float* scores, int64_t ld, int k, int32_t* idx,
                        int* err, cudaStream_t stream);

// Sparse attention, CUDA-core version: fp32 or bf16 operands, any supported shape.
cudaError_t launch_attn_simt(const QueryBatch& qb, const CacheMap& cm, const dsa_attn_inputs& at,
                             const int32_t* idx, int k, void* out, float* lse, int* err,
                             cudaStream_t stream);

// Lightning indexer on tcgen05 tensor cores: FP8 e4m3, 64 heads x 128, contiguous
// caches or paged caches whose block size is a multiple of 64.
// wait_limit: SM clocks after which any of the kernel's waits gives up
// (DSA_ERR_TIMEOUT); the default is about one second.
bool indexer_tc_supported(const CacheMap& cm, const dsa_indexer_inputs& ix);
cudaError_t launch_indexer_tc(const QueryBatch& qb, const CacheMap& cm, const dsa_indexer_inputs& ix,
                              float* scores, int64_t ld, int* err, cudaStream_t stream,
                              long long wait_limit = 2000000000LL);

inline cudaError_t launch_indexer(const QueryBatch& qb, const CacheMap& cm, const dsa_indexer_inputs& ix,
                                  float* scores, int64_t ld, int* err, cudaStream_t stream,
                                  long long wait_limit = 2000000000LL) {
  if (indexer_tc_supported(cm, ix)) return launch_indexer_tc(qb, cm, ix, scores, ld, err, stream, wait_limit);
  return launch_indexer_simt(qb, cm, ix, scores, ld, err, stream);
}

// Sparse attention on tcgen05 tensor cores: 128 heads, d_qk 576, d_v 512, bf16
// queries, a bf16 or FP8 (e4m3 + per-row scale) latent cache.
// prefix_valid: every idx row is ascending with its valid entries first
// (as the top-k stage writes them), so no row needs scanning.
cudaError_t launch_attn_tc(const QueryBatch& qb, const CacheMap& cm, const dsa_attn_inputs& at,
                           const int32_t* idx, int k, bool prefix_valid, void* out, float* lse, int* err,
                           cudaStream_t stream);

// Stage dispatch: the tensor-core kernel for the latent shape (bf16 or FP8
// cache), the CUDA-core kernel for fp32 operands.
inline cudaError_t launch_attn(const QueryBatch& qb, const CacheMap& cm, const dsa_attn_inputs& at,
                               const int32_t* idx, int k, void* out, float* lse, int* err, cudaStream_t stream,
                               bool prefix_valid = false) {
  if (at.dtype == DSA_BF16 || at.dtype == DSA_FP8_E4M3) return launch_attn_tc(qb, cm, at, idx, k, prefix_valid, out, lse, err, stream);
  return launch_attn_simt(qb, cm, at, idx, k, out, lse, err, stream);
}

// Indexer alignment loss KL(p || softmax(I)) over each query's candidate
// entries and its gradients for w, q and k (dk accumulated).  CUDA cores.
cudaError_t launch_indexer_kl_bwd(const QueryBatch& qb, const CacheMap& cm, const dsa_indexer_inputs& ix,
                                  const int32_t* idx, int k, const float* p, float* loss, float* grad_scores,
                                  float* dw, float* dq, float* dk, int* err, cudaStream_t stream);

// Appends new tokens to the caches: each key row (128 bf16 or fp32 values)
// encoded as e4m3 codes with scale amax/448, and (when kv_new is non-null)
// the latent row of d_qk bf16 values copied, or, with kv_scale, encoded the
// same way into an FP8 latent cache.  One warp per token.
cudaError_t launch_cache_append(const CacheMap& cm, int num_tok, const int32_t* tok_seq, const int32_t* tok_pos,
                                bool k_is_bf16, const void* k_new, uint8_t* k_cache, float* k_scale,
                                const void* kv_new, void* kv_cache, float* kv_scale, int d_qk, int* err,
                                cudaStream_t stream);

}  // namespace dsa
