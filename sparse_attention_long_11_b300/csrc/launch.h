// Internal host-side launchers of the DSA kernels (not part of the C ABI).
// Each enqueues one kernel on `stream` and returns the launch status.
#pragma once

#include <cuda_runtime.h>

#include <utility>

#include "common.cuh"

namespace dsa {

// Launches `kern` with programmatic stream serialization: the kernel may
// start (and run its set-up) while the previous kernel of the stream is
// still running; it waits for that kernel's completion with pdl_wait()
// before it touches memory the stream's other kernels use.  The fused
// forward's kernels are launched this way, so a decode step's six short
// launches do not each pay the launch latency and set-up on the critical path.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

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
// Where the tensor-core indexer puts its scores.
//   kFull:   score rows, scores[i * ld + s] (-inf beyond the query's position,
//            up to max_kv), every key tile.
//   kSample: only the key tiles 0, m, 2m, ...; the scores of the o-th of them
//            go to scores[i * ld + o * 128 + (s - 128 o m)] (-inf beyond the
//            query's position).
//   kFilter: every other key tile; a key is appended to the query's candidate
//            list (cand[i * cap + slot], its composite key) when its composite
//            key is at least thr[i]; cnt[i] counts the appends (entries past
//            cap are not stored).
// In kSample and kFilter, queries at positions below min_pos are skipped.
struct IndexerOut {
  enum { kFull = 0, kSample = 1, kFilter = 2 };
  int mode = kFull;
  int m = 1;
  int min_pos = 0;
  int cap = 0;
  float* scores = nullptr;
  int64_t ld = 0;
  const uint64_t* thr = nullptr;
  uint32_t* cnt = nullptr;
  uint64_t* cand = nullptr;
};

// Ordinal count of a mode's key tiles among T tiles (host side of the
// kernel's tile map).
inline int indexer_tile_count(const IndexerOut& o, int T) {
  if (o.mode == IndexerOut::kFull) return T;
  const int sampled = (T + o.m - 1) / o.m;
  return o.mode == IndexerOut::kSample ? sampled : T - sampled;
}

// wait_limit: SM clocks after which any of the kernel's waits gives up
// (DSA_ERR_TIMEOUT); the default is about one second.
bool indexer_tc_supported(const CacheMap& cm, const dsa_indexer_inputs& ix);
cudaError_t launch_indexer_tc(const QueryBatch& qb, const CacheMap& cm, const dsa_indexer_inputs& ix,
                              const IndexerOut& out, int* err, cudaStream_t stream,
                              long long wait_limit = 2000000000LL);
inline cudaError_t launch_indexer_tc(const QueryBatch& qb, const CacheMap& cm, const dsa_indexer_inputs& ix,
                                     float* scores, int64_t ld, int* err, cudaStream_t stream,
                                     long long wait_limit = 2000000000LL) {
  IndexerOut o;
  o.scores = scores;
  o.ld = ld;
  return launch_indexer_tc(qb, cm, ix, o, err, stream, wait_limit);
}

inline cudaError_t launch_indexer(const QueryBatch& qb, const CacheMap& cm, const dsa_indexer_inputs& ix,
                                  float* scores, int64_t ld, int* err, cudaStream_t stream,
                                  long long wait_limit = 2000000000LL) {
  if (indexer_tc_supported(cm, ix)) return launch_indexer_tc(qb, cm, ix, scores, ld, err, stream, wait_limit);
  return launch_indexer_simt(qb, cm, ix, scores, ld, err, stream);
}

// ---- The fused forward's selection (select.cu, select_fallback.cu)
// Sampled key tiles per query row: the sample stride m is the smallest that
// keeps a row's sampled tiles at or below this count.
constexpr int kSelSampleTiles = 32;
struct SelectPlan {
  int m;             // sample stride in key tiles
  int64_t lds;       // sample row length (floats): sampled tiles x 128
  int cap;           // candidate list capacity per row (composite keys)
  int list_cap;      // the select kernel's shared list: cap + a bound on the samples >= the threshold
  int win;           // positions per bitmap window of the ordered output (a multiple of 64)
};
SelectPlan plan_select(int max_kv, int k);
size_t select_shared_bytes(const SelectPlan& p);
// Per row: the threshold (composite key) from the sampled scores; clears the
// row's candidate count (and the fallback queue counters fail_ctr[0..1]).
cudaError_t launch_sel_threshold(const QueryBatch& qb, const SelectPlan& p, const float* samp, int k, uint64_t* thr,
                                 uint32_t* cnt, uint32_t* fail_ctr, cudaStream_t stream);
// Per row: the exact top-k from the candidates and samples, written to idx in
// ascending position; rows whose threshold missed go to the fallback queue.
cudaError_t launch_sel_select(const QueryBatch& qb, const SelectPlan& p, const float* samp, int k, const uint64_t* thr,
                              const uint32_t* cnt, const uint64_t* cand, int32_t* idx, uint32_t* fail_ctr,
                              uint32_t* fail_rows, int* err, cudaStream_t stream);
// The queued rows: scores recomputed (same arithmetic as the indexer) into
// one row of `slots` (ld floats) per CTA, then the exact top-k.  FP8 indexer
// operands only.
int sel_fallback_grid(int num_q);
cudaError_t launch_sel_fallback(const QueryBatch& qb, const CacheMap& cm, const dsa_indexer_inputs& ix, int k,
                                int32_t* idx, float* slots, int64_t ld, int grid, uint32_t* fail_ctr,
                                const uint32_t* fail_rows, int* err, cudaStream_t stream);

// Sparse attention on tcgen05 tensor cores: 128 heads, d_qk 576, d_v 512, bf16
// queries, a bf16 or FP8 (e4m3 + per-row scale) latent cache.
// prefix_valid: every idx row is ascending with its valid entries first
// (as the top-k stage writes them), so no row needs scanning.
cudaError_t launch_attn_tc(const QueryBatch& qb, const CacheMap& cm, const dsa_attn_inputs& at,
                           const int32_t* idx, int k, bool prefix_valid, void* out, float* lse, int* err,
                           cudaStream_t stream);

// An FP8 latent cache (e4m3 codes [num_rows, 576], one fp32 scale per row)
// converted to bf16 [num_rows, 576]: out = bf16(scale * code), exactly the
// values the FP8 attention's gather stages.  A plain (not programmatic)
// launch: it starts after all earlier work in the stream has finished.
cudaError_t launch_kv_dequant(const void* kv, const float* kv_scale, int64_t num_rows, void* out,
                              cudaStream_t stream);

// Stage dispatch: the tensor-core kernel for the latent shape (bf16 or FP8
// cache), the CUDA-core kernel for fp32 operands.
inline cudaError_t launch_attn(const QueryBatch& qb, const CacheMap& cm, const dsa_attn_inputs& at,
                               const int32_t* idx, int k, void* out, float* lse, int* err, cudaStream_t stream,
                               bool prefix_valid = false) {
  if (at.dtype == DSA_BF16 || at.dtype == DSA_FP8_E4M3) return launch_attn_tc(qb, cm, at, idx, k, prefix_valid, out, lse, err, stream);
  return launch_attn_simt(qb, cm, at, idx, k, out, lse, err, stream);
}

// Per-head (non-absorbed) sparse attention, the prefill attention mode:
// bf16, heads a multiple of 8, per-head keys and values of 128 and a shared
// rope part of 64 (attn_mha.cu).
cudaError_t launch_attn_mha(const QueryBatch& qb, const CacheMap& cm, int heads, const void* q, const void* k_nope,
                            const void* k_rope, const void* v, float softmax_scale, const int32_t* idx, int k,
                            void* out, float* lse, int* err, cudaStream_t stream);

// Indexer alignment loss KL(p || softmax(I)) over each query's candidate
// entries and its gradients for w, q and k (dk accumulated): on the tensor
// cores for FP8 operands with 64 heads x 128 (indexer_bwd_tc.cu), on CUDA
// cores otherwise.
cudaError_t launch_indexer_kl_bwd(const QueryBatch& qb, const CacheMap& cm, const dsa_indexer_inputs& ix,
                                  const int32_t* idx, int k, const float* p, float* loss, float* grad_scores,
                                  float* dw, float* dq, float* dk, int* err, cudaStream_t stream);
bool indexer_kl_bwd_tc_supported(const dsa_indexer_inputs& ix);
cudaError_t launch_indexer_kl_bwd_tc(const QueryBatch& qb, const CacheMap& cm, const dsa_indexer_inputs& ix,
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
