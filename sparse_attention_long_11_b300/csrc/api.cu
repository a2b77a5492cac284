// C ABI of the DSA hot path (declared in include/dsa.h): host-side argument
// validation, the per-device error word, stage dispatch and the fused
// forward schedule.  Nothing here allocates device memory.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "launch.h"

namespace dsa {
namespace {

__device__ int g_device_error;   // sticky error word (see flag_error)

// Scores of at most this many bytes are staged per indexer/top-k round of the
// fused forward, so the staged rows stay resident in the 126 MB L2 between
// the indexer writing them and the top-k reading them.
constexpr size_t kStageBytes = size_t(1) << 30;   // recommended staged-score budget (fewer, fuller stages)
constexpr int kMaxTopk = 8192;
constexpr int kMaxKv = 1 << 22;   // keeps every grid dimension in range

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

dsa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA; }

int* device_error_ptr() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}

dsa_status check_query(const dsa_query_desc* qd) {
  if (!qd || qd->num_q < 0) return DSA_ERR_INVALID_ARG;
  if (qd->num_q == 0) return DSA_OK;
  if (!qd->q_seq || !qd->q_pos || !aligned(qd->q_seq, 4) || !aligned(qd->q_pos, 4)) return DSA_ERR_INVALID_ARG;
  if (qd->max_kv < 1 || qd->max_kv > kMaxKv) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

dsa_status check_cache(const dsa_cache_desc* cd, int max_kv) {
  if (!cd || cd->num_seqs < 1 || cd->num_rows < 1) return DSA_ERR_INVALID_ARG;
  if (cd->num_rows > INT32_MAX) return DSA_ERR_INVALID_ARG;   // row ids travel as 32-bit values
  if (cd->block_table) {
    if (cd->block_size < 1 || cd->max_blocks_per_seq < 1 || !aligned(cd->block_table, 4)) return DSA_ERR_INVALID_ARG;
    if ((int64_t)cd->block_size * cd->max_blocks_per_seq < max_kv) return DSA_ERR_INVALID_ARG;
  } else {
    if (cd->seq_stride < 0) return DSA_ERR_INVALID_ARG;
    if (cd->num_seqs > 1 && cd->seq_stride < max_kv) return DSA_ERR_INVALID_ARG;   // sequences would overlap
  }
  return DSA_OK;
}

dsa_status check_indexer(const dsa_indexer_inputs* ix) {
  if (!ix || !ix->q || !ix->w || !ix->k) return DSA_ERR_INVALID_ARG;
  if (!aligned(ix->q, 16) || !aligned(ix->k, 16) || !aligned(ix->w, 4)) return DSA_ERR_INVALID_ARG;
  if (ix->dtype == DSA_FP8_E4M3) {
    if (!ix->q_scale || !ix->k_scale || !aligned(ix->q_scale, 4) || !aligned(ix->k_scale, 4)) return DSA_ERR_INVALID_ARG;
    if (ix->heads != 64 || ix->dim != 128) return DSA_ERR_UNSUPPORTED;
  } else if (ix->dtype == DSA_F32) {
    if (ix->q_scale || ix->k_scale) return DSA_ERR_INVALID_ARG;
    if (ix->heads < 1 || ix->heads > 64) return DSA_ERR_UNSUPPORTED;
    if (ix->dim != 32 && ix->dim != 64 && ix->dim != 128) return DSA_ERR_UNSUPPORTED;
  } else {
    return DSA_ERR_UNSUPPORTED;
  }
  return DSA_OK;
}

dsa_status check_attn(const dsa_attn_inputs* at) {
  if (!at || !at->q || !at->kv) return DSA_ERR_INVALID_ARG;
  if (!aligned(at->q, 16) || !aligned(at->kv, 16)) return DSA_ERR_INVALID_ARG;
  if (!std::isfinite(at->softmax_scale)) return DSA_ERR_INVALID_ARG;
  if ((at->dtype == DSA_FP8_E4M3) != (at->kv_scale != nullptr)) return DSA_ERR_INVALID_ARG;
  if (at->kv_scale && !aligned(at->kv_scale, 4)) return DSA_ERR_INVALID_ARG;
  if (at->dtype == DSA_BF16 || at->dtype == DSA_FP8_E4M3) {
    if (!(at->softmax_scale > 0.f)) return DSA_ERR_INVALID_ARG;   // the row maxima are taken on the raw dots
    if (at->heads != 128 || at->d_qk != 576 || at->d_v != 512) return DSA_ERR_UNSUPPORTED;
  } else if (at->dtype == DSA_F32) {
    if (at->heads < 8 || at->heads > 128 || at->heads % 8) return DSA_ERR_UNSUPPORTED;
    if (at->d_qk < 4 || at->d_qk > 576 || at->d_qk % 4) return DSA_ERR_UNSUPPORTED;
    if (at->d_v < 4 || at->d_v > at->d_qk || at->d_v > 512 || at->d_v % 4) return DSA_ERR_UNSUPPORTED;
  } else {
    return DSA_ERR_UNSUPPORTED;
  }
  return DSA_OK;
}

#define DSA_TRY(x)                       \
  do {                                   \
    dsa_status s_ = (x);                 \
    if (s_ != DSA_OK) return s_;         \
  } while (0)

QueryBatch to_batch(const dsa_query_desc* qd) { return QueryBatch{qd->q_seq, qd->q_pos, qd->num_q, qd->max_kv}; }

CacheMap to_map(const dsa_cache_desc* cd) {
  CacheMap m{};
  m.num_seqs = cd->num_seqs;
  m.block_size = cd->block_table ? cd->block_size : 0;
  m.max_blocks = cd->block_table ? cd->max_blocks_per_seq : 0;
  m.num_rows = cd->num_rows;
  m.seq_stride = cd->seq_stride;
  m.block_table = cd->block_table;
  return m;
}

int64_t score_ld(int max_kv) { return ((int64_t)max_kv + 3) & ~int64_t(3); }

int64_t stage_rows(int num_q, int max_kv) {
  int64_t per = score_ld(max_kv) * (int64_t)sizeof(float);
  int64_t r = (int64_t)(kStageBytes / per);
  if (r < 1) r = 1;
  if (r > num_q) r = num_q;
  return r;
}

size_t idx_elem_size(const dsa_indexer_inputs* ix) { return ix->dtype == DSA_FP8_E4M3 ? 1 : 4; }

// ---- launch accounting and the optional per-launch event profile
std::atomic<int64_t> g_launches{0};
struct ProfRec {
  int stage;
  cudaEvent_t a, b;
};
std::vector<ProfRec> g_prof;
size_t g_prof_n = 0;
bool g_prof_on = false;

thread_local char g_last_detail[256] = "no error";

void note_cuda_error(cudaError_t e, const char* where) {
  if (e == cudaSuccess) return;
  snprintf(g_last_detail, sizeof(g_last_detail), "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

template <typename F>
cudaError_t launch(int stage, cudaStream_t st, F&& f) {
  const bool rec = g_prof_on && g_prof_n < g_prof.size();
  if (rec) {
    g_prof[g_prof_n].stage = stage;
    cudaEventRecord(g_prof[g_prof_n].a, st);
  }
  cudaError_t e = f();
  note_cuda_error(e, stage == DSA_STAGE_INDEXER        ? "indexer launch"
                     : stage == DSA_STAGE_TOPK         ? "top-k launch"
                     : stage == DSA_STAGE_ATTN         ? "attention launch"
                     : stage == DSA_STAGE_APPEND       ? "cache append launch"
                     : stage == DSA_STAGE_INDEXER_BWD ? "indexer backward launch"
                                                       : "launch");
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (rec) {
    cudaEventRecord(g_prof[g_prof_n].b, st);
    ++g_prof_n;
  }
  return e;
}

// The forward's attention launch.  With an FP8 latent cache whose rows the
// call reads many times over (a prefill chunk reads each cache row about
// num_q * k / num_rows times), the whole cache is converted to bf16 once,
// into the workspace (the selection's scratch is dead by then), and the bf16
// attention runs on that copy: its gathers then move bf16 rows instead of
// converting every element of every gathered row again.  The copy holds
// exactly the values the FP8 gather stages, so the results are the same
// bits.  Without room for the copy, or with little reuse (decode), the FP8
// gather runs as it is.
constexpr int64_t kKvCopyReuse = 4;   // row reads per cache row above which the copy pays
cudaError_t launch_forward_attn(const dsa_query_desc* qd, const dsa_cache_desc* cd, const dsa_attn_inputs* at,
                                const int32_t* idx, int32_t k, void* out, float* lse, void* ws, size_t ws_bytes,
                                int* err, cudaStream_t st) {
  const CacheMap cm = to_map(cd);
  const size_t copy_bytes = (size_t)cd->num_rows * (size_t)at->d_qk * 2;
  const int64_t reads = (int64_t)qd->num_q * std::min<int64_t>(k, qd->max_kv);
  if (at->dtype == DSA_FP8_E4M3 && ws && copy_bytes <= ws_bytes && reads >= kKvCopyReuse * cd->num_rows) {
    cudaError_t e =
        launch(DSA_STAGE_ATTN, st, [&] { return launch_kv_dequant(at->kv, at->kv_scale, cd->num_rows, ws, st); });
    if (e != cudaSuccess) return e;
    dsa_attn_inputs bf = *at;
    bf.dtype = DSA_BF16;
    bf.kv = ws;
    bf.kv_scale = nullptr;
    return launch(DSA_STAGE_ATTN, st, [&] { return launch_attn(to_batch(qd), cm, bf, idx, k, out, lse, err, st, true); });
  }
  return launch(DSA_STAGE_ATTN, st, [&] { return launch_attn(to_batch(qd), cm, *at, idx, k, out, lse, err, st, true); });
}

// The fused forward over validated arguments: the queries in stages of at
// most max_rows score rows (as many as the scratch holds), each stage's
// indexer scores written to `scores` and reduced to its top-k rows, then one
// attention launch over the whole batch.  The stages are made equal in size,
// so the last one is not a sliver.
dsa_status run_staged(const dsa_query_desc* qd, const dsa_cache_desc* cd, const dsa_indexer_inputs* ix, int32_t k,
                      const dsa_attn_inputs* at, int32_t* idx, void* out, float* lse, float* scores,
                      int64_t max_rows, int* err, cudaStream_t st, size_t copy_bytes = 0) {
  const CacheMap cm = to_map(cd);
  const int64_t ld = score_ld(qd->max_kv);
  max_rows = std::max<int64_t>(1, std::min<int64_t>(max_rows, qd->num_q));
  const int64_t stages = (qd->num_q + max_rows - 1) / max_rows;
  const int64_t rows = (qd->num_q + stages - 1) / stages;
  const size_t qi_row = (size_t)ix->heads * ix->dim * idx_elem_size(ix);
  for (int64_t r0 = 0; r0 < qd->num_q; r0 += rows) {
    const int n = (int)std::min<int64_t>(rows, qd->num_q - r0);
    QueryBatch qb{qd->q_seq + r0, qd->q_pos + r0, n, qd->max_kv};
    dsa_indexer_inputs sub = *ix;
    sub.q = static_cast<const uint8_t*>(ix->q) + r0 * qi_row;
    sub.w = ix->w + r0 * ix->heads;
    if (ix->q_scale) sub.q_scale = ix->q_scale + r0 * ix->heads;
    cudaError_t e = launch(DSA_STAGE_INDEXER, st, [&] { return launch_indexer(qb, cm, sub, scores, ld, err, st); });
    if (e != cudaSuccess) return DSA_ERR_CUDA;
    e = launch(DSA_STAGE_TOPK, st, [&] { return launch_topk(qb, scores, ld, k, idx + r0 * k, err, st); });
    if (e != cudaSuccess) return DSA_ERR_CUDA;
  }
  // (the score rows are dead now: with copy_bytes > 0 their space may hold
  // the bf16 copy of an FP8 latent cache)
  return cuda_status(launch_forward_attn(qd, cd, at, idx, k, out, lse, copy_bytes ? scores : nullptr, copy_bytes,
                                         err, st));
}

// ---- The fused forward: the selection streams out of the indexer, so no
// score row is written (select.cu).  Workspace of one stage of `rows` query
// rows: sampled scores, thresholds, candidate counts and lists, the fallback
// queue, and one fallback score row per fallback CTA.
struct FusedLayout {
  SelectPlan plan;
  int64_t ld = 0;          // fallback score row length (floats)
  int64_t rows = 0;
  int fb_grid = 0;
  size_t samp = 0, thr = 0, cnt = 0, fail_rows = 0, ctr = 0, cand = 0, slots = 0, total = 0;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

FusedLayout fused_layout(int64_t rows, int fb_grid, int max_kv, int k) {
  FusedLayout L;
  L.plan = plan_select(max_kv, k);
  L.ld = score_ld(max_kv);
  L.rows = rows;
  L.fb_grid = fb_grid;
  size_t off = 0;
  L.samp = off;      off += align256((size_t)rows * L.plan.lds * sizeof(float));
  L.thr = off;       off += align256((size_t)rows * sizeof(uint64_t));
  L.cnt = off;       off += align256((size_t)rows * sizeof(uint32_t));
  L.fail_rows = off; off += align256((size_t)rows * sizeof(uint32_t));
  L.ctr = off;       off += 256;
  L.cand = off;      off += align256((size_t)rows * L.plan.cap * sizeof(uint64_t));
  L.slots = off;     off += align256((size_t)fb_grid * L.ld * sizeof(float));
  L.total = off;
  return L;
}

bool fused_supported(const dsa_cache_desc* cd, const dsa_indexer_inputs* ix) {
  return indexer_tc_supported(to_map(cd), *ix);
}

// The most rows per stage that `bytes` hold with fb_grid fallback rows (0 if
// not even one).
int64_t fused_rows_fitting(size_t bytes, int fb_grid, int max_kv, int k, int64_t num_q) {
  const FusedLayout one = fused_layout(1, fb_grid, max_kv, k);
  if (one.total > bytes) return 0;
  // the layout grows with the rows by at least `per` bytes a row: binary
  // search the largest row count that fits below that bound
  const size_t per = (size_t)one.plan.lds * 4 + 8 + 4 + 4 + (size_t)one.plan.cap * 8;
  int64_t lo = 1, hi = std::max<int64_t>(1, std::min<int64_t>(num_q, (int64_t)(bytes / per)));
  while (lo < hi) {
    const int64_t mid = lo + (hi - lo + 1) / 2;
    if (fused_layout(mid, fb_grid, max_kv, k).total <= bytes) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Rows per stage of the fused forward with ws_bytes of workspace and its
// fallback grid (fb, in/out); 0 if not even one row fits.  The stages are
// equal in size.
int64_t fused_stage_rows(const dsa_query_desc* qd, int32_t k, size_t ws_bytes, int& fb) {
  fb = sel_fallback_grid(qd->num_q);
  int64_t max_rows = fused_rows_fitting(ws_bytes, fb, qd->max_kv, k, qd->num_q);
  if (max_rows == 0) {   // a small workspace: one fallback row
    fb = 1;
    max_rows = fused_rows_fitting(ws_bytes, fb, qd->max_kv, k, qd->num_q);
    if (max_rows == 0) return 0;
  }
  const int64_t stages = (qd->num_q + max_rows - 1) / max_rows;
  return (qd->num_q + stages - 1) / stages;
}

// Rows per stage of the staged forward (score rows in the workspace).
int64_t staged_stage_rows(const dsa_query_desc* qd, size_t ws_bytes) {
  int64_t max_rows = (int64_t)(ws_bytes / (score_ld(qd->max_kv) * sizeof(float)));
  if (max_rows < 1) return 0;
  max_rows = std::min<int64_t>(max_rows, qd->num_q);
  const int64_t stages = (qd->num_q + max_rows - 1) / max_rows;
  return (qd->num_q + stages - 1) / stages;
}

dsa_status run_fused(const dsa_query_desc* qd, const dsa_cache_desc* cd, const dsa_indexer_inputs* ix, int32_t k,
                     const dsa_attn_inputs* at, int32_t* idx, void* out, float* lse, void* workspace, size_t ws_bytes,
                     int* err, cudaStream_t st) {
  const CacheMap cm = to_map(cd);
  int fb = 0;
  const int64_t rows = fused_stage_rows(qd, k, ws_bytes, fb);
  if (rows == 0) return DSA_ERR_WORKSPACE;
  const FusedLayout L = fused_layout(rows, fb, qd->max_kv, k);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  float* samp = reinterpret_cast<float*>(base + L.samp);
  uint64_t* thr = reinterpret_cast<uint64_t*>(base + L.thr);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(base + L.cnt);
  uint32_t* fail_rows = reinterpret_cast<uint32_t*>(base + L.fail_rows);
  uint32_t* ctr = reinterpret_cast<uint32_t*>(base + L.ctr);
  uint64_t* cand = reinterpret_cast<uint64_t*>(base + L.cand);
  float* slots = reinterpret_cast<float*>(base + L.slots);
  const size_t qi_row = (size_t)ix->heads * ix->dim * idx_elem_size(ix);
  for (int64_t r0 = 0; r0 < qd->num_q; r0 += rows) {
    const int n = (int)std::min<int64_t>(rows, qd->num_q - r0);
    QueryBatch qb{qd->q_seq + r0, qd->q_pos + r0, n, qd->max_kv};
    dsa_indexer_inputs sub = *ix;
    sub.q = static_cast<const uint8_t*>(ix->q) + r0 * qi_row;
    sub.w = ix->w + r0 * ix->heads;
    if (ix->q_scale) sub.q_scale = ix->q_scale + r0 * ix->heads;
    int32_t* idx_s = idx + r0 * k;
    IndexerOut so;
    so.mode = IndexerOut::kSample;
    so.m = L.plan.m;
    so.min_pos = k;
    so.scores = samp;
    so.ld = L.plan.lds;
    cudaError_t e = launch(DSA_STAGE_INDEXER, st, [&] { return launch_indexer_tc(qb, cm, sub, so, err, st); });
    if (e != cudaSuccess) return DSA_ERR_CUDA;
    e = launch(DSA_STAGE_TOPK, st, [&] { return launch_sel_threshold(qb, L.plan, samp, k, thr, cnt, ctr, st); });
    if (e != cudaSuccess) return DSA_ERR_CUDA;
    if (L.plan.m > 1) {   // with m = 1 every tile was sampled
      IndexerOut fo;
      fo.mode = IndexerOut::kFilter;
      fo.m = L.plan.m;
      fo.min_pos = k;
      fo.thr = thr;
      fo.cnt = cnt;
      fo.cand = cand;
      fo.cap = L.plan.cap;
      e = launch(DSA_STAGE_INDEXER, st, [&] { return launch_indexer_tc(qb, cm, sub, fo, err, st); });
      if (e != cudaSuccess) return DSA_ERR_CUDA;
    }
    e = launch(DSA_STAGE_TOPK, st, [&] {
      return launch_sel_select(qb, L.plan, samp, k, thr, cnt, cand, idx_s, ctr, fail_rows, err, st);
    });
    if (e != cudaSuccess) return DSA_ERR_CUDA;
    e = launch(DSA_STAGE_TOPK, st, [&] {
      return launch_sel_fallback(qb, cm, sub, k, idx_s, slots, L.ld, L.fb_grid, ctr, fail_rows, err, st);
    });
    if (e != cudaSuccess) return DSA_ERR_CUDA;
  }
  return cuda_status(launch_forward_attn(qd, cd, at, idx, k, out, lse, workspace, ws_bytes, err, st));
}

// Recommended bytes of the fused forward: every row of the call in one
// stage, up to kStageBytes.
size_t fused_workspace_size(const dsa_query_desc* qd, int32_t k) {
  const int fb = sel_fallback_grid(qd->num_q);
  int64_t r = fused_rows_fitting(kStageBytes, fb, qd->max_kv, k, qd->num_q);
  if (r == 0) r = 1;
  return fused_layout(r, fb, qd->max_kv, k).total;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" {

dsa_status dsa_index_scores(const dsa_query_desc* qd, const dsa_cache_desc* cd, const dsa_indexer_inputs* ix,
                            float* scores, int64_t ld_scores, dsa_stream_t stream) {
  DSA_TRY(check_query(qd));
  if (qd->num_q == 0) return DSA_OK;
  DSA_TRY(check_cache(cd, qd->max_kv));
  DSA_TRY(check_indexer(ix));
  if (!scores || !aligned(scores, 16) || ld_scores < qd->max_kv || ld_scores % 4) return DSA_ERR_INVALID_ARG;
  int* err = device_error_ptr();
  if (!err) return DSA_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return cuda_status(launch(DSA_STAGE_INDEXER, st, [&] {
    return launch_indexer(to_batch(qd), to_map(cd), *ix, scores, ld_scores, err, st);
  }));
}

dsa_status dsa_index_scores_wait_limit(const dsa_query_desc* qd, const dsa_cache_desc* cd,
                                      const dsa_indexer_inputs* ix, float* scores, int64_t ld_scores,
                                      int64_t wait_limit_cycles, dsa_stream_t stream) {
  if (wait_limit_cycles < 1) return DSA_ERR_INVALID_ARG;
  DSA_TRY(check_query(qd));
  if (qd->num_q == 0) return DSA_OK;
  DSA_TRY(check_cache(cd, qd->max_kv));
  DSA_TRY(check_indexer(ix));
  if (!scores || !aligned(scores, 16) || ld_scores < qd->max_kv || ld_scores % 4) return DSA_ERR_INVALID_ARG;
  int* err = device_error_ptr();
  if (!err) return DSA_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return cuda_status(launch(DSA_STAGE_INDEXER, st, [&] {
    return launch_indexer(to_batch(qd), to_map(cd), *ix, scores, ld_scores, err, st, (long long)wait_limit_cycles);
  }));
}

dsa_status dsa_topk(const dsa_query_desc* qd, const float* scores, int64_t ld_scores, int32_t k, int32_t* idx,
                    dsa_stream_t stream) {
  DSA_TRY(check_query(qd));
  if (k < 1 || k > kMaxTopk) return DSA_ERR_INVALID_ARG;
  if (qd->num_q == 0) return DSA_OK;
  if (!scores || !idx || !aligned(scores, 4) || !aligned(idx, 4) || ld_scores < qd->max_kv) return DSA_ERR_INVALID_ARG;
  int* err = device_error_ptr();
  if (!err) return DSA_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return cuda_status(launch(DSA_STAGE_TOPK, st, [&] { return launch_topk(to_batch(qd), scores, ld_scores, k, idx, err, st); }));
}

dsa_status dsa_sparse_attn(const dsa_query_desc* qd, const dsa_cache_desc* cd, const dsa_attn_inputs* at,
                           const int32_t* idx, int32_t k, void* out, float* lse, dsa_stream_t stream) {
  DSA_TRY(check_query(qd));
  if (k < 1 || k > kMaxTopk) return DSA_ERR_INVALID_ARG;
  if (qd->num_q == 0) return DSA_OK;
  DSA_TRY(check_cache(cd, qd->max_kv));
  DSA_TRY(check_attn(at));
  if (!idx || !out || !lse || !aligned(idx, 4) || !aligned(out, 16) || !aligned(lse, 4)) return DSA_ERR_INVALID_ARG;
  int* err = device_error_ptr();
  if (!err) return DSA_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return cuda_status(launch(DSA_STAGE_ATTN, st, [&] {
    return launch_attn(to_batch(qd), to_map(cd), *at, idx, k, out, lse, err, st);
  }));
}

dsa_status dsa_sparse_attn_mha(const dsa_query_desc* qd, const dsa_cache_desc* cd, const dsa_mha_inputs* at,
                               const int32_t* idx, int32_t k, void* out, float* lse, dsa_stream_t stream) {
  DSA_TRY(check_query(qd));
  if (k < 1 || k > kMaxTopk) return DSA_ERR_INVALID_ARG;
  if (qd->num_q == 0) return DSA_OK;
  DSA_TRY(check_cache(cd, qd->max_kv));
  if (!at || !at->q || !at->k_nope || !at->k_rope || !at->v) return DSA_ERR_INVALID_ARG;
  if (!aligned(at->q, 16) || !aligned(at->k_nope, 16) || !aligned(at->k_rope, 16) || !aligned(at->v, 16))
    return DSA_ERR_INVALID_ARG;
  if (!std::isfinite(at->softmax_scale)) return DSA_ERR_INVALID_ARG;
  if (at->dtype != DSA_BF16 || at->d_nope != 128 || at->d_rope != 64 || at->d_v != 128) return DSA_ERR_UNSUPPORTED;
  if (at->heads < 8 || at->heads > 128 || at->heads % 8) return DSA_ERR_UNSUPPORTED;
  if (!idx || !out || !lse || !aligned(idx, 4) || !aligned(out, 16) || !aligned(lse, 4)) return DSA_ERR_INVALID_ARG;
  int* err = device_error_ptr();
  if (!err) return DSA_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return cuda_status(launch(DSA_STAGE_ATTN, st, [&] {
    return launch_attn_mha(to_batch(qd), to_map(cd), at->heads, at->q, at->k_nope, at->k_rope, at->v,
                           at->softmax_scale, idx, k, out, lse, err, st);
  }));
}

size_t dsa_forward_workspace_size(const dsa_query_desc* qd, const dsa_indexer_inputs* ix, int32_t k,
                                  const dsa_attn_inputs* at) {
  if (check_query(qd) != DSA_OK || check_indexer(ix) != DSA_OK || check_attn(at) != DSA_OK) return 0;
  if (k < 1 || k > kMaxTopk) return 0;
  if (qd->num_q == 0) return 256;
  if (indexer_tc_supported(CacheMap{}, *ix)) return fused_workspace_size(qd, k);
  size_t bytes = (size_t)stage_rows(qd->num_q, qd->max_kv) * score_ld(qd->max_kv) * sizeof(float);
  return (bytes + 255) & ~size_t(255);
}

size_t dsa_forward_stage_workspace_size(const dsa_query_desc* qd, const dsa_indexer_inputs* ix, int32_t k,
                                        const dsa_attn_inputs* at, int64_t stage_rows) {
  if (check_query(qd) != DSA_OK || check_indexer(ix) != DSA_OK || check_attn(at) != DSA_OK) return 0;
  if (k < 1 || k > kMaxTopk || stage_rows < 1) return 0;
  if (qd->num_q == 0) return 256;
  const int64_t r = std::min<int64_t>(stage_rows, qd->num_q);
  if (indexer_tc_supported(CacheMap{}, *ix))   // one fallback score row per stage row, up to one per fallback CTA
    return fused_layout(r, (int)std::min<int64_t>(sel_fallback_grid(qd->num_q), r), qd->max_kv, k).total;
  return align256((size_t)r * score_ld(qd->max_kv) * sizeof(float));
}

int64_t dsa_forward_stage_rows(const dsa_query_desc* qd, const dsa_indexer_inputs* ix, int32_t k,
                               const dsa_attn_inputs* at, size_t workspace_bytes) {
  if (check_query(qd) != DSA_OK || check_indexer(ix) != DSA_OK || check_attn(at) != DSA_OK) return 0;
  if (k < 1 || k > kMaxTopk || qd->num_q == 0) return 0;
  int fb = 0;
  if (indexer_tc_supported(CacheMap{}, *ix)) return fused_stage_rows(qd, k, workspace_bytes, fb);
  return staged_stage_rows(qd, workspace_bytes);
}

dsa_status dsa_forward(const dsa_query_desc* qd, const dsa_cache_desc* cd, const dsa_indexer_inputs* ix, int32_t k,
                       const dsa_attn_inputs* at, int32_t* idx, void* out, float* lse, void* workspace,
                       size_t workspace_bytes, dsa_stream_t stream) {
  DSA_TRY(check_query(qd));
  if (k < 1 || k > kMaxTopk) return DSA_ERR_INVALID_ARG;
  if (qd->num_q == 0) return DSA_OK;
  DSA_TRY(check_cache(cd, qd->max_kv));
  DSA_TRY(check_indexer(ix));
  DSA_TRY(check_attn(at));
  if (!idx || !out || !lse || !aligned(idx, 4) || !aligned(out, 16) || !aligned(lse, 4)) return DSA_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256)) return DSA_ERR_WORKSPACE;
  const bool fused = fused_supported(cd, ix);
  // the least workspace: one stage of one row (and one fallback row)
  const size_t least = fused ? fused_layout(1, 1, qd->max_kv, k).total : (size_t)score_ld(qd->max_kv) * sizeof(float);
  if (workspace_bytes < least) return DSA_ERR_WORKSPACE;
  int* err = device_error_ptr();
  if (!err) return DSA_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (fused) return run_fused(qd, cd, ix, k, at, idx, out, lse, workspace, workspace_bytes, err, st);

  const int64_t rows = (int64_t)(workspace_bytes / (score_ld(qd->max_kv) * sizeof(float)));
  return run_staged(qd, cd, ix, k, at, idx, out, lse, static_cast<float*>(workspace), rows, err, st,
                    workspace_bytes);
}

dsa_status dsa_kv_dequant(int64_t num_rows, const void* kv, const float* kv_scale, void* out, dsa_stream_t stream) {
  if (num_rows < 0 || num_rows > INT32_MAX) return DSA_ERR_INVALID_ARG;
  if (num_rows == 0) return DSA_OK;
  if (!kv || !kv_scale || !out || !aligned(kv, 16) || !aligned(kv_scale, 4) || !aligned(out, 16))
    return DSA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return cuda_status(launch(DSA_STAGE_ATTN, st, [&] { return launch_kv_dequant(kv, kv_scale, num_rows, out, st); }));
}

dsa_status dsa_indexer_kl_backward(const dsa_query_desc* qd, const dsa_cache_desc* cd, const dsa_indexer_inputs* ix,
                                   const int32_t* idx, int32_t k, const float* p, float* loss, float* grad_scores,
                                   float* dw, float* dq, float* dk, dsa_stream_t stream) {
  DSA_TRY(check_query(qd));
  if (k < 1 || k > kMaxTopk) return DSA_ERR_INVALID_ARG;
  if (qd->num_q == 0) return DSA_OK;
  DSA_TRY(check_cache(cd, qd->max_kv));
  DSA_TRY(check_indexer(ix));
  if (ix->heads > 64 || (ix->dim != 32 && ix->dim != 64 && ix->dim != 128)) return DSA_ERR_UNSUPPORTED;
  if (!idx || !p || !loss || !dw || !dq || !dk) return DSA_ERR_INVALID_ARG;
  if (!aligned(idx, 4) || !aligned(p, 4) || !aligned(loss, 4) || !aligned(dw, 4) || !aligned(dq, 16) ||
      !aligned(dk, 16) || (grad_scores && !aligned(grad_scores, 4)))
    return DSA_ERR_INVALID_ARG;
  int* err = device_error_ptr();
  if (!err) return DSA_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return cuda_status(launch(DSA_STAGE_INDEXER_BWD, st, [&] {
    return launch_indexer_kl_bwd(to_batch(qd), to_map(cd), *ix, idx, k, p, loss, grad_scores, dw, dq, dk, err, st);
  }));
}

dsa_status dsa_cache_append(const dsa_cache_desc* cd, int32_t num_tok, const int32_t* tok_seq, const int32_t* tok_pos,
                            dsa_dtype k_dtype, const void* k_new, int32_t dim, uint8_t* k_cache, float* k_scale,
                            const void* kv_new, int32_t d_qk, void* kv_cache, float* kv_scale, dsa_stream_t stream) {
  if (num_tok < 0) return DSA_ERR_INVALID_ARG;
  if (num_tok == 0) return DSA_OK;
  DSA_TRY(check_cache(cd, 1));
  if (k_dtype != DSA_BF16 && k_dtype != DSA_F32) return DSA_ERR_UNSUPPORTED;
  if (dim != 128) return DSA_ERR_UNSUPPORTED;
  if (!tok_seq || !tok_pos || !aligned(tok_seq, 4) || !aligned(tok_pos, 4)) return DSA_ERR_INVALID_ARG;
  if (!k_new || !k_cache || !k_scale || !aligned(k_new, 16) || !aligned(k_cache, 16) || !aligned(k_scale, 4))
    return DSA_ERR_INVALID_ARG;
  if ((kv_new == nullptr) != (kv_cache == nullptr)) return DSA_ERR_INVALID_ARG;
  if (kv_scale && !kv_new) return DSA_ERR_INVALID_ARG;
  if (kv_new) {
    if (!aligned(kv_new, 16) || !aligned(kv_cache, 16)) return DSA_ERR_INVALID_ARG;
    if (kv_scale && !aligned(kv_scale, 4)) return DSA_ERR_INVALID_ARG;
    if (d_qk < 8 || d_qk > 4096 || (d_qk * 2) % 16) return DSA_ERR_UNSUPPORTED;
    if (kv_scale && d_qk % 16) return DSA_ERR_UNSUPPORTED;   // FP8 rows of whole 16-byte chunks
  }
  int* err = device_error_ptr();
  if (!err) return DSA_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return cuda_status(launch(DSA_STAGE_APPEND, st, [&] {
    return launch_cache_append(to_map(cd), num_tok, tok_seq, tok_pos, k_dtype == DSA_BF16, k_new, k_cache, k_scale,
                               kv_new, kv_cache, kv_scale, kv_new ? d_qk : 0, err, st);
  }));
}

const char* dsa_last_error_detail(void) { return g_last_detail; }

dsa_status dsa_check_device_error(dsa_stream_t stream) {
  const cudaError_t se = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (se != cudaSuccess) {
    note_cuda_error(se, "stream synchronize");
    return DSA_ERR_CUDA;
  }
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return DSA_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return DSA_ERR_CUDA;
  }
  return static_cast<dsa_status>(v);
}

const char* dsa_status_string(dsa_status s) {
  switch (s) {
    case DSA_OK: return "DSA_OK: success";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG: invalid argument (null/misaligned pointer, bad size or descriptor)";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED: dtype or shape combination not implemented";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA: a CUDA call failed";
    case DSA_ERR_TIMEOUT: return "DSA_ERR_TIMEOUT: a bounded device-side wait expired";
    case DSA_ERR_BOUNDS: return "DSA_ERR_BOUNDS: a device-side range check failed (element skipped)";
    case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE: workspace missing, misaligned or too small";
  }
  return "unknown dsa_status";
}

int32_t dsa_version(void) { return 100; }

}  // extern "C"

// ---- dsa_forward_noalloc: the forward with its scratch in a file-scope array

// Staged score rows of dsa_forward_noalloc (the only device memory the library
// itself owns).  Shared by every call on a device; see dsa.h.
static __device__ __align__(256) unsigned char g_noalloc_scratch[DSA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached.
dsa_status noalloc_scratch(float** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return DSA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return DSA_ERR_CUDA;
    g_noalloc_addr[dev] = p;
  }
  *out = static_cast<float*>(g_noalloc_addr[dev]);
  return DSA_OK;
}

}  // namespace

extern "C" {

dsa_status dsa_forward_noalloc(const dsa_query_desc* qd, const dsa_cache_desc* cd, const dsa_indexer_inputs* ix,
                               int32_t k, const dsa_attn_inputs* at, int32_t* idx, void* out, float* lse,
                               dsa_stream_t stream) {
  DSA_TRY(check_query(qd));
  if (k < 1 || k > kMaxTopk) return DSA_ERR_INVALID_ARG;
  if (qd->num_q == 0) return DSA_OK;
  if (qd->max_kv > DSA_NOALLOC_MAX_KV) return DSA_ERR_UNSUPPORTED;   // one staged row must fit the array
  DSA_TRY(check_cache(cd, qd->max_kv));
  DSA_TRY(check_indexer(ix));
  DSA_TRY(check_attn(at));
  if (!idx || !out || !lse || !aligned(idx, 4) || !aligned(out, 16) || !aligned(lse, 4)) return DSA_ERR_INVALID_ARG;
  float* scores = nullptr;
  DSA_TRY(noalloc_scratch(&scores));
  int* err = device_error_ptr();
  if (!err) return DSA_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  const int64_t rows = (int64_t)(DSA_NOALLOC_SCRATCH_BYTES / (score_ld(qd->max_kv) * sizeof(float)));
  return run_staged(qd, cd, ix, k, at, idx, out, lse, scores, rows, err, st);
}

dsa_status dsa_profile_start(int32_t capacity) {
  if (capacity < 1) return DSA_ERR_INVALID_ARG;
  while ((int32_t)g_prof.size() < capacity) {
    ProfRec r{0, nullptr, nullptr};
    if (cudaEventCreate(&r.a) != cudaSuccess || cudaEventCreate(&r.b) != cudaSuccess) return DSA_ERR_CUDA;
    g_prof.push_back(r);
  }
  g_prof_n = 0;
  g_prof_on = true;
  return DSA_OK;
}

int32_t dsa_profile_stop(void) {
  g_prof_on = false;
  return (int32_t)g_prof_n;
}

dsa_status dsa_profile_read(int32_t* stage, float* ms, int32_t cap, int32_t* n) {
  if (!stage || !ms || !n || cap < 0) return DSA_ERR_INVALID_ARG;
  const int32_t m = std::min<int32_t>(cap, (int32_t)g_prof_n);
  for (int32_t i = 0; i < m; ++i) {
    if (cudaEventSynchronize(g_prof[i].b) != cudaSuccess) return DSA_ERR_CUDA;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, g_prof[i].a, g_prof[i].b) != cudaSuccess) return DSA_ERR_CUDA;
    stage[i] = g_prof[i].stage;
    ms[i] = t;
  }
  *n = m;
  return DSA_OK;
}

int64_t dsa_launch_count(void) { return g_launches.load(); }

}  // extern "C"
