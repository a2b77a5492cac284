/*
 * dsa.h -- C ABI of the DeepSeek Sparse Attention (DSA) hot path on NVIDIA
 * B300 (sm_103a), implemented by libdsa.so.
 *
 * What is computed (web pages about DeepSeek-V3.2; the formula itself is
 * fixed by this library because the pages print none):
 *   - "DeepSeek-V3.2: Pushing the Frontier of Open Large Language Models"
 *     summary card, section "How DSA Works": a lightning indexer scores a
 *     query against all keys cheaply in FP8, a top-k step keeps the 2048 most
 *     relevant tokens, and full attention runs only on the selected tokens.
 *   - News article "DeepSeek researchers announce DeepSeek-V3.2 and
 *     DeepSeek-V3.2-Speciale ...", section on sparse attention with
 *     near-linear long-context cost: a few low-precision indexer heads run on
 *     every token pair; a fine-grained selector keeps the top-k key/value
 *     positions per query; multi-query / latent attention runs on that set.
 *
 *   indexer   I[t,s] = sum_j w[t,j] * ReLU(sq[t,j] * sk[s] * <q_I[t,j,:], k_I[s,:]>),  s <= t
 *   top-k     the min(k, t+1) largest I[t,s] over s <= t; equal scores -> lower s
 *             first (+0 == -0); written in ascending s, padded with -1
 *   attention O[t,h,:] = sum_{s in sel(t)} softmax_s(scale * <q[t,h,:], kv[s,:]>) * kv[s,0:d_v]
 *             LSE[t,h] = ln sum_{s in sel(t)} exp(scale * <q[t,h,:], kv[s,:]>)
 *
 * Conventions shared by every entry point
 *   - Every tensor pointer is a DEVICE pointer unless marked "host".  The
 *     caller owns all memory; the library never allocates device memory and
 *     writes only the outputs and the caller-provided workspace.
 *   - Tensors are dense and row-major in the order their shape is written.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and the call returns without synchronising.  Only
 *     dsa_check_device_error() synchronises.
 *   - Arguments are validated on the host before anything is launched; a
 *     failed check returns DSA_ERR_INVALID_ARG or DSA_ERR_UNSUPPORTED and
 *     enqueues nothing.  A failed launch returns DSA_ERR_CUDA.  Nothing
 *     aborts, throws or prints.
 *   - Device-side checks (positions, sequence ids, block ids and selected
 *     indices out of range) never fault: the offending element is skipped
 *     (it contributes nothing; its score is -inf, its output row zero) and a
 *     sticky device error word records DSA_ERR_BOUNDS, which
 *     dsa_check_device_error() reports and clears.
 *   - Positions are logical positions inside a sequence.  The cache
 *     descriptor maps (sequence b, position s) to a physical cache row.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DSA_API __attribute__((visibility("default")))
#else
#define DSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dsa_stream_t; /* identical to cudaStream_t */

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1, /* NULL/misaligned pointer, bad size, inconsistent descriptor */
  DSA_ERR_UNSUPPORTED = 2, /* valid but not implemented (dtype / shape combination) */
  DSA_ERR_CUDA = 3,        /* a CUDA runtime or driver call failed */
  DSA_ERR_TIMEOUT = 4,     /* a bounded device-side wait expired (reported by dsa_check_device_error) */
  DSA_ERR_BOUNDS = 5,      /* device-side range check failed (reported by dsa_check_device_error) */
  DSA_ERR_WORKSPACE = 6    /* workspace NULL, misaligned (256 B) or smaller than one stage of one row */
} dsa_status;

typedef enum { DSA_F32 = 0, DSA_BF16 = 1, DSA_FP8_E4M3 = 2 } dsa_dtype;

/* The batch of query tokens.  Query row i is the token at position
 * q_pos[i] of sequence q_seq[i]; it sees keys 0..q_pos[i] of that sequence
 * (causal, inclusive).  Rows may come in any order and from any mix of
 * sequences (prefill chunks, decode tokens, both); throughput is best when
 * the rows of one sequence are consecutive and at consecutive positions. */
typedef struct {
  int32_t num_q;          /* number of query rows (0 = nothing to do) */
  const int32_t* q_seq;   /* [num_q] sequence id, 0 <= q_seq < num_seqs */
  const int32_t* q_pos;   /* [num_q] position, 0 <= q_pos < max_kv */
  int32_t max_kv;         /* host: an upper bound on q_pos[i] + 1 over the batch (>= 1) */
} dsa_query_desc;

/* Where the rows of each sequence live in the caches.  Both caches (indexer
 * keys and latent KV) use the same row map.
 *   contiguous (block_table == NULL): row(b, s) = b * seq_stride + s
 *   paged      (block_table != NULL): row(b, s) = block_table[b * max_blocks_per_seq + s / block_size]
 *                                                  * block_size + s % block_size                       */
typedef struct {
  int32_t num_seqs;            /* >= 1 */
  int64_t num_rows;            /* physical rows in each cache tensor (1 .. 2^31-1) */
  int64_t seq_stride;          /* contiguous: rows between sequences (>= 0) */
  const int32_t* block_table;  /* paged: [num_seqs, max_blocks_per_seq] physical block ids, or NULL */
  int32_t block_size;          /* paged: rows per block (> 0) */
  int32_t max_blocks_per_seq;  /* paged: width of block_table (> 0) */
} dsa_cache_desc;

/* Lightning-indexer operands.
 *   DSA_FP8_E4M3: heads = 64, dim = 128; q and k hold OCP e4m3 ("fn") codes
 *                 with one positive fp32 dequantisation scale per row
 *                 (q_scale [num_q, heads], k_scale [num_rows]).
 *   DSA_F32:      heads <= 64, dim in {32, 64, 128}; q and k hold fp32
 *                 values; q_scale and k_scale must be NULL.
 * q and k must be 16-byte aligned. */
typedef struct {
  dsa_dtype dtype;
  int32_t heads;          /* H_I */
  int32_t dim;            /* d_I */
  const void* q;          /* [num_q, heads, dim] */
  const float* q_scale;   /* [num_q, heads] or NULL */
  const float* w;         /* [num_q, heads] head weights (any sign) */
  const void* k;          /* [num_rows, dim] indexer key cache */
  const float* k_scale;   /* [num_rows] or NULL */
} dsa_indexer_inputs;

/* Attention operands: MQA over one shared latent row per token; the value of
 * a row is its first d_v entries.
 *   DSA_BF16:     heads = 128, d_qk = 576, d_v = 512 (the DeepSeek-V3.2
 *                 latent shape), q and kv bf16, output bf16;
 *   DSA_FP8_E4M3: the same shape with the latent cache stored as FP8: kv
 *                 holds OCP e4m3 codes [num_rows, 576] and kv_scale one fp32
 *                 scale per row; row s is read as the bf16 values
 *                 bf16(kv_scale[s] * code), the product in fp32 rounded once
 *                 to nearest even.  q bf16, output bf16.  (The pages name no
 *                 KV-cache format; this one reuses the indexer keys'
 *                 per-row encoding and halves the bytes a gathered row costs.)
 *   DSA_F32:      heads in {8, 16, ..., 128} (multiple of 8), d_qk <= 576 and
 *                 a multiple of 4, d_v <= d_qk and a multiple of 4, output
 *                 fp32.
 * q and kv must be 16-byte aligned; kv_scale 4-byte aligned for
 * DSA_FP8_E4M3 and NULL otherwise. */
typedef struct {
  dsa_dtype dtype;
  int32_t heads;          /* H */
  int32_t d_qk;
  int32_t d_v;
  const void* q;          /* [num_q, heads, d_qk] */
  const void* kv;         /* [num_rows, d_qk] latent KV cache */
  float softmax_scale;    /* finite (positive for DSA_BF16 and DSA_FP8_E4M3); logits are scale * <q, kv> */
  const float* kv_scale;  /* DSA_FP8_E4M3: [num_rows] per-row scales; else NULL */
} dsa_attn_inputs;

/* Stage 1 alone (debug / parity API): materialises the score rows.
 * scores[i * ld_scores + s] = I[i, s] for s <= q_pos[i] and -INFINITY for
 * q_pos[i] < s < max_kv (entries at s >= max_kv are not written).
 * ld_scores >= max_kv; scores 16-byte aligned, ld_scores a multiple of 4. */
DSA_API dsa_status dsa_index_scores(const dsa_query_desc* qd, const dsa_cache_desc* cd,
                            const dsa_indexer_inputs* ix, float* scores, int64_t ld_scores,
                            dsa_stream_t stream);

/* dsa_index_scores with an explicit bound on the kernel's device-side waits:
 * every wait of the tensor-core indexer gives up after wait_limit_cycles SM
 * clocks (dsa_index_scores uses about 2e9, one second).  A test aid for the
 * timeout path: with a limit of a few hundred clocks the kernel's pipeline
 * waits expire, the kernel drains its own in-flight copies and MMAs, frees
 * its tensor memory and returns, and dsa_check_device_error() reports
 * DSA_ERR_TIMEOUT; the scores are then undefined and the context stays
 * usable.  Ignored by the CUDA-core indexer (DSA_F32), which has no waits.
 * wait_limit_cycles >= 1, else DSA_ERR_INVALID_ARG. */
DSA_API dsa_status dsa_index_scores_wait_limit(const dsa_query_desc* qd, const dsa_cache_desc* cd,
                                               const dsa_indexer_inputs* ix, float* scores, int64_t ld_scores,
                                               int64_t wait_limit_cycles, dsa_stream_t stream);

/* Stage 2 alone: per query row i, the top-k of scores[i * ld_scores + s] over
 * s = 0..q_pos[i] (scores at larger s are ignored), written to
 * idx[i * k .. i * k + k) in ascending s, padded with -1 when q_pos[i] + 1 < k.
 * Exact: the selected set is unique (score desc, then s asc; -0 == +0;
 * scores must not be NaN).  1 <= k <= 8192; ld_scores >= max_kv.
 * Uses no workspace. */
DSA_API dsa_status dsa_topk(const dsa_query_desc* qd, const float* scores, int64_t ld_scores, int32_t k,
                    int32_t* idx, dsa_stream_t stream);

/* Stage 3 alone: attention of every query row over its selected logical
 * positions idx[i * k .. i * k + k) (entries -1 are skipped; any order; a
 * position must be <= q_pos[i]).  out [num_q, heads, d_v] (bf16 for
 * DSA_BF16, fp32 for DSA_F32), lse [num_q, heads] fp32 natural-log
 * log-sum-exp of the logits (-INFINITY and a zero output row if nothing is
 * selected).  1 <= k <= 8192. */
DSA_API dsa_status dsa_sparse_attn(const dsa_query_desc* qd, const dsa_cache_desc* cd,
                           const dsa_attn_inputs* at, const int32_t* idx, int32_t k,
                           void* out, float* lse, dsa_stream_t stream);

/* Per-head attention operands: the prefill attention mode.
 *
 * Susan Zhang's thread on the DeepSeek-V3.2 write-up names separate attention
 * modes for disaggregated prefill and decode.  dsa_sparse_attn is the latent
 * (absorbed) form, one shared row per key; this is the per-head
 * (non-absorbed) form of the same attention: every head has its own key and
 * value rows, as up-projected from the latent rows, and the rope part of the
 * key is shared by all heads.  With k_nope[s,h] = W_K[h] c[s], v[s,h] =
 * W_V[h] c[s] and the absorbed query (W_K[h]^T q_nope[h], q_rope[h]), the two
 * give the same attention (the output up-projected by W_V[h]).  The pages
 * give no shapes; this library fixes d_nope = 128, d_rope = 64, d_v = 128,
 * bf16, heads a multiple of 8 up to 128.  A selected pair then moves
 * heads x 512 + 128 bytes of rows (65,664 at 128 heads) against 1,152 for the
 * latent row: the mode is bound by the gathers.
 * All pointers 16-byte aligned. */
typedef struct {
  dsa_dtype dtype;        /* DSA_BF16 */
  int32_t heads;          /* H: 8 .. 128, a multiple of 8 */
  int32_t d_nope;         /* 128 */
  int32_t d_rope;         /* 64 */
  int32_t d_v;            /* 128 */
  const void* q;          /* [num_q, heads, d_nope + d_rope] */
  const void* k_nope;     /* [num_rows, heads, d_nope] per-head key rows */
  const void* k_rope;     /* [num_rows, d_rope] the rope part, shared by all heads */
  const void* v;          /* [num_rows, heads, d_v] per-head value rows */
  float softmax_scale;    /* finite */
} dsa_mha_inputs;

/* Per-head sparse attention of every query row over its selected positions
 * idx[i * k .. i * k + k) (entries -1 are skipped; any order; a position must
 * be <= q_pos[i]):
 *   O[i,h,:] = sum_s softmax_s(scale * (<q_nope[i,h], k_nope[s,h]> + <q_rope[i,h], k_rope[s]>)) v[s,h,:]
 * out [num_q, heads, d_v] bf16, lse [num_q, heads] fp32 (natural log; -inf
 * and a zero row if nothing is selected).  1 <= k <= 8192.  Cache rows are
 * mapped by the cache descriptor as for the other stages. */
DSA_API dsa_status dsa_sparse_attn_mha(const dsa_query_desc* qd, const dsa_cache_desc* cd, const dsa_mha_inputs* at,
                                       const int32_t* idx, int32_t k, void* out, float* lse, dsa_stream_t stream);

/* Recommended bytes of workspace for dsa_forward on this batch (0 if the
 * arguments are invalid): every query row in one stage, capped at 1 GiB.
 * With the FP8 indexer (the streamed selection below) a row needs its
 * sampled scores and candidate list, O(k + max_kv / 32) entries, not a score
 * row; with fp32 indexer operands a row is one staged score row.  Depends
 * only on the host-side fields (num_q, max_kv, k, dtypes, shapes). */
DSA_API size_t dsa_forward_workspace_size(const dsa_query_desc* qd, const dsa_indexer_inputs* ix, int32_t k,
                                  const dsa_attn_inputs* at);

/* Bytes of workspace with which dsa_forward runs this batch in stages of at
 * most stage_rows query rows (0 if the arguments are invalid or stage_rows <
 * 1).  dsa_forward_workspace_size() is this for the recommended stage;
 * stage_rows = 1 gives the least workspace dsa_forward accepts. */
DSA_API size_t dsa_forward_stage_workspace_size(const dsa_query_desc* qd, const dsa_indexer_inputs* ix, int32_t k,
                                                const dsa_attn_inputs* at, int64_t stage_rows);

/* The number of query rows per stage that dsa_forward runs with a workspace
 * of workspace_bytes (its stages are equal in size, so this is
 * ceil(num_q / stages)); 0 if the workspace is below the least
 * dsa_forward accepts or the arguments are invalid.  A workspace of
 * dsa_forward_workspace_size() bytes runs the whole batch in one stage
 * whenever that size is below the recommended cap.  Host-side only: no
 * device work, no pointer is dereferenced. */
DSA_API int64_t dsa_forward_stage_rows(const dsa_query_desc* qd, const dsa_indexer_inputs* ix, int32_t k,
                                       const dsa_attn_inputs* at, size_t workspace_bytes);

/* The whole hot path: indexer -> top-k -> sparse attention for a batch of
 * prefill chunks and/or decode tokens.  Writes idx [num_q, k] (the selected
 * positions, exactly as dsa_topk would write them for dsa_index_scores'
 * rows), out and lse (as dsa_sparse_attn).
 *
 * With FP8 indexer operands (the tensor-core indexer) the score rows are
 * never written: the indexer first scores every m-th key tile of each query
 * (at most 32 tiles a row), a per-query threshold is taken from those
 * samples, the indexer then scores the other tiles and keeps only the keys at
 * or above the threshold, and an exact selection runs on those candidates.
 * A row whose threshold misses (too few keys above it, or more than its list
 * holds: adversarial or heavily tied rows) is recomputed exactly by a
 * fallback, with the same arithmetic, so every row's selection is exact and
 * bitwise equal to dsa_topk on dsa_index_scores.  Otherwise (fp32 operands,
 * or a paged cache whose block size is not a multiple of 64) the score rows
 * are staged through the workspace.
 *
 * workspace: 256-byte aligned, owned by the caller and not read before it is
 * written (no zeroing needed); it must not be used by other work while this
 * call's kernels run.  The queries run in equal stages of as many rows as it
 * holds: dsa_forward_stage_workspace_size() gives the bytes for a stage size
 * (1 row is the least; DSA_ERR_WORKSPACE below it) and
 * dsa_forward_workspace_size() the recommended size.  Any size gives the same
 * results; fewer, fuller stages run faster.
 *
 * With an FP8 latent cache (at->dtype DSA_FP8_E4M3), when the call reads each
 * cache row at least 4 times on average (num_q * min(k, max_kv) >= 4 *
 * num_rows: prefill chunks) and the workspace holds num_rows * 1152 bytes,
 * the workspace is then reused for a bf16 copy of the whole cache
 * (dsa_kv_dequant) and the attention runs on that copy instead of converting
 * the rows in its gather; the results are the same bits either way. */
DSA_API dsa_status dsa_forward(const dsa_query_desc* qd, const dsa_cache_desc* cd,
                       const dsa_indexer_inputs* ix, int32_t k, const dsa_attn_inputs* at,
                       int32_t* idx, void* out, float* lse,
                       void* workspace, size_t workspace_bytes, dsa_stream_t stream);

/* dsa_forward for callers that cannot allocate device memory.
 *
 * The paper has no counterpart to this entry point; it exists for users of
 * this library.  Some callers cannot call cudaMalloc (or any allocator) when
 * they run the forward: an inference engine whose memory plan is fixed before
 * serving starts, a plugin whose host forbids allocation, or a serving loop
 * that must not let cudaMalloc synchronise the device.  This variant takes no
 * workspace.  Its scratch (the staged score rows) lives in one file-scope
 * device array of DSA_NOALLOC_SCRATCH_BYTES bytes inside libdsa.so; every GPU
 * that loads the library holds that array until the process exits.
 *
 *   - Arguments and outputs are exactly those of dsa_forward without the
 *     workspace; results equal dsa_forward's.
 *   - max_kv above DSA_NOALLOC_MAX_KV (one staged score row must fit in the
 *     array) is rejected with DSA_ERR_UNSUPPORTED before anything runs.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it; make that first call before any
 *     stream capture.
 *   - Every call on a device shares the one array, which keeps the last
 *     call's contents.  Nothing in it needs to start at zero (each staged row
 *     is written before it is read).  Calls whose kernels overlap on the GPU
 *     (different streams, or different host threads) race on the array:
 *     order them on one stream or with events.
 *   - Calls no cudaMalloc, cudaFree or other allocating routine. */
#define DSA_NOALLOC_SCRATCH_BYTES (8u << 20)
#define DSA_NOALLOC_MAX_KV 2097152
DSA_API dsa_status dsa_forward_noalloc(const dsa_query_desc* qd, const dsa_cache_desc* cd,
                                       const dsa_indexer_inputs* ix, int32_t k, const dsa_attn_inputs* at,
                                       int32_t* idx, void* out, float* lse, dsa_stream_t stream);

/* Synchronises `stream`, then reads and clears the device error word of the
 * current device: DSA_OK, DSA_ERR_BOUNDS or DSA_ERR_TIMEOUT (or DSA_ERR_CUDA
 * if the synchronisation itself failed). */
DSA_API dsa_status dsa_check_device_error(dsa_stream_t stream);

/* Text of the last CUDA error this library saw on the calling host thread
 * (which call, the CUDA error name and message), or "no error".  The pointer
 * stays valid until the next call into the library on this thread. */
DSA_API const char* dsa_last_error_detail(void);

/* Static, NUL-terminated description of a status code (never NULL). */
DSA_API const char* dsa_status_string(dsa_status status);

/*
 * dsa_cache_append -- write num_tok new tokens into the caches the forward
 * reads (the step that precedes the indexer in every decode iteration).
 * The FP8 keys are the operands of the summary card's "cheap FP8 relevance
 * scores" (DeepSeek-V3.2 summary card, "How DSA Works"); the pages print no
 * encoding, so this library fixes one: per key row, scale = amax(|row|) /
 * 448 (1 for an all-zero row) and codes = e4m3(row / scale), round to
 * nearest with ties to even, saturated to +-448, the scale and the division
 * in fp32.
 *
 *   cache     physical-row map shared by both caches (as for dsa_forward)
 *   tok_seq, tok_pos  [num_tok] int32: sequence and logical position of each
 *             new token; its physical row is written
 *   k_dtype   DSA_BF16 or DSA_F32: element type of k_new
 *   k_new     [num_tok, dim] new indexer keys, rows 16-byte aligned; dim must
 *             be 128 (else DSA_ERR_UNSUPPORTED)
 *   k_cache   [num_rows, 128] uint8 e4m3 key cache (16-byte aligned)
 *   k_scale   [num_rows] fp32 per-row scales
 *   kv_new    [num_tok, d_qk] bf16 new latent rows, or NULL (then kv_cache
 *             and kv_scale must be NULL too and only the keys are written)
 *   kv_cache  [num_rows, d_qk] latent cache: bf16 (rows copied; d_qk * 2 a
 *             multiple of 16) when kv_scale is NULL, else the FP8 latent
 *             cache of dsa_attn_inputs' DSA_FP8_E4M3: uint8 e4m3 codes, each
 *             row encoded like the keys (d_qk a multiple of 16, <= 4096)
 *   kv_scale  [num_rows] fp32 per-row scales of the FP8 latent cache, or NULL
 *
 * Rows of tokens whose position lies outside the descriptor are skipped and
 * DSA_ERR_BOUNDS is recorded for dsa_check_device_error().  Two tokens that
 * map to the same row race.  num_tok == 0 enqueues nothing.
 */
DSA_API dsa_status dsa_cache_append(const dsa_cache_desc* cache, int32_t num_tok, const int32_t* tok_seq,
                                    const int32_t* tok_pos, dsa_dtype k_dtype, const void* k_new, int32_t dim,
                                    uint8_t* k_cache, float* k_scale, const void* kv_new, int32_t d_qk,
                                    void* kv_cache, float* kv_scale, dsa_stream_t stream);

/*
 * dsa_kv_dequant -- the bf16 values an FP8 latent cache stands for.
 * DeepSeek-V3.2 summary card, "How DSA Works": full attention runs on the
 * selected tokens' latent rows; with the FP8 cache of dsa_attn_inputs'
 * DSA_FP8_E4M3 those rows are read as
 *     out[r][c] = bf16(kv_scale[r] * code[r][c])   (the product in fp32,
 *                                                    rounded once to nearest even)
 * which are exactly the values dsa_sparse_attn and dsa_forward read for row r.
 *
 *   num_rows  rows to convert (0 enqueues nothing; at most 2^31 - 1)
 *   kv        [num_rows, 576] uint8 e4m3 codes, 16-byte aligned
 *   kv_scale  [num_rows] fp32 per-row scales, 4-byte aligned
 *   out       [num_rows, 576] bf16, 16-byte aligned; must not overlap kv
 *
 * dsa_forward does this itself, into its workspace, when a call reads each
 * cache row many times over (prefill) and the workspace holds num_rows *
 * 1152 bytes: its attention then gathers bf16 rows instead of converting
 * every gathered element, with the same results bit for bit.  No device
 * error is recorded (every code has a value).  Invalid arguments return
 * DSA_ERR_INVALID_ARG before anything runs.
 */
DSA_API dsa_status dsa_kv_dequant(int64_t num_rows, const void* kv, const float* kv_scale, void* out,
                                  dsa_stream_t stream);

/*
 * dsa_indexer_kl_backward -- the indexer's training step: its alignment loss
 * and the gradients of that loss.  News article on DeepSeek-V3.2,
 * continued-pre-training section: the indexer is trained with a
 * Kullback-Leibler loss to match the main attention's distribution -- over
 * all keys in the dense warm-up, over the selected entries only in the
 * sparse phase, where that loss is the indexer's only gradient.  The target
 * distribution is an input here (the pages give no formula for it).
 *
 * For query t, its candidate entries are the valid entries e of idx[t]
 * (0 <= idx[t][e] <= q_pos[t]; -1 = padding, ignored), and p[t][e] is the
 * target probability of entry e (summing to 1 over the valid entries).  With
 * the dequantised operands q_j = q_scale[t][j] * q[t][j] and
 * k_s = k_scale[s] * k[s] (scales 1 for DSA_F32) and x_js = <q_j, k_s>:
 *   I_e  = sum_j w[t][j] ReLU(x_j,idx[t][e]),   pi = softmax over the entries of I
 *   loss[t]           = sum_e p_e (log p_e - log pi_e)     (0 log 0 = 0)
 *   grad_scores[t][e] = pi_e - p_e (0 at padding)           (optional: may be NULL)
 *   dw[t][j]          = sum_e g_e ReLU(x_je)
 *   dq[t][j][:]       = w[t][j] sum_e g_e [x_je > 0] k_{idx[t][e]}
 *   dk[s][:]         += sum over (t, e) with idx[t][e] = s of g_e sum_j w[t][j] [x_je > 0] q_j
 * ReLU'(0) = 0, and every [x > 0] decision is exact (a dot near zero is
 * recomputed in fp64).  The dense warm-up is the same call with every
 * position 0..q_pos[t] as an entry (k >= max_kv).
 *
 *   ix        indexer operands as for the forward (FP8 with heads = 64,
 *             dim = 128, or fp32 with heads <= 64, dim in {32, 64, 128})
 *   idx, p    [num_q, k] int32 and fp32; 1 <= k <= 8192
 *   loss      [num_q] fp32; dw [num_q, heads] fp32; dq [num_q, heads, dim]
 *             fp32 (16-byte aligned)
 *   dk        [num_rows, dim] fp32 (16-byte aligned), ADDED to: zero it first
 *             for a fresh gradient.  Additions are atomic, so the bits of dk
 *             depend on their order; loss, dw and dq do not.
 *
 * CUDA cores (one block per query); asynchronous on `stream`.
 */
DSA_API dsa_status dsa_indexer_kl_backward(const dsa_query_desc* qd, const dsa_cache_desc* cd,
                                           const dsa_indexer_inputs* ix, const int32_t* idx, int32_t k,
                                           const float* p, float* loss, float* grad_scores, float* dw, float* dq,
                                           float* dk, dsa_stream_t stream);

/* ---- Measurement aids (host-side state; not thread-safe) ----------------
 * While a profile is open, every kernel the library launches is bracketed by
 * a pair of CUDA events recorded on its launch stream, and tagged with its
 * stage.  dsa_profile_read() waits for the recorded events and returns each
 * launch's stage and device duration.  Events are created by the library (no
 * device memory); at most `capacity` launches are recorded. */
typedef enum {
  DSA_STAGE_INDEXER = 1,
  DSA_STAGE_TOPK = 2,
  DSA_STAGE_ATTN = 3,
  DSA_STAGE_APPEND = 4,
  DSA_STAGE_INDEXER_BWD = 5
} dsa_stage;
DSA_API dsa_status dsa_profile_start(int32_t capacity);
/* Closes the profile; returns the number of launches recorded. */
DSA_API int32_t dsa_profile_stop(void);
/* stage[i] (dsa_stage) and ms[i] for i < min(cap, recorded); *n = that count. */
DSA_API dsa_status dsa_profile_read(int32_t* stage, float* ms, int32_t cap, int32_t* n);
/* Kernels launched by this library in this process so far. */
DSA_API int64_t dsa_launch_count(void);

/* ABI version: major * 10000 + minor * 100 + patch. */
DSA_API int32_t dsa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DSA_H_ */
