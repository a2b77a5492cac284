// Lightning indexer on the 5th-generation tensor cores: an FP8 (e4m3) GEMM
// with the ReLU, weighted head sum and scales fused into the epilogue
// (DeepSeek-V3.2 summary card, "How DSA Works": the lightning indexer scores
// every key of a query cheaply in FP8; news article on DeepSeek-V3.2,
// sparse-attention section: a few low-precision heads on every token pair).
//
//   I[t,s] = sk[s] * sum_j (w[t,j] sq[t,j]) * ReLU(<q8[t,j,:], k8[s,:]>)
// (the positive scales move out of the ReLU).
//
// Layout: keys on M (128 TMEM lanes), (4 queries x 64 heads) on N = 256, so
// the head sum of one (key, query) pair lies in one thread's TMEM row and
// needs no cross-thread reduction.  K = 128 (4 MMAs of K = 32).  D is double
// buffered (2 x 256 of the 512 TMEM columns) so the epilogue of tile g
// overlaps the MMAs of tile g+1.
//
// Persistent: one CTA per SM walks work items (group of 4 consecutive query
// rows, chunk of CH key tiles), strided over the grid.  When the four rows
// belong to one sequence (prefill chunks) they share every key tile: one
// pass with N = 256.  Otherwise (decode batches, chunk boundaries) each
// query makes its own pass over its own sequence with N = 64.  The query
// tile (B operand) and the folded weights are double buffered across items.
// Key tiles are loaded by TMA: 2 boxes of 64 rows, so paged caches whose
// block size is a multiple of 64 are read block by block.
//
// An accumulator buffer holds one shared-pass tile (N = 256) or up to four
// consecutive per-query tiles (N = 64 each, in 64-column slices), so that
// per-query work (decode batches) keeps eight tiles in flight.
//
// Warps: 0 = TMA producer, 1 = TMEM owner + MMA issuer, 2..17 = epilogue
// (warp w reads TMEM lane quadrant w%4 and the 64 columns of slice (w-2)/4:
// the slice's query of a shared pass, or the slice's own per-query tile).
// A score is the sum of four 16-head partials in one fixed order in both
// modes, so a query's scores do not depend on its batch.  All waits are
// bounded (see tc.cuh).
#include <algorithm>
#include <cstdint>
#include <cstddef>

#include "indexer_epi.cuh"
#include "launch.h"
#include "tc.cuh"
#include "tmap.h"

namespace dsa {
namespace {
using namespace tc;

constexpr int kQG = 4;                          // queries per group
constexpr int kHI = 64, kDI = 128;
constexpr int kKT = 128;                        // keys per tile
constexpr int kStagesA = 6;
constexpr uint32_t kBBytes = kQG * kHI * 128;   // 32 KB
constexpr uint32_t kABytes = kKT * 128;         // 16 KB
constexpr uint32_t kOffA = 2 * kBBytes;
constexpr uint32_t kSmemBytes = kOffA + kStagesA * kABytes;   // 160 KB
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;
constexpr int kThreads = 576;
constexpr int kEpiThreads = 512;

constexpr int kStageCap = 128;                  // candidates an epilogue warp stages before a flush (kFilter)

// One group of 4 consecutive query rows: either one pass over a shared
// sequence (uniform) or one pass per active query.
struct Group {
  int seq[kQG], pos[kQG];
  bool active[kQG];
  bool uniform;
  int npass;
  int pass_q[kQG], pass_seq[kQG], pass_T[kQG], pass_N[kQG], pass_maxpos[kQG];   // T tiles, N ordinals
};

struct __align__(16) Shared {
  uint64_t stage[kEpiThreads / 32][kStageCap];  // kFilter: each epilogue warp's admitted candidates
  uint64_t a_full[kStagesA], a_empty[kStagesA], d_full[2], d_empty[2];
  uint64_t b_full[2], b_empty[2], epi_sync[2], fin;
  alignas(16) float wq[2][kQG][kHI];   // w * q_scale of the item's group (double buffered; read as float4)
  Group grp[2];                        // the epilogue's description of its current item (double buffered)
  uint32_t tmem_base;
  int abort;
};

static_assert(offsetof(Shared, wq) % 16 == 0, "wq is read with 16-byte vector loads");

// Which key tiles a launch processes (IndexerOut::mode): every tile (kFull),
// the sampled tiles 0, m, 2m, ... (kSample), or all the others (kFilter).
// A pass's tiles are numbered by ordinal o = 0, 1, ...; tile(o) maps an
// ordinal to its key tile.
template <int kMode>
struct TileMap {
  static constexpr int mode = kMode;
  int m;
  uint32_t inv;   // kFilter: division by m - 1 as a multiply-high (exact for ordinals and m below 2^16)
  __device__ __forceinline__ int count(int T) const {
    return mode == IndexerOut::kFull ? T : mode == IndexerOut::kSample ? (T + m - 1) / m : T - (T + m - 1) / m;
  }
  __device__ __forceinline__ int tile(int o) const {
    if (mode == IndexerOut::kFull) return o;
    if (mode == IndexerOut::kSample) return o * m;
    const int q = m == 2 ? o : (int)__umulhi((uint32_t)o, inv);   // o / (m - 1)
    return q * m + 1 + (o - q * (m - 1));
  }
};

// The multiply-high reciprocal of d >= 2 (o / d == umulhi(o, r) for o, d < 2^16;
// d = 1 needs 2^32 and is handled by the caller).
__host__ __device__ __forceinline__ uint32_t recip32(uint32_t d) {
  return d <= 1u ? 0u : (uint32_t)(0xffffffffull / d) + 1u;
}


template <class TM>
__device__ __forceinline__ void describe_group(const QueryBatch& qb, const CacheMap& cm, int gi, int min_pos,
                                               const TM& tm, Group& G) {
  int first_seq = -1, nact = 0;
  bool same = true;
#pragma unroll
  for (int qq = 0; qq < kQG; ++qq) {
    const int r = gi * kQG + qq;
    int sq = 0, ps = -1;
    bool act = false;
    if (r < qb.num_q) {
      sq = __ldg(qb.q_seq + r);
      ps = __ldg(qb.q_pos + r);
      act = ps >= min_pos && ps < qb.max_kv && sq >= 0 && sq < cm.num_seqs;
    }
    G.seq[qq] = sq;
    G.pos[qq] = ps;
    G.active[qq] = act;
    if (act) {
      if (first_seq < 0) first_seq = sq;
      else if (sq != first_seq) same = false;
      ++nact;
    }
  }
  G.uniform = same && nact > 0;
  int np = 0;
  if (G.uniform) {
    int mp = -1;
#pragma unroll
    for (int qq = 0; qq < kQG; ++qq)
      if (G.active[qq]) mp = max(mp, G.pos[qq]);
    G.pass_q[0] = -1;
    G.pass_seq[0] = first_seq;
    G.pass_maxpos[0] = mp;
    G.pass_T[0] = mp / kKT + 1;
    np = 1;
  } else {
#pragma unroll
    for (int qq = 0; qq < kQG; ++qq) {
      if (!G.active[qq]) continue;
      G.pass_q[np] = qq;
      G.pass_seq[np] = G.seq[qq];
      G.pass_maxpos[np] = G.pos[qq];
      G.pass_T[np] = G.pos[qq] / kKT + 1;
      ++np;
    }
  }
  G.npass = np;
#pragma unroll
  for (int p = 0; p < kQG; ++p) G.pass_N[p] = p < np ? tm.count(G.pass_T[p]) : 0;
}

// Ordinals of pass p in chunk c: [t0, t1).
__device__ __forceinline__ void pass_range(const Group& G, int p, int c, int ch, int& t0, int& t1) {
  t0 = c * ch;
  t1 = min(t0 + ch, G.pass_N[p]);
}

// Entry e of an item (its tiles in pass order) -> pass and tile.
__device__ __forceinline__ void entry_at(const Group& G, int c, int ch, int e, int& p_out, int& t_out) {
  p_out = 0;
  t_out = 0;
  for (int p = 0; p < G.npass; ++p) {
    int t0, t1;
    pass_range(G, p, c, ch, t0, t1);
    const int n = max(0, t1 - t0);
    if (e < n) {
      p_out = p;
      t_out = t0 + e;
      return;
    }
    e -= n;
  }
}

__device__ __forceinline__ int item_tiles(const Group& G, int c, int ch) {
  int n = 0;
  for (int p = 0; p < G.npass; ++p) {
    int t0, t1;
    pass_range(G, p, c, ch, t0, t1);
    n += max(0, t1 - t0);
  }
  return n;
}

// kFilter: an epilogue warp's staged candidates (warp-uniform state): the
// query row they belong to and how many are staged in its buffer.
struct Stager {
  int row = -1;
  uint32_t n = 0;
};

// Appends the staged candidates to the query's list: one atomic reserves
// their slots, then the warp copies them (entries past the list's capacity
// are counted but not stored).  Called by a whole warp.
__device__ __forceinline__ void stage_flush(const IndexerOut& o, Stager& st, const uint64_t* buf, int lane) {
  if (st.n == 0) return;
  uint32_t base = 0;
  if (lane == 0) base = atomicAdd(o.cnt + st.row, st.n);
  base = __shfl_sync(0xffffffffu, base, 0);
  __syncwarp();
  uint64_t* dst = o.cand + (int64_t)st.row * o.cap;
  for (uint32_t i = lane; i < st.n; i += 32)
    if (base + i < (uint32_t)o.cap) dst[base + i] = buf[i];
  __syncwarp();
  st.n = 0;
}

// Output of one (key, query) score, by mode.  Called by a whole warp (the
// filter stages with a warp ballot): row_q, t (the tile's ordinal) and thr
// are warp-uniform, s is this lane's key, live whether it is a causal key of
// a valid query with a readable cache row.
template <int kMode>
__device__ __forceinline__ void emit(const IndexerOut& o, const QueryBatch& qb, int row_q, int t, int s, float sc,
                                     bool live, uint64_t thr, int lane, Stager& st, uint64_t* buf) {
  if (kMode == IndexerOut::kFull) {
    if (s < qb.max_kv && row_q < qb.num_q) o.scores[(int64_t)row_q * o.ld + s] = live ? sc : -INFINITY;
  } else if (kMode == IndexerOut::kSample) {
    if (row_q < qb.num_q) o.scores[(int64_t)row_q * o.ld + t * kKT + (s & (kKT - 1))] = live ? sc : -INFINITY;
  } else {
    // composite key >= thr, decided on the score (the high word orders like
    // the score with -0 == +0) and the position (the low word)
    // (a threshold of 0 admits every key: its high word stands for no score)
    const float ts = key_score((uint32_t)(thr >> 32));
    const int tp = composite_pos(thr);
    const bool admit = live && row_q < qb.num_q && (thr == 0ull || sc > ts || (sc == ts && s <= tp));
    const uint32_t m = __ballot_sync(0xffffffffu, admit);
    if (!m) return;
    const uint64_t ck = composite_key(sc, s);
    if (st.row != row_q) {   // the warp moves on to another query's candidates
      stage_flush(o, st, buf, lane);
      st.row = row_q;
    }
    const uint32_t nn = __popc(m);
    if (st.n + nn > (uint32_t)kStageCap) stage_flush(o, st, buf, lane);
    if (admit) buf[st.n + __popc(m & ((1u << lane) - 1u))] = ck;
    st.n += nn;
  }
}

// kMode: the pass (IndexerOut::kFull, kSample, kFilter) as a compile-time
// constant, so the per-key epilogue carries no mode branches.
template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
indexer_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  QueryBatch qb, CacheMap cm, const float* __restrict__ q_scale, const float* __restrict__ w,
                  const float* __restrict__ k_scale, const IndexerOut out, int ngroups, int nchunk, int ch,
                  long long wait_limit, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Shared S;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort = &S.abort;
  const uint32_t sB = smem_u32(sm), sA = smem_u32(sm + kOffA);
  const int n_items = ngroups * nchunk;
  const TileMap<kMode> tmap{out.m, recip32((uint32_t)max(out.m - 1, 1))};
  float* __restrict__ scores = out.scores;
  const int64_t ld = out.ld;

  if (tid == 0) {
    for (int s = 0; s < kStagesA; ++s) {
      mbar_init(&S.a_full[s], 1);
      mbar_init(&S.a_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.d_full[b], 1);
      mbar_init(&S.d_empty[b], kEpiThreads);
      mbar_init(&S.b_full[b], 1);
      mbar_init(&S.b_empty[b], 1);
      mbar_init(&S.epi_sync[b], kEpiThreads);
    }
    mbar_init(&S.fin, 1);
    S.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();      // the set-up above ran while the stream's previous kernel finished
  pdl_release();
  const uint32_t tmem = S.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      uint32_t g = 0, j = 0;   // key tiles and query tiles issued
      for (int item = blockIdx.x; item < n_items && !*abort; item += gridDim.x) {
        const int gi = item % ngroups, c = item / ngroups;
        Group G;
        describe_group(qb, cm, gi, out.min_pos, tmap, G);
        if (item_tiles(G, c, ch) == 0) continue;
        const int bb = j & 1;
        if (!mbar_wait(&S.b_empty[bb], ((j >> 1) & 1) ^ 1, abort, wait_limit)) break;
        mbar_arrive_expect_tx(&S.b_full[bb], kBBytes);
        tma_load_2d(sB + bb * kBBytes, &tm_q, 0, gi * kQG * kHI, &S.b_full[bb]);
        ++j;
        bool ok = true;
        for (int p = 0; p < G.npass && ok; ++p) {
          const int seq = G.pass_seq[p], mp = G.pass_maxpos[p];
          int t0, t1;
          pass_range(G, p, c, ch, t0, t1);
          for (int t = t0; t < t1; ++t, ++g) {
            const int st = g % kStagesA;
            if (!(ok = mbar_wait(&S.a_empty[st], ((g / kStagesA) & 1) ^ 1, abort, wait_limit))) break;
            int64_t rows[2];
            uint32_t bytes = 0;
            const int tile = tmap.tile(t);
            for (int hh = 0; hh < 2; ++hh) {
              const int sh = tile * kKT + 64 * hh;
              rows[hh] = -1;
              if (sh > mp) continue;
              if (cm.block_size == 0) {
                rows[hh] = (int64_t)seq * cm.seq_stride + sh;
              } else {
                const int blk = sh / cm.block_size;
                const int phys =
                    blk < cm.max_blocks ? __ldg(cm.block_table + (int64_t)seq * cm.max_blocks + blk) : -1;
                const int64_t r0 = (int64_t)phys * cm.block_size + (sh - blk * cm.block_size);
                if (phys < 0 || r0 + 64 > cm.num_rows) flag_error(err, DSA_ERR_BOUNDS);
                else rows[hh] = r0;
              }
              if (rows[hh] >= 0) bytes += 64 * 128;
            }
            mbar_arrive_expect_tx(&S.a_full[st], bytes);
            for (int hh = 0; hh < 2; ++hh)
              if (rows[hh] >= 0)
                tma_load_2d(sA + st * kABytes + hh * 8192, &tm_k, 0, (int32_t)rows[hh], &S.a_full[st]);
          }
        }
        if (!ok) break;
      }
      // Before the CTA may exit (after an abort the consumers stop waiting),
      // every TMA load issued here must have landed: wait for the last phase
      // armed on each stage and query buffer (each completes by its own bytes).
      for (uint32_t st = 0; st < (uint32_t)kStagesA && st < g; ++st) {
        const uint32_t last = st + kStagesA * ((g - 1 - st) / kStagesA);
        mbar_wait_own(&S.a_full[st], (last / kStagesA) & 1);
      }
      for (uint32_t b = 0; b < 2 && b < j; ++b) {
        const uint32_t last = b + 2 * ((j - 1 - b) / 2);
        mbar_wait_own(&S.b_full[b], (last >> 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    uint32_t g = 0, j = 0, dq = 0;   // key tiles, items with tiles, accumulator-buffer uses
    for (int item = blockIdx.x; item < n_items && !*abort; item += gridDim.x) {
      const int gi = item % ngroups, c = item / ngroups;
      Group G;
      describe_group(qb, cm, gi, out.min_pos, tmap, G);
      if (item_tiles(G, c, ch) == 0) continue;
      const int bb = j & 1;
      if (!mbar_wait_warp(&S.b_full[bb], (j >> 1) & 1, abort, wait_limit)) break;
      bool ok = true;
      // One accumulator buffer holds one shared-pass tile (4 queries x 64
      // heads) or up to four consecutive per-query tiles (64 columns each),
      // so that per-query work keeps eight tiles in flight, not two.
      const bool uni = G.uniform;
      const int ne = item_tiles(G, c, ch), per_d = uni ? 1 : 4;
      const uint32_t idesc = idesc_e4m3(128, uni ? 256 : 64);
      if (uni) {   // one pass, one tile per buffer
        int t0, t1;
        pass_range(G, 0, c, ch, t0, t1);
        const uint32_t boff = bb * kBBytes;
        for (int t = t0; t < t1; ++t, ++g, ++dq) {
          const int st = g % kStagesA, b = dq & 1;
          if (!(ok = mbar_wait_warp(&S.a_full[st], (g / kStagesA) & 1, abort, wait_limit))) break;
          if (!(ok = mbar_wait_warp(&S.d_empty[b], ((dq >> 1) & 1) ^ 1, abort, wait_limit))) break;
          tc_fence_after();
          if (lane == 0) {
            const Desc2 ad = desc2(sdesc(sA + st * kABytes, 16, 1024)), bd = desc2(sdesc(sB + boff, 16, 1024));
            mma_e4m3_2<0>(tmem + 256 * b, ad, bd, idesc);
#pragma unroll
            for (int kk = 1; kk < 4; ++kk) mma_e4m3_2<1>(tmem + 256 * b, desc_at(ad, kk * 32), desc_at(bd, kk * 32), idesc);
            mma_commit(&S.a_empty[st]);
            mma_commit(&S.d_full[b]);
          }
          __syncwarp();
        }
      }
      for (int e0 = 0; e0 < ne && ok && !uni; e0 += per_d, ++dq) {
        const int b = dq & 1, nsub = min(per_d, ne - e0);
        if (!(ok = mbar_wait_warp(&S.d_empty[b], ((dq >> 1) & 1) ^ 1, abort, wait_limit))) break;
        for (int u = 0; u < nsub; ++u, ++g) {
          int p, t;
          entry_at(G, c, ch, e0 + u, p, t);
          const uint32_t boff = bb * kBBytes + (uni ? 0u : (uint32_t)G.pass_q[p] * (kHI * 128));
          const int st = g % kStagesA;
          if (!(ok = mbar_wait_warp(&S.a_full[st], (g / kStagesA) & 1, abort, wait_limit))) break;
          tc_fence_after();
          if (lane == 0) {
            const Desc2 ad = desc2(sdesc(sA + st * kABytes, 16, 1024)), bd = desc2(sdesc(sB + boff, 16, 1024));
            mma_e4m3_2<0>(tmem + 256 * b + 64 * u, ad, bd, idesc);
#pragma unroll
            for (int kk = 1; kk < 4; ++kk)
              mma_e4m3_2<1>(tmem + 256 * b + 64 * u, desc_at(ad, kk * 32), desc_at(bd, kk * 32), idesc);
            mma_commit(&S.a_empty[st]);
          }
          __syncwarp();
        }
        if (!ok) break;
        if (lane == 0) mma_commit(&S.d_full[b]);
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) mma_commit(&S.b_empty[bb]);   // this item's query tile is no longer read
      __syncwarp();
      ++j;
    }
    if (lane == 0) mma_commit(&S.fin);
    __syncwarp();
    mbar_wait_own(&S.fin, 0);
  } else {
    // ------------------------------------------------------------ epilogue
    const int qd = warp & 3, uq = (warp - 2) >> 2, et = tid - 64;
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    Stager stg;
    uint64_t* sbuf = S.stage[warp - 2];
    uint32_t dq = 0, ep = 0;   // accumulator-buffer uses, items
    for (int item = blockIdx.x; item < n_items && !*abort; item += gridDim.x) {
      const int gi = item % ngroups, c = item / ngroups;
      const int bb = ep & 1;
      {   // the item's description (one copy in shared memory for all epilogue
          // threads, instead of one per thread in local memory) and the folded
          // weights of its group (threads et < 256 fetch one each).  Slot bb
          // is rewritten two items later, once every epilogue thread has
          // passed the next item's barrier, i.e. finished with this item.
        if (et == 0) describe_group(qb, cm, gi, out.min_pos, tmap, S.grp[bb]);
        if (et < kQG * kHI) {
          const int qq = et / kHI, jj = et % kHI, r = gi * kQG + qq;
          S.wq[bb][qq][jj] = r < qb.num_q ? idx_epi::fold_weight(jj, __ldg(w + (int64_t)r * kHI + jj) *
                                                                         __ldg(q_scale + (int64_t)r * kHI + jj))
                                          : 0.f;
        }
        mbar_arrive(&S.epi_sync[bb]);
        if (!mbar_wait_warp(&S.epi_sync[bb], (ep >> 1) & 1, abort, wait_limit)) break;
        ++ep;
      }
      const Group& G = S.grp[bb];
      if (item_tiles(G, c, ch) > 0) {
        bool ok = true;
        const bool uni = G.uniform;
        const int ne = item_tiles(G, c, ch), per_d = uni ? 1 : 4;
        if (uni) {   // one pass, one tile per buffer: this warp's query is uq
          int t0, t1;
          pass_range(G, 0, c, ch, t0, t1);
          const int seq = G.pass_seq[0], maxpos = G.pass_maxpos[0];
          const bool q_act = G.active[uq];
          const int q_pos = G.pos[uq], row_q = gi * kQG + uq;
          const float4* wq4 = reinterpret_cast<const float4*>(S.wq[bb][uq]);
          const uint64_t thr = kMode == IndexerOut::kFilter && row_q < qb.num_q ? __ldg(out.thr + row_q) : 0ull;
          // a contiguous cache holds this pass's keys at rows seq_base + s: one
          // range check per item instead of one row lookup per key
          const int64_t seq_base = (int64_t)seq * cm.seq_stride;
          const bool contig = cm.block_size == 0 && seq_base + maxpos < cm.num_rows;
          for (int t = t0; t < t1; ++t, ++dq) {
            const int b = dq & 1;
            // this lane's key and its scale, fetched before the wait
            const int s = tmap.tile(t) * kKT + qd * 32 + lane;
            float sk = 0.f;
            bool key_ok = s <= maxpos;
            if (key_ok) {
              const int64_t row = contig ? seq_base + s : cache_row(cm, seq, s, err);
              key_ok = row >= 0;
              if (key_ok) sk = __ldg(k_scale + row);
            }
            if (!(ok = mbar_wait_warp(&S.d_full[b], (dq >> 1) & 1, abort, wait_limit))) break;
            tc_fence_after();
            const float acc = idx_epi::head_sum64(tmem + lane_base + 256 * b + uq * 64, wq4);
            emit<kMode>(out, qb, row_q, t, s, acc * sk, q_act && key_ok && s <= q_pos, thr, lane, stg, sbuf);
            tc_fence_before();
            mbar_arrive(&S.d_empty[b]);
          }
        }
        for (int e0 = 0; e0 < ne && ok && !uni; e0 += per_d, ++dq) {
          const int b = dq & 1, nsub = min(per_d, ne - e0);
          // this warp's part of the buffer: query uq of a shared-pass tile, or
          // per-query tile e0 + uq (both at columns 64 uq)
          const bool mine = uni || uq < nsub;
          int p = 0, t = 0;
          entry_at(G, c, ch, uni ? e0 : e0 + min(uq, nsub - 1), p, t);
          const int qq = uni ? uq : G.pass_q[p];
          // this lane's key and its scale, fetched before the wait so that
          // the load (from HBM when every key is read once) overlaps the MMA
          const int s = tmap.tile(t) * kKT + qd * 32 + lane;
          const int row_q = gi * kQG + qq;
          const uint64_t thr =
              kMode == IndexerOut::kFilter && mine && row_q < qb.num_q ? __ldg(out.thr + row_q) : 0ull;
          float sk = 0.f;
          bool key_ok = mine && s <= G.pass_maxpos[p];
          if (key_ok) {
            const int64_t pbase = (int64_t)G.pass_seq[p] * cm.seq_stride;
            const bool contig = cm.block_size == 0 && pbase + G.pass_maxpos[p] < cm.num_rows;
            const int64_t row = contig ? pbase + s : cache_row(cm, G.pass_seq[p], s, err);
            key_ok = row >= 0;
            if (key_ok) sk = __ldg(k_scale + row);
          }
          if (!(ok = mbar_wait_warp(&S.d_full[b], (dq >> 1) & 1, abort, wait_limit))) break;
          tc_fence_after();
          if (mine) {
            // the same arithmetic as the shared pass, so a query's scores do
            // not depend on its batch
            const float4* wq4 = reinterpret_cast<const float4*>(S.wq[bb][qq]);
            const float acc = idx_epi::head_sum64(tmem + lane_base + 256 * b + uq * 64, wq4);
            emit<kMode>(out, qb, row_q, t, s, acc * sk, G.active[qq] && key_ok && s <= G.pos[qq], thr, lane, stg, sbuf);
          }
          tc_fence_before();
          mbar_arrive(&S.d_empty[b]);
        }
        if (!ok) break;
        if (kMode == IndexerOut::kFilter) stage_flush(out, stg, sbuf, lane);
      }
      // the item holding a group's last chunk also writes -inf from the end
      // of the group's scanned tiles to max_kv
      if (kMode == IndexerOut::kFull && c == nchunk - 1) {
        for (int qq = 0; qq < kQG; ++qq) {
          const int row_q = gi * kQG + qq;
          if (row_q >= qb.num_q) break;
          int from = 0;
          if (G.active[qq]) {
            int T = 0;
            for (int p = 0; p < G.npass; ++p)
              if (G.uniform || G.pass_q[p] == qq) T = G.pass_T[p];
            from = T * kKT;
          }
          for (int s2 = from + et; s2 < qb.max_kv; s2 += kEpiThreads) scores[(int64_t)row_q * ld + s2] = -INFINITY;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (tid == 0 && S.abort) flag_error(err, DSA_ERR_TIMEOUT);
}

int sm_count_here() {
  static int cache[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (!cache[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 148;
  }
  return cache[dev];
}

}  // namespace

bool indexer_tc_supported(const CacheMap& cm, const dsa_indexer_inputs& ix) {
  if (ix.dtype != DSA_FP8_E4M3 || ix.heads != kHI || ix.dim != kDI) return false;
  if (cm.block_size != 0 && cm.block_size % 64 != 0) return false;
  return true;
}

cudaError_t launch_indexer_tc(const QueryBatch& qb, const CacheMap& cm, const dsa_indexer_inputs& ix,
                              const IndexerOut& out, int* err, cudaStream_t stream, long long wait_limit) {
  const int tmax = indexer_tile_count(out, (qb.max_kv + kKT - 1) / kKT);   // most tiles (ordinals) of one pass
  if (tmax == 0 || qb.num_q == 0) return cudaSuccess;
  CUtensorMap tm_q, tm_k;
  if (!make_tmap_rows128(&tm_q, ix.q, (uint64_t)qb.num_q * kHI, 128, kQG * kHI)) return cudaErrorInvalidValue;
  if (!make_tmap_rows128(&tm_k, ix.k, (uint64_t)cm.num_rows, 128, 64)) return cudaErrorInvalidValue;
  const int sms = sm_count_here();
  const int ngroups = (qb.num_q + kQG - 1) / kQG;
  // chunks of ch key tiles: the CTAs take items round-robin, so pick the ch
  // that minimises the busiest CTA's load (items x tiles, plus about one
  // tile's worth of fixed cost per item); ties go to the larger chunk
  int ch = 2;
  int64_t best = INT64_MAX;
  for (int c = 2; c <= 64; ++c) {
    const int64_t nch = (tmax + c - 1) / c, items = (int64_t)ngroups * nch;
    const int64_t per_cta = (items + sms - 1) / sms;
    const int64_t cost = per_cta * (std::min<int64_t>(c, tmax) + 1);
    if (cost <= best) {
      best = cost;
      ch = c;
    }
  }
  const int nchunk = (tmax + ch - 1) / ch;
  const int grid = (int)std::min<int64_t>(sms, (int64_t)ngroups * nchunk);
  auto kern = out.mode == IndexerOut::kSample   ? indexer_tc_kernel<IndexerOut::kSample>
              : out.mode == IndexerOut::kFilter ? indexer_tc_kernel<IndexerOut::kFilter>
                                                 : indexer_tc_kernel<IndexerOut::kFull>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(kThreads), kSmemAlloc, stream, tm_q, tm_k, qb, cm, ix.q_scale, ix.w,
                    ix.k_scale, out, ngroups, nchunk, ch, wait_limit, err);
}

}  // namespace dsa
