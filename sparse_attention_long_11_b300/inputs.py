"""Seeded synthetic workloads for the DeepSeek Sparse Attention (DSA) hot path.

This module only *makes inputs*: random tensors of the shapes, dtypes and
distributions of the five DSA workloads, the FP8/BF16 encodings of those
tensors, and the batch layout (which query sits at which position of which
sequence, and where each cache row lives).  It holds none of the method's
arithmetic: no indexer score, no selection, no softmax.  Both the CUDA path
and the CPU oracle consume the tensors built here.

Every tensor is drawn from its own ``torch.Generator`` whose seed is derived
from (workload seed, tensor name), so adding or reordering tensors never
changes the others.  Generation can run on the CPU (small cases, CPU tests) or
directly on a CUDA device (full-size cases: config 4 holds ~10 GB of bf16
queries); the two devices give different numbers for the same seed, so a test
always hands the *same* generated tensors to both sides.

Workloads (sizes from the DSA description of DeepSeek-V3.2: 128 query heads
sharing one 576-wide latent KV row with a 512-wide value part, an FP8
lightning indexer with 64 heads of width 128, top-k of 2048):

  tiny     L=256 prefill, fp32, H_I=4, d_I=64, k=32, 8 heads, d=128
  prefill  L=4096 prefill, one chunk
  long     L=32768 prefill in 8 chunks of 4096 queries
  decode   64 sequences x 65536 cached rows, one query each
  mixed    8 paged sequences (block 64, permuted), lengths U{8192..131072},
           a prefill chunk of 8192 queries plus 32 single-token decode
           queries at the tail of each sequence
"""
from __future__ import annotations

import dataclasses
import math
import zlib
from typing import List, Optional, Tuple

import torch

FP8_MAX = 448.0  # largest finite OCP e4m3 ("fn") magnitude


def _gen(seed: int, name: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + zlib.crc32(name.encode())) & 0x7FFF_FFFF_FFFF)
    return g


def randn(shape, seed: int, name: str, device="cpu", std: float = 1.0) -> torch.Tensor:
    x = torch.randn(shape, generator=_gen(seed, name, device), device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x


def rand(shape, seed: int, name: str, device="cpu", scale: float = 1.0) -> torch.Tensor:
    x = torch.rand(shape, generator=_gen(seed, name, device), device=device, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x


def quantize_fp8_rows(x: torch.Tensor) -> Tuple[torch.Tensor, torch.Tensor]:
    """Encode the last axis of ``x`` as OCP e4m3 bytes with one fp32 scale per row.

    scale = amax(|row|) / 448 (1.0 for an all-zero row); code = RNE(x / scale)
    saturated to +-448.  Returns (uint8 codes, fp32 scales).  This is input
    preparation: the indexer consumes the bytes and scales as given.
    """
    amax = x.abs().amax(dim=-1)
    # tensor / tensor: an IEEE fp32 division (dividing by a Python number
    # multiplies by its reciprocal on the GPU, which can differ in the last bit)
    scale = torch.where(amax > 0, amax / torch.full_like(amax, FP8_MAX), torch.ones_like(amax))
    y = (x / scale.unsqueeze(-1)).clamp_(-FP8_MAX, FP8_MAX)
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.contiguous(), scale.contiguous()


@dataclasses.dataclass
class Workload:
    """One DSA batch: indexer inputs, attention inputs, batch layout.

    Cache tensors are *physical*: row r of ``k_idx``/``k_scale``/``kv`` is the
    row the batch layout maps a (sequence, position) pair to.  ``logical_rows``
    gives that map for the oracle.
    """
    name: str
    seed: int
    # indexer
    idx_dtype: str            # "f32" or "fp8"
    H_I: int
    d_I: int
    q_idx: torch.Tensor       # [num_q, H_I, d_I] f32 or uint8 (e4m3 codes)
    q_scale: Optional[torch.Tensor]  # [num_q, H_I] f32 (fp8 only)
    w: torch.Tensor           # [num_q, H_I] f32
    k_idx: torch.Tensor       # [rows, d_I] f32 or uint8
    k_scale: Optional[torch.Tensor]  # [rows] f32 (fp8 only)
    topk: int
    # attention
    attn_dtype: str           # "f32", "bf16", or "fp8kv" (bf16 queries, FP8 latent cache)
    H: int
    d_qk: int
    d_v: int
    q: torch.Tensor           # [num_q, H, d_qk]
    kv: torch.Tensor          # [rows, d_qk] (uint8 e4m3 codes for "fp8kv")
    softmax_scale: float
    # batch layout
    q_seq: torch.Tensor       # [num_q] int32
    q_pos: torch.Tensor       # [num_q] int32
    seq_lens: List[int]       # cached rows per sequence (host)
    seq_stride: int           # contiguous layout: row = seq * seq_stride + pos
    block_table: Optional[torch.Tensor]  # [num_seqs, max_blocks] int32 (paged) or None
    block_size: int
    chunks: List[Tuple[int, int]]  # query-row ranges processed as one call each
    kv_scale: Optional[torch.Tensor] = None  # [rows] f32 ("fp8kv" only)

    @property
    def num_q(self) -> int:
        return int(self.q_pos.shape[0])

    @property
    def num_seqs(self) -> int:
        return len(self.seq_lens)

    @property
    def num_rows(self) -> int:
        return int(self.kv.shape[0])

    @property
    def max_kv(self) -> int:
        return int(self.q_pos.max().item()) + 1 if self.num_q else 0

    def logical_rows(self, seq: int, n: int) -> torch.Tensor:
        """Physical row of positions 0..n-1 of sequence ``seq`` (int64, CPU)."""
        pos = torch.arange(n, dtype=torch.int64)
        if self.block_table is None:
            return pos + seq * self.seq_stride
        bt = self.block_table[seq].to("cpu", torch.int64)
        return bt[pos // self.block_size] * self.block_size + pos % self.block_size


CONFIG_NAMES = ["tiny", "prefill", "long", "decode", "mixed"]


def _runs_layout(runs, device):
    """runs: list of (seq, first_pos, n) -> q_seq, q_pos int32 tensors."""
    seqs, poss = [], []
    for seq, p0, n in runs:
        seqs.append(torch.full((n,), seq, dtype=torch.int32))
        poss.append(torch.arange(p0, p0 + n, dtype=torch.int32))
    return torch.cat(seqs).to(device), torch.cat(poss).to(device)


def _indexer_fp8(seed, num_q, rows, device, w_dist):
    q_raw = randn((num_q, 64, 128), seed, "q_idx", device)
    q_idx, q_scale = quantize_fp8_rows(q_raw)
    del q_raw
    k_raw = randn((rows, 128), seed, "k_idx", device)
    k_idx, k_scale = quantize_fp8_rows(k_raw)
    del k_raw
    if w_dist == "uniform":
        w = rand((num_q, 64), seed, "w", device, scale=1.0 / math.sqrt(64))
    else:
        w = randn((num_q, 64), seed, "w", device)
    return q_idx, q_scale, w, k_idx, k_scale


def _bf16_normal(shape, seed, name, device, chunk_rows=1 << 14):
    """N(0,1) rounded to bf16, drawn in row chunks to bound the fp32 transient."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(shape[0], -1)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        flat[r0:r1] = randn((r1 - r0, flat.shape[1]), seed, f"{name}[{r0}]", device).to(torch.bfloat16)
    return out


def with_fp8_kv(wl: Workload, chunk_rows: int = 1 << 16) -> Workload:
    """The same workload with its latent KV cache stored as FP8: every bf16
    row encoded like the indexer keys (e4m3 codes, one fp32 scale amax/448),
    in row chunks to bound the fp32 transient.  Input preparation only."""
    n = wl.kv.shape[0]
    codes = torch.empty(wl.kv.shape, dtype=torch.uint8, device=wl.kv.device)
    scale = torch.empty((n,), dtype=torch.float32, device=wl.kv.device)
    for r0 in range(0, n, chunk_rows):
        r1 = min(n, r0 + chunk_rows)
        codes[r0:r1], scale[r0:r1] = quantize_fp8_rows(wl.kv[r0:r1].float())
    return dataclasses.replace(wl, attn_dtype="fp8kv", kv=codes, kv_scale=scale)


def make_tiny(seed=0, device="cpu", L=256, topk=32) -> Workload:
    """L=256 causal prefill, fp32 everywhere; indexer 4 heads x 64, attention 8 heads x 128."""
    q_seq, q_pos = _runs_layout([(0, 0, L)], device)
    d = 128
    return Workload(
        name="tiny", seed=seed, idx_dtype="f32", H_I=4, d_I=64,
        q_idx=randn((L, 4, 64), seed, "q_idx", device), q_scale=None,
        w=rand((L, 4), seed, "w", device),
        k_idx=randn((L, 64), seed, "k_idx", device), k_scale=None,
        topk=topk, attn_dtype="f32", H=8, d_qk=d, d_v=d,
        q=randn((L, 8, d), seed, "q", device, std=1.0 / math.sqrt(d)),
        kv=randn((L, d), seed, "kv", device, std=1.0 / math.sqrt(d)),
        softmax_scale=1.0 / math.sqrt(d),
        q_seq=q_seq, q_pos=q_pos, seq_lens=[L], seq_stride=L,
        block_table=None, block_size=0, chunks=[(0, L)])


def make_prefill(seed=0, device="cpu", L=4096, chunk=None, name="prefill", topk=2048,
                 q_rows: Optional[Tuple[int, int]] = None) -> Workload:
    """Single-sequence causal prefill of length L with the DSA shapes.

    ``chunk`` splits the queries into calls of that many rows (the long
    prefill uses 4096).  ``q_rows`` keeps only query positions [a, b) (all
    keys 0..L-1 stay cached): used for bounded samples of a long prefill.
    """
    a, b = q_rows if q_rows is not None else (0, L)
    nq = b - a
    q_seq, q_pos = _runs_layout([(0, a, nq)], device)
    q_idx, q_scale, w, k_idx, k_scale = _indexer_fp8(seed, nq, L, device, "uniform")
    chunk = chunk or nq
    return Workload(
        name=name, seed=seed, idx_dtype="fp8", H_I=64, d_I=128,
        q_idx=q_idx, q_scale=q_scale, w=w, k_idx=k_idx, k_scale=k_scale,
        topk=topk, attn_dtype="bf16", H=128, d_qk=576, d_v=512,
        q=_bf16_normal((nq, 128, 576), seed, "q", device),
        kv=_bf16_normal((L, 576), seed, "kv", device),
        softmax_scale=1.0 / math.sqrt(576),
        q_seq=q_seq, q_pos=q_pos, seq_lens=[L], seq_stride=L,
        block_table=None, block_size=0,
        chunks=[(c, min(nq, c + chunk)) for c in range(0, nq, chunk)])


def make_long(seed=0, device="cpu", L=32768, chunk=4096) -> Workload:
    return make_prefill(seed, device, L=L, chunk=chunk, name="long")


def make_decode(seed=0, device="cpu", batch=64, ctx=65536, topk=2048) -> Workload:
    """``batch`` sequences of ``ctx`` cached rows, one query each at position ctx-1."""
    q_seq, q_pos = _runs_layout([(b, ctx - 1, 1) for b in range(batch)], device)
    rows = batch * ctx
    q_idx, q_scale, w, k_idx, k_scale = _indexer_fp8(seed, batch, rows, device, "normal")
    return Workload(
        name="decode", seed=seed, idx_dtype="fp8", H_I=64, d_I=128,
        q_idx=q_idx, q_scale=q_scale, w=w, k_idx=k_idx, k_scale=k_scale,
        topk=topk, attn_dtype="bf16", H=128, d_qk=576, d_v=512,
        q=_bf16_normal((batch, 128, 576), seed, "q", device),
        kv=_bf16_normal((rows, 576), seed, "kv", device),
        softmax_scale=1.0 / math.sqrt(576),
        q_seq=q_seq, q_pos=q_pos, seq_lens=[ctx] * batch, seq_stride=ctx,
        block_table=None, block_size=0, chunks=[(0, batch)])


def mixed_lengths(seed: int, batch: int, lo: int, hi: int) -> List[int]:
    g = torch.Generator().manual_seed((int(seed) * 1_000_003 + zlib.crc32(b"ctx")) & 0x7FFF_FFFF_FFFF)
    return [int(v) for v in torch.randint(lo, hi + 1, (batch,), generator=g)]


def make_mixed(seed=0, device="cpu", batch=8, lo=8192, hi=131072, prefill=8192, decode=32,
               block=64, topk=2048, lengths: Optional[List[int]] = None) -> Workload:
    """Paged mixed batch: per sequence a prefill run of ``prefill`` queries at
    positions [C-prefill-decode, C-decode) and ``decode`` single-token queries
    at [C-decode, C).  Physical blocks of all sequences form one pool under one
    seeded permutation."""
    lens = lengths if lengths is not None else mixed_lengths(seed, batch, lo, hi)
    tail = prefill + decode
    assert all(c >= tail for c in lens)
    runs = []
    for b, c in enumerate(lens):
        if prefill:
            runs.append((b, c - tail, prefill))
        for p in range(c - decode, c):
            runs.append((b, p, 1))
    q_seq, q_pos = _runs_layout(runs, device)
    nblk = [(c + block - 1) // block for c in lens]
    total_blocks = sum(nblk)
    maxb = max(nblk)
    g = torch.Generator().manual_seed((int(seed) * 1_000_003 + zlib.crc32(b"perm")) & 0x7FFF_FFFF_FFFF)
    perm = torch.randperm(total_blocks, generator=g).to(torch.int32)
    bt = torch.zeros((len(lens), maxb), dtype=torch.int32)
    off = 0
    for b, n in enumerate(nblk):
        bt[b, :n] = perm[off:off + n]
        off += n
    rows = total_blocks * block
    nq = q_pos.shape[0]
    q_idx, q_scale, w, k_idx, k_scale = _indexer_fp8(seed, nq, rows, device, "uniform")
    return Workload(
        name="mixed", seed=seed, idx_dtype="fp8", H_I=64, d_I=128,
        q_idx=q_idx, q_scale=q_scale, w=w, k_idx=k_idx, k_scale=k_scale,
        topk=topk, attn_dtype="bf16", H=128, d_qk=576, d_v=512,
        q=_bf16_normal((nq, 128, 576), seed, "q", device),
        kv=_bf16_normal((rows, 576), seed, "kv", device),
        softmax_scale=1.0 / math.sqrt(576),
        q_seq=q_seq, q_pos=q_pos, seq_lens=lens, seq_stride=0,
        block_table=bt.to(device), block_size=block,
        chunks=[(0, nq)])   # the whole mixed batch is one call


def make_config(i: int, seed: int = 0, device="cpu") -> Workload:
    return [make_tiny, make_prefill, make_long, make_decode, make_mixed][i](seed=seed, device=device)


def make_scores(num_q: int, n: int, seed: int, device="cpu", kind: str = "normal") -> torch.Tensor:
    """Seeded fp32 score rows for the stand-alone top-k stage.

    kind="normal": N(0,1); "ties": N(0,1) rounded to multiples of 1/4 with
    random signed zeros, so many exact ties and +-0 pairs occur;
    "const": every score 1.0 (all tied).
    """
    x = randn((num_q, n), seed, "scores", device)
    if kind == "ties":
        x = torch.round(x * 4) / 4
        sgn = rand((num_q, n), seed, "zsign", device) < 0.5
        x = torch.where((x == 0) & sgn, torch.full_like(x, -0.0), x)
    elif kind == "const":
        x = torch.ones_like(x)
    return x


def kl_targets(idx: torch.Tensor, seed: int) -> torch.Tensor:
    """Seeded synthetic target distributions for the indexer's alignment loss:
    one row per query over its idx entries, u^3 (u uniform) normalised over
    the valid entries (idx >= 0), 0 at padding; about 1 entry in 16 is set to
    exactly 0 so zero targets occur.  fp32, on idx's device."""
    u = rand(tuple(idx.shape), seed, "kl_target", idx.device) ** 3
    u = torch.where(rand(tuple(idx.shape), seed, "kl_zero", idx.device) < 1.0 / 16, torch.zeros_like(u), u)
    u = torch.where(idx >= 0, u, torch.zeros_like(u))
    tot = u.sum(dim=1, keepdim=True)
    return torch.where(tot > 0, u / torch.where(tot > 0, tot, torch.ones_like(tot)), u).contiguous()


def random_index_sets(q_pos: torch.Tensor, k: int, seed: int) -> torch.Tensor:
    """For each query position p, a seeded random subset of min(k, p+1)
    positions in [0, p], ascending, padded with -1 to width k (CPU int32)."""
    g = torch.Generator().manual_seed((int(seed) * 1_000_003 + zlib.crc32(b"idxsets")) & 0x7FFF_FFFF_FFFF)
    pos = q_pos.to("cpu")
    out = torch.full((pos.shape[0], k), -1, dtype=torch.int32)
    for i, p in enumerate(pos.tolist()):
        n = p + 1
        if n <= k:
            out[i, :n] = torch.arange(n, dtype=torch.int32)
        else:
            sel = torch.randperm(n, generator=g)[:k].sort().values
            out[i] = sel.to(torch.int32)
    return out


@dataclasses.dataclass
class MhaWorkload:
    """Inputs of the per-head (non-absorbed) attention mode for one
    single-sequence causal prefill: per-head key rows k_nope [L, H, 128], the
    shared rope part k_rope [L, 64] and per-head values v [L, H, 128], bf16
    ~ N(0,1); queries q [nq, H, 192] at positions q_pos; softmax scale
    1/sqrt(192).  Cache rows are contiguous (row = position)."""
    q: torch.Tensor
    k_nope: torch.Tensor
    k_rope: torch.Tensor
    v: torch.Tensor
    q_seq: torch.Tensor
    q_pos: torch.Tensor
    L: int
    softmax_scale: float

    @property
    def num_q(self) -> int:
        return int(self.q_pos.shape[0])

    @property
    def heads(self) -> int:
        return int(self.q.shape[1])


def make_mha_prefill(seed=0, device="cpu", L=4096, heads=128, q_rows: Optional[Tuple[int, int]] = None) -> MhaWorkload:
    a, b = q_rows if q_rows is not None else (0, L)
    q_seq, q_pos = _runs_layout([(0, a, b - a)], device)
    return MhaWorkload(
        q=_bf16_normal((b - a, heads, 192), seed, "mha_q", device),
        k_nope=_bf16_normal((L, heads, 128), seed, "mha_k_nope", device),
        k_rope=_bf16_normal((L, 64), seed, "mha_k_rope", device),
        v=_bf16_normal((L, heads, 128), seed, "mha_v", device),
        q_seq=q_seq, q_pos=q_pos, L=L, softmax_scale=1.0 / math.sqrt(192))
