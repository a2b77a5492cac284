"""Feeds a generated DSA workload to the oracle, one query at a time.

TEST INFRASTRUCTURE ONLY (see ``dsa_oracle``).  The workload object is duck
typed (any object with the attributes of a generated workload); tensors may
live on the CPU or on a GPU, and only the rows the oracle needs are copied to
the host.  The cache is read in *logical* order through the workload's own
row map (contiguous or paged), which is input layout, not arithmetic.
"""
from __future__ import annotations

import numpy as np
import torch

from . import dsa_oracle as O


def _np_bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def _decode_idx(t: torch.Tensor, dtype: str) -> np.ndarray:
    t = t.detach().to("cpu").contiguous()
    if dtype == "fp8":
        return O.decode_e4m3(t.view(torch.uint8).numpy())
    return t.numpy().astype(np.float64)


def _decode_attn(t: torch.Tensor, dtype: str) -> np.ndarray:
    if dtype in ("bf16", "fp8kv"):          # queries are bf16 in both
        return O.decode_bf16(_np_bits16(t))
    return t.detach().to("cpu").numpy().astype(np.float64)


def _decode_kv(wl, rows: torch.Tensor) -> np.ndarray:
    if wl.attn_dtype == "fp8kv":
        codes = wl.kv[rows].detach().to("cpu").contiguous().view(torch.uint8).numpy()
        scale = wl.kv_scale[rows].detach().to("cpu").numpy().astype(np.float32)
        return O.dequantize_kv_e4m3(codes, scale)
    return _decode_attn(wl.kv[rows], wl.attn_dtype)


class OracleView:
    def __init__(self, wl):
        self.wl = wl
        self.q_seq = wl.q_seq.to("cpu").numpy()
        self.q_pos = wl.q_pos.to("cpu").numpy()
        self._seq_cache = {}

    def _rows(self, seq: int, n: int) -> torch.Tensor:
        return self.wl.logical_rows(seq, n).to(self.wl.kv.device)

    def seq_cache(self, seq: int, n: int):
        """Decoded logical cache of ``seq`` positions 0..n-1 (memoised for the
        longest n requested so far)."""
        c = self._seq_cache.get(seq)
        if c is not None and c[0] >= n:
            return c[1]
        rows = self._rows(seq, n)
        wl = self.wl
        k_vals = _decode_idx(wl.k_idx[rows], wl.idx_dtype)
        k_scale = None if wl.k_scale is None else wl.k_scale[rows].to("cpu").numpy().astype(np.float64)
        kv = _decode_kv(wl, rows)
        self._seq_cache = {seq: (n, (k_vals, k_scale, kv))}  # keep one sequence resident
        return k_vals, k_scale, kv

    def query_inputs(self, i: int):
        wl = self.wl
        qi = _decode_idx(wl.q_idx[i], wl.idx_dtype)
        qs = None if wl.q_scale is None else wl.q_scale[i].to("cpu").numpy().astype(np.float64)
        w = wl.w[i].to("cpu").numpy().astype(np.float64)
        qa = _decode_attn(wl.q[i], wl.attn_dtype)
        return qi, qs, w, qa

    def scores(self, i: int) -> np.ndarray:
        seq, pos = int(self.q_seq[i]), int(self.q_pos[i])
        k_vals, k_scale, _ = self.seq_cache(seq, pos + 1)
        qi, qs, w, _ = self.query_inputs(i)
        return O.index_scores(qi, w, k_vals, pos, qs, k_scale)

    def attention(self, i: int, idx) -> tuple:
        """Oracle attention of query i over the logical positions ``idx``
        (-1 entries skipped)."""
        seq, pos = int(self.q_seq[i]), int(self.q_pos[i])
        _, _, kv = self.seq_cache(seq, pos + 1)
        _, _, _, qa = self.query_inputs(i)
        sel = np.asarray(idx)
        sel = sel[sel >= 0]
        return O.sparse_attention(qa, kv[sel], self.wl.softmax_scale, self.wl.d_v)

    def run(self, i: int):
        """Whole path for query i: (scores, idx, O, LSE)."""
        seq, pos = int(self.q_seq[i]), int(self.q_pos[i])
        k_vals, k_scale, kv = self.seq_cache(seq, pos + 1)
        qi, qs, w, qa = self.query_inputs(i)
        return O.dsa_query(qi, qs, w, k_vals, k_scale, pos, self.wl.topk, qa, kv,
                           self.wl.softmax_scale, self.wl.d_v)
