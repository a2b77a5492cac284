"""Shared helpers of the GPU parity tests: running the library's stages on a
generated workload, and the comparison rules against the oracle."""
from __future__ import annotations

import numpy as np
import torch

from oracle import dsa_oracle as O
from sparse_attention_long_11_b300 import api

# Attention output tolerance (bf16 inputs, fp32 accumulation, bf16 output).
ATTN_ATOL_BF16 = 2e-2
# fp32 operands: only fp32 rounding of the dot products and the softmax.
ATTN_ATOL_F32 = 2e-5
# Indexer: relative 1e-3 of max(|I|, A/16), A = sum_j |w_j| sq_j sk_s sum_d |q_jd k_sd|.
IDX_RTOL = 1e-3


def indexer_tolerance(view, i: int) -> np.ndarray:
    """Per-key tolerance of query i's indexer scores: an fp32-accumulating
    kernel's rounding error is below 2^-16 * A, so 1e-3 * max(|I|, A/16)
    never fails a correct kernel yet stays tight on typical entries."""
    seq, pos = int(view.q_seq[i]), int(view.q_pos[i])
    k_vals, k_scale, _ = view.seq_cache(seq, pos + 1)
    qi, qs, w, _ = view.query_inputs(i)
    a = np.abs(k_vals[:pos + 1]) @ np.abs(qi).T            # [n, H_I]
    if qs is not None:
        a = a * qs[None, :]
    if k_scale is not None:
        a = a * k_scale[:pos + 1, None]
    A = a @ np.abs(w)
    ref = O.index_scores(qi, w, k_vals, pos, qs, k_scale)
    return IDX_RTOL * np.maximum(np.abs(ref), A / 16.0), ref


def run_forward(prob: api.Problem, chunks=None):
    """dsa_forward over the workload's chunks (one call per chunk) -> (idx, O, LSE)."""
    wl = prob.wl
    nq = wl.num_q
    dev = wl.q.device
    idx = torch.empty((nq, wl.topk), dtype=torch.int32, device=dev)
    out = torch.empty((nq, wl.H, wl.d_v), dtype=prob.out_dtype(), device=dev)
    lse = torch.empty((nq, wl.H), dtype=torch.float32, device=dev)
    chunks = chunks or wl.chunks
    wsb = max(api.dsa_forward_workspace_size(*_ws_args(prob, a, b)) for a, b in chunks)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    cache = prob.cache.desc()
    for a, b in chunks:
        qd, ix, at = prob.rows(a, b)
        api.dsa_forward(qd, cache, ix, wl.topk, at, idx[a:b], out[a:b], lse[a:b], ws)
    return idx, out, lse


def _ws_args(prob, a, b):
    qd, ix, at = prob.rows(a, b)
    return qd, ix, prob.wl.topk, at


def check_selection(view, i: int, got_idx: np.ndarray, k: int):
    """End-to-end selection check for query i against oracle float64 scores.

    The GPU ranks fp32 scores, the oracle float64 ones, so two candidates
    whose scores differ by less than the indexer tolerance may swap places
    at the k-th boundary.  Returns (oracle idx, number of swapped entries);
    asserts that every swap is such a near tie and that the GPU's list is a
    valid selection (ascending, distinct, causal, -1 padded)."""
    tol, ref = indexer_tolerance(view, i)
    want = O.topk_select(ref, k)
    pos = int(view.q_pos[i])
    n = min(k, pos + 1)
    g = got_idx[:n]
    assert np.all(got_idx[n:] == -1), "padding"
    assert np.all(np.diff(g) > 0) and g[0] >= 0 and g[-1] <= pos, "not ascending/causal"
    gs, ws_ = set(g.tolist()), set(want[:n].tolist())
    extra, missing = sorted(gs - ws_), sorted(ws_ - gs)
    if extra:
        kth = np.sort(ref[want[:n]])[0]                     # oracle's k-th largest score
        for s in extra:
            assert ref[s] >= kth - 2 * tol[s], f"q{i}: GPU kept {s} ({ref[s]}) far below the cut {kth}"
        for s in missing:
            assert ref[s] <= kth + 2 * tol[s], f"q{i}: GPU dropped {s} ({ref[s]}) far above the cut {kth}"
    return want, len(extra)
