"""The fused forward's streamed selection (sampled threshold, filtered
candidates, exact select, fallback) against the stand-alone stages: the
selection must equal dsa_topk on dsa_index_scores' rows bit for bit, for
random rows, for rows built so that the sampled threshold misses (every key
tile 0, m, 2m, ... the indexer samples holds the row's largest scores, so too
few keys pass it; or the other tiles hold them, so the candidate list
overflows), and for all-tied rows (w = 0: every score is 0 and the lowest
positions win).  The sample stride m of the FP8 path is the smallest that
keeps a row at 32 sampled key tiles of 128 keys."""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import dsa_oracle as O
from sparse_attention_long_11_b300 import api, inputs
from dsa_testutil import run_forward

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _sample_stride(max_kv):
    tiles = (max_kv + 127) // 128
    return max(1, -(-tiles // 32))


def _staged(prob):
    wl = prob.wl
    ld = (wl.max_kv + 3) // 4 * 4
    sc = torch.empty((wl.num_q, ld), dtype=torch.float32, device=DEV)
    api.dsa_index_scores(prob.batch.desc(), prob.cache.desc(), prob.ix, sc)
    idx = torch.empty((wl.num_q, wl.topk), dtype=torch.int32, device=DEV)
    api.dsa_topk(prob.batch.desc(), sc, wl.topk, idx)
    assert api.dsa_check_device_error() == api.DSA_OK
    return sc, idx


def _scale_key_tiles(wl, sampled, factor):
    """Multiplies the key scales of the sampled tiles (or of all the others)
    by `factor`: those keys' scores scale by it exactly in exponent terms."""
    m = _sample_stride(wl.max_kv)
    tile = torch.arange(wl.num_rows, device=DEV) // 128           # contiguous single-sequence cache
    hit = (tile % m == 0) if sampled else (tile % m != 0)
    ks = torch.where(hit, wl.k_scale * factor, wl.k_scale)
    return dataclasses.replace(wl, k_scale=ks.contiguous())


@pytest.mark.parametrize("case", ["random", "sampled_tiles_win", "other_tiles_win", "all_tied"])
def test_fused_selection_equals_topk_of_the_score_rows(case):
    wl = inputs.make_prefill(seed=61, device=DEV, L=9000)          # m = 3 at this length
    if case == "sampled_tiles_win":
        wl = _scale_key_tiles(wl, sampled=True, factor=64.0)
    elif case == "other_tiles_win":
        wl = _scale_key_tiles(wl, sampled=False, factor=64.0)
    elif case == "all_tied":
        wl = dataclasses.replace(wl, w=torch.zeros_like(wl.w))
    prob = api.Problem(wl)
    idx, out, lse = run_forward(prob)
    assert api.dsa_check_device_error() == api.DSA_OK
    sc, want = _staged(prob)
    assert torch.equal(idx, want)
    if case == "all_tied":
        k = wl.topk
        first = torch.arange(k, dtype=torch.int32, device=DEV)
        assert torch.equal(idx[k:], first.expand(wl.num_q - k, k))
    # spot check against the oracle's exact selection on the GPU's own scores
    s_np, i_np = sc.cpu().numpy(), idx.cpu().numpy()
    for i in (2048, 5000, 8999):
        assert np.array_equal(i_np[i], O.topk_select(s_np[i, :i + 1], wl.topk)), i
    # attention on the selection equals the stand-alone attention bit for bit
    out2 = torch.empty_like(out)
    lse2 = torch.empty_like(lse)
    api.dsa_sparse_attn(prob.batch.desc(), prob.cache.desc(), prob.at, want, wl.topk, out2, lse2)
    assert api.dsa_check_device_error() == api.DSA_OK
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


@pytest.mark.parametrize("L,k", [(3000, 100), (5000, 8192), (40000, 2048), (20000, 1), (131072, 2048),
                                 (131072, 8192)])
def test_fused_selection_other_shapes(L, k):
    """Small and large k, every tile sampled (m = 1, L <= 4096), rows shorter
    than k, long rows (m = 10; m = 32 at L = 131072, whose 2^17 positions fill
    the select kernel's position window exactly), decode-style single rows
    included."""
    q_rows = (L - 600, L) if 20000 < L < 100000 else ((L - 256, L) if L >= 100000 else None)
    wl = inputs.make_prefill(seed=62 + k, device=DEV, L=L, topk=k, q_rows=q_rows)
    prob = api.Problem(wl)
    idx, _, _ = run_forward(prob)
    assert api.dsa_check_device_error() == api.DSA_OK
    _, want = _staged(prob)
    assert torch.equal(idx, want)
    one = run_forward(prob, chunks=[(wl.num_q - 1, wl.num_q)])[0]   # the last row as a one-query call
    assert torch.equal(one[-1], want[-1])


def test_fused_selection_paged_decode_batch():
    """Decode-style rows of several paged sequences (per-query indexer passes
    spread over many CTAs, all appending to one candidate list per query)."""
    wm = inputs.make_mixed(seed=63, device=DEV, batch=4, lo=9000, hi=20000, prefill=0, decode=16, block=64)
    prob = api.Problem(wm)
    idx, _, _ = run_forward(prob)
    assert api.dsa_check_device_error() == api.DSA_OK
    _, want = _staged(prob)
    assert torch.equal(idx, want)


def test_fused_selection_full_size_decode():
    """The decode workload at full size (64 sequences x 65536 cached rows, one
    query each, k = 2048, sample stride 16): the streamed selection equals the
    stand-alone stages' selection on every row."""
    wd = inputs.make_decode(seed=64, device=DEV)
    prob = api.Problem(wd)
    idx, _, _ = run_forward(prob)
    assert api.dsa_check_device_error() == api.DSA_OK
    _, want = _staged(prob)
    assert torch.equal(idx, want)
