"""The per-head (non-absorbed) attention mode, dsa_sparse_attn_mha, against
the oracle's sparse_attention_mha on identical bf16 inputs: sampled rows of
a prefill (rows below and above k, padding, a ragged last batch of entries),
a paged copy of the same cache giving the same bits, and an out-of-range
entry that is flagged and skipped."""
import numpy as np
import pytest
import torch

from oracle import dsa_oracle as O
from sparse_attention_long_11_b300 import api, inputs
from dsa_testutil import ATTN_ATOL_BF16

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _f64(t):
    return O.decode_bf16(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _run(wl, sel, k, cache):
    out = torch.empty((wl.num_q, wl.heads, 128), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((wl.num_q, wl.heads), dtype=torch.float32, device=DEV)
    at = api.mha_inputs(wl.q, wl.k_nope, wl.k_rope, wl.v, wl.softmax_scale)
    batch = api.Batch(wl.q_seq, wl.q_pos, wl.L)
    api.dsa_sparse_attn_mha(batch.desc(), cache.desc(), at, sel.to(DEV), k, out, lse)
    return out, lse


@pytest.mark.parametrize("heads,k", [(128, 100), (16, 300)])
def test_mha_mode_matches_oracle(heads, k):
    wl = inputs.make_mha_prefill(seed=71 + heads, device=DEV, L=700, heads=heads)
    sel = inputs.random_index_sets(wl.q_pos, k, seed=3)
    out, lse = _run(wl, sel, k, api.Cache(1, wl.L, wl.L))
    assert api.dsa_check_device_error() == api.DSA_OK
    q, kn, kr, v = _f64(wl.q), _f64(wl.k_nope), _f64(wl.k_rope), _f64(wl.v)
    o_h, l_h = out.float().cpu().numpy(), lse.cpu().numpy()
    for i in sorted({0, 1, k - 2, k - 1, k, 350, wl.num_q - 1}):
        s = sel[i].numpy()
        s = s[s >= 0]
        ro, rl = O.sparse_attention_mha(q[i], kn[s], kr[s], v[s], wl.softmax_scale)
        assert np.abs(o_h[i] - ro).max() <= ATTN_ATOL_BF16, i
        assert np.abs(l_h[i] - rl).max() <= 1e-3 * max(1.0, np.abs(rl).max()), i


def test_mha_mode_paged_equals_contiguous_and_flags_bad_entries():
    wl = inputs.make_mha_prefill(seed=75, device=DEV, L=512, heads=32)
    k = 128
    sel = inputs.random_index_sets(wl.q_pos, k, seed=4)
    ref = _run(wl, sel, k, api.Cache(1, wl.L, wl.L))
    assert api.dsa_check_device_error() == api.DSA_OK
    # the same rows in a pool of 64-row blocks under a permutation
    perm = torch.randperm(8, generator=torch.Generator().manual_seed(5))
    phys = (perm[:, None] * 64 + torch.arange(64)[None, :]).reshape(-1)   # logical row r -> physical row phys[r]
    pool = [torch.empty_like(t) for t in (wl.k_nope, wl.k_rope, wl.v)]
    for dst, src in zip(pool, (wl.k_nope, wl.k_rope, wl.v)):
        dst[phys.to(DEV)] = src
    import dataclasses
    wp = dataclasses.replace(wl, k_nope=pool[0], k_rope=pool[1], v=pool[2])
    bt = perm.to(torch.int32)[None, :].to(DEV)
    got = _run(wp, sel, k, api.Cache(1, wl.L, 0, bt, 64))
    assert api.dsa_check_device_error() == api.DSA_OK
    assert torch.equal(ref[0], got[0]) and torch.equal(ref[1], got[1])
    # an entry after the query's position is flagged and contributes nothing
    bad = sel.clone()
    bad[5, 6] = 400                                    # query 5 selects positions 0..5, then padding
    out, lse = _run(wl, bad, k, api.Cache(1, wl.L, wl.L))
    assert api.dsa_check_device_error() == api.DSA_ERR_BOUNDS
    assert torch.equal(out[5], ref[0][5]) and torch.equal(lse[5], ref[1][5])
