"""End-to-end parity of dsa_forward (indexer -> top-k -> sparse attention)
with the CPU oracle, plus GPU-vs-GPU invariants (paged == contiguous,
chunked == whole, decode row == prefill row, fused == staged).  The
full-size cases run each workload exactly as the benchmark launches it and
check a sample of queries the oracle can afford."""
import numpy as np
import pytest
import torch

from oracle.workload_view import OracleView
from sparse_attention_long_11_b300 import api, inputs
from dsa_testutil import ATTN_ATOL_BF16, ATTN_ATOL_F32, check_selection, run_forward

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _check_rows(wl, idx, out, lse, rows, atol):
    view = OracleView(wl)
    idx = idx.cpu().numpy()
    swaps = 0
    for i in rows:
        want, nswap = check_selection(view, i, idx[i], wl.topk)
        swaps += nswap
        if nswap == 0:
            # same selected set: attention must match the oracle on it
            ro, rl = view.attention(i, want)
            o = out[i].float().cpu().numpy()
            err = np.abs(o - ro).max()
            assert err <= atol, f"query {i}: max |O - O_ref| = {err}"
            l = lse[i].cpu().numpy()
            assert np.abs(l - rl).max() <= 1e-3 * max(1.0, np.abs(rl).max()), f"query {i}: LSE"
    assert swaps <= max(2, len(rows) // 4), f"{swaps} near-tie swaps in {len(rows)} queries"
    return swaps


def _sample(nq, m, extra=()):
    return sorted(set(np.linspace(0, nq - 1, m).astype(int).tolist()) | set(extra))


def test_forward_tiny_all_queries():
    wl = inputs.make_tiny(seed=0, device=DEV)
    idx, out, lse = run_forward(api.Problem(wl))
    assert api.dsa_check_device_error() == api.DSA_OK
    _check_rows(wl, idx, out, lse, range(wl.num_q), ATTN_ATOL_F32)


def test_forward_fp8_bf16_small():
    wl = inputs.make_prefill(seed=1, device=DEV, L=2600)      # spans k=2048 and a ragged tail
    idx, out, lse = run_forward(api.Problem(wl))
    assert api.dsa_check_device_error() == api.DSA_OK
    _check_rows(wl, idx, out, lse, _sample(wl.num_q, 40, [2046, 2047, 2048, 2049]), ATTN_ATOL_BF16)


@pytest.mark.parametrize("k", [1024, 4096, 8192])
def test_forward_other_k(k):
    """The top-k sweep beyond the 2048 of the pages: rows below and above k."""
    wl = inputs.make_prefill(seed=3, device=DEV, L=9000, topk=k)
    idx, out, lse = run_forward(api.Problem(wl))
    assert api.dsa_check_device_error() == api.DSA_OK
    _check_rows(wl, idx, out, lse, _sample(wl.num_q, 12, [k - 2, k - 1, k, wl.num_q - 1]), ATTN_ATOL_BF16)


@pytest.mark.parametrize("kind", ["decode", "prefill"])
def test_forward_fp8_kv_cache(kind):
    """The FP8 latent cache through the fused forward: the decode batch at full
    size (64 x 65536) and a 4096-token prefill, sampled rows vs the oracle."""
    torch.cuda.empty_cache()
    if kind == "decode":
        wl = inputs.with_fp8_kv(inputs.make_decode(seed=2, device=DEV))
        rows = _sample(wl.num_q, 8, [wl.num_q - 1])
    else:
        wl = inputs.with_fp8_kv(inputs.make_prefill(seed=2, device=DEV, L=4096))
        rows = _sample(wl.num_q, 10, [2047, 2048, 4095])
    idx, out, lse = run_forward(api.Problem(wl))
    assert api.dsa_check_device_error() == api.DSA_OK
    _check_rows(wl, idx, out, lse, rows, ATTN_ATOL_BF16)
    del wl, idx, out, lse
    torch.cuda.empty_cache()


@pytest.mark.parametrize("kind", ["contiguous", "paged"])
def test_forward_fp8_kv_copy_equals_gather(kind):
    """An FP8 latent cache in a prefill: with room in the workspace the
    forward converts the cache to bf16 once and runs the bf16 attention on
    the copy; with a workspace too small for the copy it gathers the FP8 rows
    directly.  Both give the same indices, outputs and LSE, bit for bit, for
    a contiguous cache and for a paged pool (the copy keeps the physical row
    numbering, so the block table applies to it unchanged)."""
    torch.cuda.empty_cache()
    if kind == "contiguous":
        base = inputs.make_prefill(seed=3, device=DEV, L=3000)
    else:
        base = inputs.make_mixed(seed=4, device=DEV, batch=2, lengths=[3000, 2500], prefill=1024, decode=4)
    wl = inputs.with_fp8_kv(base)
    prob = api.Problem(wl)
    qd, ix, at = prob.rows(0, wl.num_q)
    cache = prob.cache.desc()
    copy_bytes = wl.kv.shape[0] * 576 * 2
    assert wl.num_q * wl.topk >= 4 * wl.kv.shape[0]                   # enough reuse for the copy
    big = api.dsa_forward_workspace_size(qd, ix, wl.topk, at)
    assert big >= copy_bytes
    # the largest stage whose workspace cannot hold the copy
    lo, hi = 1, wl.num_q
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if api.dsa_forward_stage_workspace_size(qd, ix, wl.topk, at, mid) < copy_bytes:
            lo = mid
        else:
            hi = mid - 1
    small = api.dsa_forward_stage_workspace_size(qd, ix, wl.topk, at, lo)
    assert 0 < small < copy_bytes
    res = []
    for wsb in (big, small):
        idx = torch.empty((wl.num_q, wl.topk), dtype=torch.int32, device=DEV)
        out = torch.empty((wl.num_q, wl.H, wl.d_v), dtype=torch.bfloat16, device=DEV)
        lse = torch.empty((wl.num_q, wl.H), dtype=torch.float32, device=DEV)
        ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
        api.dsa_forward(qd, cache, ix, wl.topk, at, idx, out, lse, ws)
        assert api.dsa_check_device_error() == api.DSA_OK
        res.append((idx, out, lse))
    (i1, o1, l1), (i2, o2, l2) = res
    assert torch.equal(i1, i2) and torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)
    del wl, prob, res
    torch.cuda.empty_cache()


def test_forward_128k_context():
    """A 131072-token prefill context (the long-context end of the sweep):
    the last 4096 queries, one bench-sized call, sampled rows vs the oracle."""
    torch.cuda.empty_cache()
    L = 131072
    wl = inputs.make_prefill(seed=6, device=DEV, L=L, q_rows=(L - 4096, L))
    idx, out, lse = run_forward(api.Problem(wl))
    assert api.dsa_check_device_error() == api.DSA_OK
    _check_rows(wl, idx, out, lse, [0, 1500, 4095], ATTN_ATOL_BF16)
    assert bool((idx >= 0).all()) and bool(torch.isfinite(out.float()).all())
    del wl, idx, out, lse
    torch.cuda.empty_cache()


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_forward_full_size(cfg):
    """Full workload sizes, launched as the benchmark launches them."""
    torch.cuda.empty_cache()
    wl = inputs.make_config(cfg, seed=0, device=DEV)
    idx, out, lse = run_forward(api.Problem(wl))
    assert api.dsa_check_device_error() == api.DSA_OK
    nq = wl.num_q
    rows = _sample(nq, 10 if cfg in (1, 3) else 8, [nq - 1])
    _check_rows(wl, idx, out, lse, rows, ATTN_ATOL_BF16)
    # properties at every row: causal, ascending, padded exactly where t+1 < k
    pos = wl.q_pos.to(torch.int64)
    valid = idx >= 0
    assert torch.equal(valid.sum(1), torch.clamp(pos + 1, max=wl.topk))
    assert bool((idx.to(torch.int64) <= pos[:, None]).all())
    d = idx[:, 1:].to(torch.int64) - idx[:, :-1].to(torch.int64)
    assert bool(((d > 0) | ~valid[:, 1:]).all())
    assert bool(torch.isfinite(out.float()).all()) and bool(torch.isfinite(lse).all())
    del wl, idx, out, lse
    torch.cuda.empty_cache()


# --------------------------------------------------------------------------- invariants (bitwise)

def test_paged_equals_contiguous():
    wm = inputs.make_mixed(seed=5, device=DEV, batch=3, lo=2200, hi=3000, prefill=200, decode=4, block=64)
    # the same logical caches laid out contiguously, one sequence after another
    stride = max(wm.seq_lens)
    rows = torch.full((wm.num_seqs * stride,), 0, dtype=torch.int64)
    for b, c in enumerate(wm.seq_lens):
        rows[b * stride:b * stride + c] = wm.logical_rows(b, c)
    rows = rows.to(DEV)
    import dataclasses
    wc = dataclasses.replace(wm, k_idx=wm.k_idx[rows], k_scale=wm.k_scale[rows], kv=wm.kv[rows],
                             seq_stride=stride, block_table=None, block_size=0)
    a = run_forward(api.Problem(wm))
    b = run_forward(api.Problem(wc))
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_chunked_equals_whole_and_decode_equals_prefill_row():
    wl = inputs.make_prefill(seed=6, device=DEV, L=3000)
    whole = run_forward(api.Problem(wl), chunks=[(0, 3000)])
    chunked = run_forward(api.Problem(wl), chunks=[(0, 1000), (1000, 2100), (2100, 3000)])
    for x, y in zip(whole, chunked):
        assert torch.equal(x, y)
    # decode: rows 2999 and 2500 issued as single-token calls
    for r in (2999, 2500):
        one = run_forward(api.Problem(wl), chunks=[(r, r + 1)])
        for x, y in zip(whole, one):
            assert torch.equal(x[r], y[r])


def test_workspace_size_does_not_change_results():
    """Stages of 1, 100 (not a divisor of the batch) and all rows give the same bits."""
    wl = inputs.make_prefill(seed=8, device=DEV, L=2600)
    prob = api.Problem(wl)
    qd, ix, at = prob.rows(0, wl.num_q)
    res = []
    for rows in (None, 100, 1):
        nb = (api.dsa_forward_workspace_size(qd, ix, wl.topk, at) if rows is None
              else api.dsa_forward_stage_workspace_size(qd, ix, wl.topk, at, rows))
        ws = torch.empty(nb, dtype=torch.uint8, device=DEV)
        idx = torch.empty((wl.num_q, wl.topk), dtype=torch.int32, device=DEV)
        out = torch.empty((wl.num_q, wl.H, wl.d_v), dtype=prob.out_dtype(), device=DEV)
        lse = torch.empty((wl.num_q, wl.H), dtype=torch.float32, device=DEV)
        api.dsa_forward(qd, prob.cache.desc(), ix, wl.topk, at, idx, out, lse, ws)
        assert api.dsa_check_device_error() == api.DSA_OK
        res.append((idx, out, lse))
    for other in res[1:]:
        for x, y in zip(res[0], other):
            assert torch.equal(x, y)


def test_fused_selection_equals_staged_stages():
    wl = inputs.make_prefill(seed=7, device=DEV, L=2500)
    prob = api.Problem(wl)
    idx, out, lse = run_forward(prob)
    sc = torch.empty((wl.num_q, 2500), dtype=torch.float32, device=DEV)
    api.dsa_index_scores(prob.batch.desc(), prob.cache.desc(), prob.ix, sc)
    idx2 = torch.empty_like(idx)
    api.dsa_topk(prob.batch.desc(), sc, wl.topk, idx2)
    assert torch.equal(idx, idx2)
    out2 = torch.empty_like(out)
    lse2 = torch.empty_like(lse)
    api.dsa_sparse_attn(prob.batch.desc(), prob.cache.desc(), prob.at, idx2, wl.topk, out2, lse2)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
