"""Stage-by-stage parity of the CUDA path (through the C ABI) with the CPU
oracle, on identical seeded inputs.  Needs a B300 and the built library."""
import math

import dataclasses

import numpy as np
import pytest
import torch

from oracle import dsa_oracle as O
from oracle.workload_view import OracleView
from sparse_attention_long_11_b300 import api, inputs
from dsa_testutil import ATTN_ATOL_BF16, ATTN_ATOL_F32, indexer_tolerance

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _scores(prob):
    wl = prob.wl
    ld = (wl.max_kv + 3) // 4 * 4
    sc = torch.empty((wl.num_q, ld), dtype=torch.float32, device=DEV)
    api.dsa_index_scores(prob.batch.desc(), prob.cache.desc(), prob.ix, sc)
    assert api.dsa_check_device_error() == api.DSA_OK
    return sc


# --------------------------------------------------------------------------- indexer

@pytest.mark.parametrize("make", [
    lambda: inputs.make_tiny(seed=0, device=DEV),                                   # fp32, 4 x 64
    lambda: inputs.make_prefill(seed=1, device=DEV, L=777, topk=2048),               # fp8, ragged tail
])
def test_index_scores_match_oracle(make):
    wl = make()
    prob = api.Problem(wl)
    sc = _scores(prob).cpu().numpy()
    view = OracleView(wl)
    rows = range(wl.num_q) if wl.num_q <= 256 else sorted(set(np.linspace(0, wl.num_q - 1, 40).astype(int)))
    for i in rows:
        tol, ref = indexer_tolerance(view, i)
        pos = int(view.q_pos[i])
        got = sc[i, :pos + 1].astype(np.float64)
        bad = np.abs(got - ref) > tol
        assert not bad.any(), f"query {i}: {np.flatnonzero(bad)[:5]} got {got[bad][:3]} want {ref[bad][:3]}"
        assert np.all(np.isneginf(sc[i, pos + 1:wl.max_kv]))


def test_index_scores_decode_batch_and_paged():
    # many sequences, one query each (contiguous), and the same under a paged layout
    wl = inputs.make_decode(seed=2, device=DEV, batch=5, ctx=1000)
    view = OracleView(wl)
    sc = _scores(api.Problem(wl)).cpu().numpy()
    for i in range(5):
        tol, ref = indexer_tolerance(view, i)
        assert np.all(np.abs(sc[i, :1000] - ref) <= tol)
    wm = inputs.make_mixed(seed=3, device=DEV, batch=3, lo=300, hi=700, prefill=100, decode=5, block=64)
    view = OracleView(wm)
    sc = _scores(api.Problem(wm)).cpu().numpy()
    for i in list(range(0, wm.num_q, 17)) + [wm.num_q - 1]:
        tol, ref = indexer_tolerance(view, i)
        pos = int(view.q_pos[i])
        assert np.all(np.abs(sc[i, :pos + 1] - ref) <= tol), i


# --------------------------------------------------------------------------- top-k

@pytest.mark.parametrize("kind", ["normal", "ties", "const"])
@pytest.mark.parametrize("n,k", [(300, 32), (5000, 2048), (5000, 2047), (3000, 1), (70000, 2048)])
def test_topk_exact(kind, n, k):
    nq = 24 if n < 60000 else 4
    sc = inputs.make_scores(nq, n, seed=n + k, device=DEV, kind=kind)
    # positions: some rows with fewer than k candidates, the last row full
    pos = torch.linspace(0, n - 1, nq).round().to(torch.int32)
    pos[0] = min(k - 1, n - 1)
    batch = api.Batch(torch.zeros(nq, dtype=torch.int32, device=DEV), pos.to(DEV), n)
    idx = torch.empty((nq, k), dtype=torch.int32, device=DEV)
    api.dsa_topk(batch.desc(), sc, k, idx)
    assert api.dsa_check_device_error() == api.DSA_OK
    got = idx.cpu().numpy()
    s_np = sc.cpu().numpy()
    for i in range(nq):
        p = int(pos[i])
        want = O.topk_select(s_np[i, :p + 1], k)
        assert np.array_equal(got[i], want), f"row {i} pos {p}"


@pytest.mark.parametrize("kind", ["normal", "ties", "const"])
def test_topk_exact_many_rows(kind):
    """Enough rows that the kernel runs several narrow blocks per SM."""
    nq, n, k = 400, 6000, 2048
    sc = inputs.make_scores(nq, n, seed=77, device=DEV, kind=kind)
    pos = torch.linspace(0, n - 1, nq).round().to(torch.int32)
    batch = api.Batch(torch.zeros(nq, dtype=torch.int32, device=DEV), pos.to(DEV), n)
    idx = torch.empty((nq, k), dtype=torch.int32, device=DEV)
    api.dsa_topk(batch.desc(), sc, k, idx)
    assert api.dsa_check_device_error() == api.DSA_OK
    got, s_np = idx.cpu().numpy(), sc.cpu().numpy()
    for i in range(0, nq, 7):
        p = int(pos[i])
        assert np.array_equal(got[i], O.topk_select(s_np[i, :p + 1], k)), f"row {i} pos {p}"


@pytest.mark.parametrize("nq", [4, 400])
def test_topk_exact_when_evenly_spaced_positions_hold_the_largest_scores(nq):
    """Rows whose largest scores sit exactly at evenly spaced positions (every
    n/1024-th): a threshold estimated from such positions overshoots, and
    the selection must still be exact."""
    n, k = 70000, 2048
    sc = inputs.make_scores(nq, n, seed=5, device=DEV)
    s_pos = (torch.arange(1024, dtype=torch.int64) * n) // 1024
    sc[:, s_pos.to(DEV)] += 100.0
    pos = torch.full((nq,), n - 1, dtype=torch.int32)
    batch = api.Batch(torch.zeros(nq, dtype=torch.int32, device=DEV), pos.to(DEV), n)
    idx = torch.empty((nq, k), dtype=torch.int32, device=DEV)
    api.dsa_topk(batch.desc(), sc, k, idx)
    assert api.dsa_check_device_error() == api.DSA_OK
    got, s_np = idx.cpu().numpy(), sc.cpu().numpy()
    for i in range(0, nq, max(1, nq // 8)):
        assert np.array_equal(got[i], O.topk_select(s_np[i], k)), f"row {i}"


@pytest.mark.parametrize("k", [4096, 8192])
@pytest.mark.parametrize("nq", [6, 400])
def test_topk_exact_large_k(k, nq):
    """k beyond 2048, for the wide-block (few rows) and narrow-block paths."""
    n = 20000
    sc = inputs.make_scores(nq, n, seed=k + nq, device=DEV, kind="ties")
    pos = torch.linspace(0, n - 1, nq).round().to(torch.int32)
    batch = api.Batch(torch.zeros(nq, dtype=torch.int32, device=DEV), pos.to(DEV), n)
    idx = torch.empty((nq, k), dtype=torch.int32, device=DEV)
    api.dsa_topk(batch.desc(), sc, k, idx)
    assert api.dsa_check_device_error() == api.DSA_OK
    got, s_np = idx.cpu().numpy(), sc.cpu().numpy()
    for i in range(0, nq, max(1, nq // 12)):
        p = int(pos[i])
        assert np.array_equal(got[i], O.topk_select(s_np[i, :p + 1], k)), f"row {i} pos {p}"


@pytest.mark.parametrize("k", [2048, 4096])
def test_topk_exact_long_rows(k):
    """Rows up to 131072 keys (a 128K context): the candidate list is sized
    for the longest row, so the sampled path holds the expected candidates."""
    n, nq = 131072, 400
    sc = inputs.make_scores(nq, n, seed=k + 7, device=DEV)
    pos = torch.linspace(k, n - 1, nq).round().to(torch.int32)
    batch = api.Batch(torch.zeros(nq, dtype=torch.int32, device=DEV), pos.to(DEV), n)
    idx = torch.empty((nq, k), dtype=torch.int32, device=DEV)
    api.dsa_topk(batch.desc(), sc, k, idx)
    assert api.dsa_check_device_error() == api.DSA_OK
    got, s_np = idx.cpu().numpy(), sc.cpu().numpy()
    for i in list(range(0, nq, nq // 10)) + [nq - 1]:
        p = int(pos[i])
        assert np.array_equal(got[i], O.topk_select(s_np[i, :p + 1], k)), f"row {i} pos {p}"


def test_topk_ignores_scores_beyond_position():
    n, k = 4096, 64
    sc = inputs.make_scores(2, n, seed=9, device=DEV)
    sc[:, 2000:] = 1e30                      # huge scores after the causal bound must not be picked
    pos = torch.tensor([1999, 1500], dtype=torch.int32, device=DEV)
    batch = api.Batch(torch.zeros(2, dtype=torch.int32, device=DEV), pos, n)
    idx = torch.empty((2, k), dtype=torch.int32, device=DEV)
    api.dsa_topk(batch.desc(), sc, k, idx)
    s_np = sc.cpu().numpy()
    for i, p in enumerate([1999, 1500]):
        assert np.array_equal(idx[i].cpu().numpy(), O.topk_select(s_np[i, :p + 1], k))


# --------------------------------------------------------------------------- attention

def _attn(prob, idx_cpu, k):
    wl = prob.wl
    out = torch.empty((wl.num_q, wl.H, wl.d_v), dtype=prob.out_dtype(), device=DEV)
    lse = torch.empty((wl.num_q, wl.H), dtype=torch.float32, device=DEV)
    api.dsa_sparse_attn(prob.batch.desc(), prob.cache.desc(), prob.at, idx_cpu.to(DEV), k, out, lse)
    assert api.dsa_check_device_error() == api.DSA_OK
    return out.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("case", ["tiny", "bf16_k2048", "bf16_k100", "paged", "fp8kv_k2048", "fp8kv_paged"])
def test_sparse_attn_matches_oracle(case):
    if case == "tiny":
        wl, k, atol = inputs.make_tiny(seed=4, device=DEV), 32, ATTN_ATOL_F32
    elif case == "bf16_k2048":
        wl, k, atol = inputs.make_prefill(seed=5, device=DEV, L=2600), 2048, ATTN_ATOL_BF16
    elif case == "bf16_k100":
        wl, k, atol = inputs.make_prefill(seed=6, device=DEV, L=700, topk=100), 100, ATTN_ATOL_BF16
    elif case == "fp8kv_k2048":
        wl, k, atol = inputs.with_fp8_kv(inputs.make_prefill(seed=12, device=DEV, L=2600)), 2048, ATTN_ATOL_BF16
    else:
        wl = inputs.make_mixed(seed=7, device=DEV, batch=2, lo=2100, hi=2500, prefill=60, decode=3, block=64)
        k, atol = 2048, ATTN_ATOL_BF16
        if case == "fp8kv_paged":
            wl = inputs.with_fp8_kv(wl)
    prob = api.Problem(wl)
    sel = inputs.random_index_sets(wl.q_pos, k, seed=11)
    o, lse = _attn(prob, sel, k)
    view = OracleView(wl)
    rows = sorted(set(np.linspace(0, wl.num_q - 1, 24).astype(int)) | {0, wl.num_q - 1})
    for i in rows:
        ro, rl = view.attention(i, sel[i].numpy())
        err = np.abs(o[i] - ro).max()
        assert err <= atol, f"query {i}: max |O - O_ref| = {err}"
        assert np.abs(lse[i] - rl).max() <= 1e-3 * max(1.0, np.abs(rl).max()), i


def test_fp8_kv_attention_equals_bf16_attention_on_the_dequantised_cache():
    """The FP8 gather writes the same bf16 tiles as the bf16 path would for
    the cache bf16(scale * code): outputs and LSE agree bit for bit.  The
    dequantised cache here is torch's float8 decode, a float32 multiply and
    its bfloat16 cast."""
    w8 = inputs.with_fp8_kv(inputs.make_prefill(seed=13, device=DEV, L=2200))
    deq = (w8.kv.view(torch.float8_e4m3fn).float() * w8.kv_scale[:, None]).to(torch.bfloat16)
    wb = dataclasses.replace(w8, attn_dtype="bf16", kv=deq, kv_scale=None)
    sel = inputs.random_index_sets(w8.q_pos, 2048, seed=2)
    o8, l8 = _attn(api.Problem(w8), sel, 2048)
    ob, lb = _attn(api.Problem(wb), sel, 2048)
    assert np.array_equal(o8, ob) and np.array_equal(l8, lb)


def test_kv_dequant_equals_the_oracle():
    """dsa_kv_dequant writes bf16(scale * code) for every code (both zeros,
    subnormals, the largest finite values; NaN codes excluded) and scales
    from tiny to large, bit for bit as the oracle's dequantisation."""
    from oracle import dsa_oracle as ref
    g = torch.Generator().manual_seed(11)
    finite = torch.tensor([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=torch.uint8)
    n = 1000
    codes = finite[torch.randint(0, finite.numel(), (n, 576), generator=g)]
    codes[0] = finite[torch.arange(576) % finite.numel()]            # every finite code in one row
    scale = torch.exp(torch.empty(n).uniform_(-30.0, 30.0, generator=g)).float()
    scale[1], scale[2], scale[3] = 1.0, 2.0 ** -20, 2.0 ** 20
    out = torch.empty((n, 576), dtype=torch.bfloat16, device=DEV)
    api.dsa_kv_dequant(codes.to(DEV), scale.to(DEV), out)
    got = out.float().cpu().numpy().astype(np.float64)
    want = ref.dequantize_kv_e4m3(codes.numpy(), scale.numpy())
    assert np.array_equal(got, want)
    api.dsa_kv_dequant(codes[:0].to(DEV), scale[:0].to(DEV), out[:0])   # no rows: nothing to do


def test_sparse_attn_skips_padding_and_any_order():
    wl = inputs.make_tiny(seed=8, device=DEV, L=128, topk=48)
    prob = api.Problem(wl)
    sel = inputs.random_index_sets(wl.q_pos, 48, seed=3)
    o1, l1 = _attn(prob, sel, 48)
    g = torch.Generator().manual_seed(0)
    perm = torch.stack([r[torch.randperm(48, generator=g)] for r in sel])   # shuffled, -1s anywhere
    o2, l2 = _attn(prob, perm, 48)
    np.testing.assert_allclose(o1, o2, atol=1e-5)
    np.testing.assert_allclose(l1, l2, atol=1e-5)


# --------------------------------------------------------------------------- device-side checks

def test_out_of_range_inputs_are_flagged_not_faulted():
    wl = inputs.make_tiny(seed=9, device=DEV, L=64, topk=16)
    prob = api.Problem(wl)
    assert api.dsa_check_device_error() == api.DSA_OK
    bad_pos = wl.q_pos.clone()
    bad_pos[5] = 1000                                   # beyond max_kv
    batch = api.Batch(wl.q_seq, bad_pos, wl.max_kv)
    sc = torch.zeros((wl.num_q, 64), dtype=torch.float32, device=DEV)
    api.dsa_index_scores(batch.desc(), prob.cache.desc(), prob.ix, sc)
    assert api.dsa_check_device_error() == api.DSA_ERR_BOUNDS
    assert api.dsa_check_device_error() == api.DSA_OK          # the word was cleared
    assert torch.isneginf(sc[5]).all()
    sel = inputs.random_index_sets(wl.q_pos, 16, seed=1)
    sel[7, 0] = 50                                      # later than the query's position (7)
    out = torch.empty((wl.num_q, wl.H, wl.d_v), dtype=torch.float32, device=DEV)
    lse = torch.empty((wl.num_q, wl.H), dtype=torch.float32, device=DEV)
    api.dsa_sparse_attn(prob.batch.desc(), prob.cache.desc(), prob.at, sel.to(DEV), 16, out, lse)
    assert api.dsa_check_device_error() == api.DSA_ERR_BOUNDS
    assert torch.isfinite(out).all()


# --------------------------------------------------------------------------- peaked softmax

@pytest.mark.parametrize("scale,fp8kv", [(8, False), (32, False), (8, True)])
def test_sparse_attn_peaked_logits(scale, fp8kv):
    """Queries scaled up (x8: logits of about +-30 in natural units; x32:
    about +-100) so the softmax is dominated by a few keys and each CTA's
    partial logits are large.  The two-CTA split must still give O within
    the bf16 tolerance and LSE within 1e-3 relative.  Scaling bf16 values
    by a power of two is exact, so the oracle sees the same operands."""
    wl = inputs.make_prefill(seed=31 + scale, device=DEV, L=2600)
    wl = dataclasses.replace(wl, q=wl.q * scale)
    if fp8kv:
        wl = inputs.with_fp8_kv(wl)
    k = 2048
    prob = api.Problem(wl)
    sel = inputs.random_index_sets(wl.q_pos, k, seed=5)
    o, lse = _attn(prob, sel, k)
    view = OracleView(wl)
    rows = sorted(set(np.linspace(0, wl.num_q - 1, 24).astype(int)) | {0, 2047, wl.num_q - 1})
    worst = 0.0
    for i in rows:
        ro, rl = view.attention(i, sel[i].numpy())
        err = np.abs(o[i] - ro).max()
        worst = max(worst, err)
        assert err <= ATTN_ATOL_BF16, f"query {i}: max |O - O_ref| = {err}"
        assert np.abs(lse[i] - rl).max() <= 1e-3 * max(1.0, np.abs(rl).max()), i
    print(f"peaked x{scale} fp8kv={fp8kv}: worst |O - O_ref| = {worst:.3e}")


# --------------------------------------------------------------------------- device-side checks, tensor-core paths

def test_tensor_core_attention_flags_index_past_position():
    """bf16 latent attention (tcgen05 kernel): an entry later than the query's
    position is flagged, masked, and the row equals attention without it."""
    wl = inputs.make_prefill(seed=41, device=DEV, L=300, topk=64)
    prob = api.Problem(wl)
    assert api.dsa_check_device_error() == api.DSA_OK
    sel = inputs.random_index_sets(wl.q_pos, 64, seed=4)
    bad = sel.clone()
    bad[7, 8] = 50                                   # query 7 selects positions 0..7, then padding
    out = torch.empty((wl.num_q, wl.H, wl.d_v), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((wl.num_q, wl.H), dtype=torch.float32, device=DEV)
    api.dsa_sparse_attn(prob.batch.desc(), prob.cache.desc(), prob.at, bad.to(DEV), 64, out, lse)
    assert api.dsa_check_device_error() == api.DSA_ERR_BOUNDS
    assert api.dsa_check_device_error() == api.DSA_OK
    assert bool(torch.isfinite(out.float()).all()) and bool(torch.isfinite(lse).all())
    o_ref, l_ref = _attn(prob, sel, 64)
    assert np.array_equal(out.float().cpu().numpy(), o_ref) and np.array_equal(lse.cpu().numpy(), l_ref)


@pytest.mark.parametrize("bad_block", [-1, 10_000])
def test_tensor_core_paths_flag_bad_block_ids(bad_block):
    """Paged FP8 indexer and bf16 attention (tcgen05 kernels) with a block
    table entry that is negative or past the pool: the access is skipped,
    DSA_ERR_BOUNDS is recorded, the keys of that block score -inf, and every
    output stays finite."""
    wm = inputs.make_mixed(seed=42, device=DEV, batch=2, lo=600, hi=900, prefill=100, decode=3, block=64)
    bt = wm.block_table.clone()
    bt[0, 2] = bad_block                             # positions 128..191 of sequence 0
    wm = dataclasses.replace(wm, block_table=bt)
    prob = api.Problem(wm)
    assert api.dsa_check_device_error() == api.DSA_OK
    ld = (wm.max_kv + 3) // 4 * 4
    sc = torch.empty((wm.num_q, ld), dtype=torch.float32, device=DEV)
    api.dsa_index_scores(prob.batch.desc(), prob.cache.desc(), prob.ix, sc)
    assert api.dsa_check_device_error() == api.DSA_ERR_BOUNDS
    rows0 = (wm.q_seq == 0).nonzero().flatten()
    assert bool(torch.isneginf(sc[rows0][:, 128:192]).all())
    assert bool(torch.isfinite(sc[rows0][:, :128]).all())
    from dsa_testutil import run_forward
    idx, out, lse = run_forward(prob)
    assert api.dsa_check_device_error() == api.DSA_ERR_BOUNDS
    assert bool(torch.isfinite(out.float()).all()) and bool(torch.isfinite(lse).all())
    assert api.dsa_check_device_error() == api.DSA_OK
