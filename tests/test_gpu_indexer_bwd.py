"""dsa_indexer_kl_backward on the GPU against the oracle's
indexer_kl_backward: loss, pi - p, dw and dq per query, dk summed over the
batch, with tolerances from each sum's magnitude; plus the identity
sum_e g_e I_e = sum_j w_j dw_j = sum_j <dq_j, q_j> at full size."""
import numpy as np
import pytest
import torch

from oracle import dsa_oracle as O
from oracle.workload_view import OracleView
from sparse_attention_long_11_b300 import api, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = 1e-3   # times the magnitude of each sum (|g| widened by 1e-4 (pi + p))


def _run(wl, idx, k, p):
    prob = api.Problem(wl)
    nq, H, d = wl.num_q, wl.H_I, wl.d_I
    loss = torch.empty(nq, dtype=torch.float32, device=DEV)
    g = torch.empty((nq, k), dtype=torch.float32, device=DEV)
    dw = torch.empty((nq, H), dtype=torch.float32, device=DEV)
    dq = torch.empty((nq, H, d), dtype=torch.float32, device=DEV)
    dk = torch.zeros((wl.num_rows, d), dtype=torch.float32, device=DEV)
    api.dsa_indexer_kl_backward(prob.batch.desc(), prob.cache.desc(), prob.ix, idx, k, p, loss, dw, dq, dk, g)
    assert api.dsa_check_device_error() == api.DSA_OK
    return [x.cpu().numpy() for x in (loss, g, dw, dq, dk)]


def _selected(wl, k):
    """The top-k entries the forward would select (the GPU's own stages)."""
    prob = api.Problem(wl)
    ld = (wl.max_kv + 3) // 4 * 4
    sc = torch.empty((wl.num_q, ld), dtype=torch.float32, device=DEV)
    api.dsa_index_scores(prob.batch.desc(), prob.cache.desc(), prob.ix, sc)
    idx = torch.empty((wl.num_q, k), dtype=torch.int32, device=DEV)
    api.dsa_topk(prob.batch.desc(), sc, k, idx)
    assert api.dsa_check_device_error() == api.DSA_OK
    return idx


def _check(wl, idx, p, got, rows=None):
    loss, g, dw, dq, dk = got
    view = OracleView(wl)
    idx_h, p_h = idx.cpu().numpy(), p.cpu().numpy()
    rows = range(wl.num_q) if rows is None else rows
    dk_ref = np.zeros_like(dk, dtype=np.float64)
    dk_mag = np.zeros_like(dk, dtype=np.float64)
    for i in rows:
        seq, pos = int(view.q_seq[i]), int(view.q_pos[i])
        k_vals, k_scale, _ = view.seq_cache(seq, pos + 1)
        qi, qs, w, _ = view.query_inputs(i)
        r = O.indexer_kl_backward(qi, w, k_vals, idx_h[i], p_h[i], qs, k_scale)
        assert abs(loss[i] - r["loss"]) <= 1e-4 * max(1.0, abs(r["loss"])), f"query {i}: loss"
        assert np.all(np.abs(g[i] - r["g"]) <= 1e-4 * (np.abs(r["g"]) + p_h[i]) + 1e-7), f"query {i}: g"
        assert np.all(np.abs(dw[i] - r["dw"]) <= TOL * r["mag_dw"] + 1e-30), f"query {i}: dw"
        assert np.all(np.abs(dq[i] - r["dq"]) <= TOL * r["mag_dq"] + 1e-30), f"query {i}: dq"
        phys = wl.logical_rows(seq, pos + 1).numpy()
        for e, s in enumerate(idx_h[i]):
            if s >= 0:
                dk_ref[phys[s]] += r["dk"][e]
                dk_mag[phys[s]] += r["mag_dk"][e]
    return dk_ref, dk_mag


def test_kl_backward_fp8_selected_entries():
    wl = inputs.make_prefill(seed=21, device=DEV, L=700, topk=128)
    idx = _selected(wl, 128)
    p = inputs.kl_targets(idx, seed=3)
    got = _run(wl, idx, 128, p)
    dk_ref, dk_mag = _check(wl, idx, p, got)
    assert np.all(np.abs(got[4] - dk_ref) <= TOL * dk_mag + 1e-30)


def test_kl_backward_dense_warmup():
    """Every position 0..t is an entry (k >= L): the dense warm-up's loss."""
    L = 300
    wl = inputs.make_prefill(seed=22, device=DEV, L=L, topk=L)
    pos = torch.arange(L, dtype=torch.int32)
    idx = torch.where(torch.arange(L)[None, :] <= pos[:, None], torch.arange(L, dtype=torch.int32)[None, :],
                      torch.full((L, L), -1, dtype=torch.int32)).to(DEV)
    p = inputs.kl_targets(idx, seed=4)
    got = _run(wl, idx, L, p)
    dk_ref, dk_mag = _check(wl, idx, p, got)
    assert np.all(np.abs(got[4] - dk_ref) <= TOL * dk_mag + 1e-30)


def test_kl_backward_f32_operands_and_random_entries():
    wl = inputs.make_tiny(seed=23, device=DEV)
    idx = inputs.random_index_sets(wl.q_pos, 32, seed=5).to(DEV)
    p = inputs.kl_targets(idx, seed=5)
    got = _run(wl, idx, 32, p)
    dk_ref, dk_mag = _check(wl, idx, p, got)
    assert np.all(np.abs(got[4] - dk_ref) <= TOL * dk_mag + 1e-30)


def test_kl_backward_paged_cache():
    wl = inputs.make_mixed(seed=24, device=DEV, batch=2, lo=1200, hi=1500, prefill=40, decode=3, block=64)
    idx = _selected(wl, 256)
    p = inputs.kl_targets(idx, seed=6)
    got = _run(wl, idx, 256, p)
    dk_ref, dk_mag = _check(wl, idx, p, got)
    assert np.all(np.abs(got[4] - dk_ref) <= TOL * dk_mag + 1e-30)


def test_kl_backward_edge_rows():
    """A row of padding only (nothing to learn), a one-hot target, one entry."""
    wl = inputs.make_prefill(seed=25, device=DEV, L=200, topk=64)
    idx = inputs.random_index_sets(wl.q_pos, 64, seed=7)
    idx[10] = -1                                   # no entries
    idx[20, 1:] = -1                               # a single entry
    idx = idx.to(DEV)
    p = inputs.kl_targets(idx, seed=8)
    p[20] = 0.0
    p[20, 0] = 1.0                                 # the single entry holds all the target
    p[30] = 0.0
    p[30, 0] = 1.0                                 # one-hot target
    got = _run(wl, idx, 64, p)
    loss, g, dw, dq, _ = got
    assert loss[10] == 0 and np.all(dw[10] == 0) and np.all(dq[10] == 0) and np.all(g[10] == 0)
    assert abs(loss[20]) < 1e-6 and np.all(np.abs(dw[20]) < 1e-6)
    _check(wl, idx, p, got, rows=[10, 20, 30, 31, 199])


def test_kl_backward_full_size_identities():
    """4096 queries x k = 2048 (the long prefill's last call): sampled queries
    against the oracle, and at every query sum_e g_e I_e = sum_j w_j dw_j =
    sum_j <dq_j, q_j>, and over the batch sum_s <dk_s, k_s> = sum_t sum_e g_e I_e."""
    torch.cuda.empty_cache()
    L = 4096
    wl = inputs.make_prefill(seed=26, device=DEV, L=L)
    idx = _selected(wl, 2048)
    p = inputs.kl_targets(idx, seed=9)
    loss, g, dw, dq, dk = _run(wl, idx, 2048, p)
    _check(wl, idx, p, (loss, g, dw, dq, dk), rows=[0, 2047, 2048, 3000, 4095])
    # the scores of the selected entries, in fp64 from the dequantised operands
    qd = O.decode_e4m3(wl.q_idx.cpu().numpy()) * wl.q_scale.cpu().numpy()[..., None]
    kd = O.decode_e4m3(wl.k_idx.cpu().numpy()) * wl.k_scale.cpu().numpy()[:, None]
    w = wl.w.cpu().numpy().astype(np.float64)
    idx_h = idx.cpu().numpy()
    gI_tot, gI_mag = 0.0, 0.0
    for i in range(0, L, 97):
        sel = idx_h[i][idx_h[i] >= 0]
        x = qd[i] @ kd[sel].T
        I = w[i] @ np.maximum(x, 0)
        gI = float(g[i][: len(sel)] @ I)
        scale = float(np.abs(g[i][: len(sel)]) @ np.abs(I)) + 1e-12
        assert abs(float(w[i] @ dw[i]) - gI) <= 1e-3 * scale, i
        assert abs(float((dq[i] * qd[i]).sum()) - gI) <= 1e-3 * scale, i
    for i in range(L):
        sel = idx_h[i][idx_h[i] >= 0]
        x = qd[i] @ kd[sel].T
        I = w[i] @ np.maximum(x, 0)
        gI_tot += float(g[i][: len(sel)] @ I)
        gI_mag += float(np.abs(g[i][: len(sel)]) @ np.abs(I))
    assert abs(float((dk.astype(np.float64) * kd).sum()) - gI_tot) <= 1e-4 * gI_mag
