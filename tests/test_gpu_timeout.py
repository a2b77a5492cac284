"""Failure detection on the GPU without a fault: every device-side wait of the
tensor-core kernels is bounded, and an expired wait ends the kernel with
DSA_ERR_TIMEOUT instead of a hang.  Here the tensor-core indexer runs with
its waits bounded by a few hundred clocks, far less than one TMA load takes,
so its pipeline gives up; the kernel must drain its own copies and MMAs,
free its tensor memory, report the timeout, and leave the context usable for
the correct calls that follow."""
import numpy as np
import pytest
import torch

from oracle.workload_view import OracleView
from sparse_attention_long_11_b300 import api, inputs
from dsa_testutil import ATTN_ATOL_BF16, indexer_tolerance, run_forward

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _scores(prob, limit=None):
    wl = prob.wl
    ld = (wl.max_kv + 3) // 4 * 4
    sc = torch.zeros((wl.num_q, ld), dtype=torch.float32, device=DEV)
    if limit is None:
        api.dsa_index_scores(prob.batch.desc(), prob.cache.desc(), prob.ix, sc)
    else:
        api.dsa_index_scores_wait_limit(prob.batch.desc(), prob.cache.desc(), prob.ix, sc, limit)
    return sc


def test_expired_wait_reports_timeout_and_the_context_recovers():
    wl = inputs.make_prefill(seed=51, device=DEV, L=1500)      # FP8 tensor-core indexer, several key tiles
    prob = api.Problem(wl)
    assert api.dsa_check_device_error() == api.DSA_OK
    for _ in range(2):                                          # twice: recovery is repeatable
        _scores(prob, limit=300)
        assert api.dsa_check_device_error() == api.DSA_ERR_TIMEOUT
        assert api.dsa_check_device_error() == api.DSA_OK       # the word was cleared
    # a generous explicit limit behaves like the default
    a = _scores(prob, limit=2_000_000_000)
    assert api.dsa_check_device_error() == api.DSA_OK
    b = _scores(prob)
    assert api.dsa_check_device_error() == api.DSA_OK
    assert torch.equal(a, b)
    view = OracleView(wl)
    sc = b.cpu().numpy()
    for i in (0, 700, 1499):
        tol, ref = indexer_tolerance(view, i)
        assert np.all(np.abs(sc[i, :i + 1] - ref) <= tol), i
    # the whole forward is correct right after a timeout
    _scores(prob, limit=300)
    assert api.dsa_check_device_error() == api.DSA_ERR_TIMEOUT
    idx, out, lse = run_forward(prob)
    assert api.dsa_check_device_error() == api.DSA_OK
    for i in (100, 1499):
        ro, rl = view.attention(i, idx[i].cpu().numpy())
        assert np.abs(out[i].float().cpu().numpy() - ro).max() <= ATTN_ATOL_BF16


def test_wait_limit_is_validated():
    wl = inputs.make_tiny(seed=52, device=DEV, L=64, topk=16)
    prob = api.Problem(wl)
    sc = torch.zeros((wl.num_q, 64), dtype=torch.float32, device=DEV)
    with pytest.raises(api.DSAError) as e:
        api.dsa_index_scores_wait_limit(prob.batch.desc(), prob.cache.desc(), prob.ix, sc, 0)
    assert e.value.status == api.DSA_ERR_INVALID_ARG
