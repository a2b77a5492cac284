"""dsa_forward_noalloc: the forward for callers that cannot allocate device
memory (a fixed memory plan, a plugin host that forbids allocation, a serving
loop where cudaMalloc must not synchronise the device).  Its scratch is a
fixed array inside the library, so the test checks that two calls in a row --
the second one seeing the first one's leftovers in that array -- both match
dsa_forward with a caller-provided workspace.  Collected last on purpose."""
import numpy as np
import pytest
import torch

from sparse_attention_long_11_b300 import api, inputs
from dsa_testutil import ATTN_ATOL_BF16, ATTN_ATOL_F32, run_forward

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _noalloc(wl):
    prob = api.Problem(wl)
    idx = torch.full((wl.num_q, wl.topk), -7, dtype=torch.int32, device=DEV)
    out = torch.full((wl.num_q, wl.H, wl.d_v), float("nan"), dtype=prob.out_dtype(), device=DEV)
    lse = torch.full((wl.num_q, wl.H), float("nan"), dtype=torch.float32, device=DEV)
    qd, ix, at = prob.rows(0, wl.num_q)
    api.dsa_forward_noalloc(qd, prob.cache.desc(), ix, wl.topk, at, idx, out, lse)
    assert api.dsa_check_device_error() == api.DSA_OK
    return idx, out, lse


def _compare(wl, atol):
    ref = run_forward(api.Problem(wl), chunks=[(0, wl.num_q)])
    got = _noalloc(wl)
    assert torch.equal(got[0], ref[0])
    err = (got[1].float() - ref[1].float()).abs().max().item()
    assert err <= atol, err
    assert torch.allclose(got[2], ref[2], rtol=1e-5, atol=1e-5)


def test_noalloc_matches_forward_on_two_calls_in_a_row():
    # first call: FP8/BF16 shapes, enough rows to need several staging rounds
    _compare(inputs.make_prefill(seed=21, device=DEV, L=2600), ATTN_ATOL_BF16)
    # second call: different shapes, scratch still holds the first call's rows
    _compare(inputs.make_tiny(seed=22, device=DEV), ATTN_ATOL_F32)


def test_noalloc_rejects_too_long_context():
    wl = inputs.make_tiny(seed=23, device=DEV, L=64, topk=16)
    prob = api.Problem(wl)
    qd, ix, at = prob.rows(0, wl.num_q)
    qd.max_kv = api.NOALLOC_MAX_KV + 4
    idx = torch.empty((wl.num_q, 16), dtype=torch.int32, device=DEV)
    out = torch.empty((wl.num_q, wl.H, wl.d_v), dtype=torch.float32, device=DEV)
    lse = torch.empty((wl.num_q, wl.H), dtype=torch.float32, device=DEV)
    with pytest.raises(api.DSAError) as e:
        api.dsa_forward_noalloc(qd, prob.cache.desc(), ix, 16, at, idx, out, lse)
    assert e.value.status == api.DSA_ERR_UNSUPPORTED
