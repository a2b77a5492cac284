"""The seeded input generators (CPU): determinism, and the properties the
tests and the benchmark rely on.  They hold none of the method's
arithmetic; these checks are about the inputs only."""
import numpy as np
import torch

from oracle import dsa_oracle as O
from sparse_attention_long_11_b300 import inputs


def test_generators_are_seeded_and_deterministic():
    a = inputs.randn((64, 32), 3, "x")
    assert torch.equal(a, inputs.randn((64, 32), 3, "x"))
    assert not torch.equal(a, inputs.randn((64, 32), 4, "x"))
    assert not torch.equal(a, inputs.randn((64, 32), 3, "y"))


def test_kl_targets_are_distributions_over_the_valid_entries():
    pos = torch.arange(0, 400, 7, dtype=torch.int32)
    idx = inputs.random_index_sets(pos, 32, seed=2)
    idx[5] = -1                                             # a row with no entries
    p = inputs.kl_targets(idx, seed=2)
    valid = idx >= 0
    assert torch.all(p[~valid] == 0) and torch.all(p >= 0)
    sums = p.sum(dim=1)
    has = valid.any(dim=1)
    assert torch.allclose(sums[has], torch.ones_like(sums[has]), atol=1e-6)
    assert torch.all(sums[~has] == 0)
    assert bool(((p == 0) & valid).any())                   # exact zero targets occur (0 log 0)
    assert torch.equal(p, inputs.kl_targets(idx, seed=2))


def test_fp8_kv_cache_is_the_key_encoding_of_the_bf16_rows():
    wl = inputs.make_prefill(seed=1, L=96, topk=32)
    w8 = inputs.with_fp8_kv(wl, chunk_rows=40)              # several chunks
    assert w8.attn_dtype == "fp8kv" and w8.kv.dtype == torch.uint8 and w8.kv.shape == wl.kv.shape
    codes, scale = O.quantize_e4m3_rows(wl.kv.float().numpy())
    assert np.array_equal(w8.kv.numpy(), codes)
    assert np.array_equal(w8.kv_scale.numpy().view(np.uint32), scale.view(np.uint32))
    # everything else is shared with the bf16 workload
    assert w8.q is wl.q and w8.k_idx is wl.k_idx and w8.chunks == wl.chunks
