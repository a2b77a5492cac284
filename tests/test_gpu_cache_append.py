"""dsa_cache_append on the GPU against the oracle's key-cache encoding:
codes and scales bit for bit, latent rows copied exactly, only the addressed
rows written, out-of-range tokens flagged and skipped."""
import numpy as np
import pytest
import torch

from oracle import dsa_oracle as O
from sparse_attention_long_11_b300 import api, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _paged_cache(num_seqs=3, blocks_per_seq=5, block=64, seed=4):
    g = torch.Generator().manual_seed(seed)
    total = num_seqs * blocks_per_seq
    perm = torch.randperm(total, generator=g).to(torch.int32).view(num_seqs, blocks_per_seq)
    rows = total * block
    return api.Cache(num_seqs, rows, 0, perm.to(DEV), block), perm, rows, block


def _special_rows(n, seed, dtype):
    x = inputs.randn((n, 128), seed, "append_k", DEV)
    x[0] = 0.0                                  # all-zero row: scale 1, codes 0
    x[1, ::2] = -0.0                            # signed zeros keep their sign
    x[2] *= 1e-6                                # tiny values: subnormal codes after scaling
    x[3, 7] = 3e4                               # one outlier: everything else rounds towards 0
    return x.to(dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_cache_append_matches_oracle_bit_for_bit(dtype):
    cache, perm, rows, block = _paged_cache()
    n = 40
    g = torch.Generator().manual_seed(8)
    seq = torch.randint(0, 3, (n,), generator=g, dtype=torch.int32)
    pos = torch.randperm(5 * block, generator=g)[:n].to(torch.int32)      # distinct positions
    pos[:3] = torch.tensor([0, block - 1, 5 * block - 1], dtype=torch.int32)
    seq[:3] = torch.tensor([0, 1, 2], dtype=torch.int32)
    # make (seq, pos) pairs distinct
    key = seq.to(torch.int64) * 100000 + pos.to(torch.int64)
    _, first = np.unique(key.numpy(), return_index=True)
    keep = torch.from_numpy(np.sort(first))
    seq, pos = seq[keep], pos[keep]
    n = seq.numel()
    k_new = _special_rows(n, 9, dtype)
    kv_new = inputs.randn((n, 576), 9, "append_kv", DEV).to(torch.bfloat16)
    k_cache = torch.full((rows, 128), 0x5A, dtype=torch.uint8, device=DEV)     # sentinels
    k_scale = torch.full((rows,), -7.0, dtype=torch.float32, device=DEV)
    kv_cache = torch.full((rows, 576), 3.0, dtype=torch.bfloat16, device=DEV)
    api.dsa_cache_append(cache.desc(), seq.to(DEV), pos.to(DEV), k_new, k_cache, k_scale, kv_new, kv_cache)
    assert api.dsa_check_device_error() == api.DSA_OK

    codes, scale = O.quantize_e4m3_rows(k_new.float().cpu().numpy())
    phys = (perm[seq.long(), (pos // block).long()].to(torch.int64) * block + (pos % block)).numpy()
    kc, ks, kvc = k_cache.cpu().numpy(), k_scale.cpu().numpy(), kv_cache.cpu()
    assert np.array_equal(kc[phys], codes)
    assert np.array_equal(ks[phys].view(np.uint32), scale.view(np.uint32))
    assert torch.equal(kvc[torch.from_numpy(phys)], kv_new.cpu())
    untouched = np.setdiff1d(np.arange(rows), phys)
    assert np.all(kc[untouched] == 0x5A) and np.all(ks[untouched] == -7.0)
    assert bool((kvc[torch.from_numpy(untouched)] == 3.0).all())
    # the special rows came out as the encoding says
    assert np.all(codes[0] == 0) and scale[0] == 1.0
    assert np.all(codes[1, ::2][k_new[1, ::2].float().cpu().numpy() == 0] == 0x80)


def test_cache_append_flags_and_skips_out_of_range_tokens():
    cache, perm, rows, block = _paged_cache()
    seq = torch.tensor([0, 1, 2, 7], dtype=torch.int32)            # sequence 7 does not exist
    pos = torch.tensor([3, 5 * block, 4, 0], dtype=torch.int32)    # position 5*block is past the table
    k_new = _special_rows(4, 12, torch.float32)
    k_cache = torch.zeros((rows, 128), dtype=torch.uint8, device=DEV)
    k_scale = torch.zeros((rows,), dtype=torch.float32, device=DEV)
    api.dsa_cache_append(cache.desc(), seq.to(DEV), pos.to(DEV), k_new, k_cache, k_scale)
    assert api.dsa_check_device_error() == api.DSA_ERR_BOUNDS
    codes, scale = O.quantize_e4m3_rows(k_new.cpu().numpy())
    ok = [0, 2]
    phys = (perm[seq[ok].long(), (pos[ok] // block).long()].to(torch.int64) * block + pos[ok] % block).numpy()
    kc, ks = k_cache.cpu().numpy(), k_scale.cpu().numpy()
    assert np.array_equal(kc[phys], codes[ok]) and np.array_equal(ks[phys], scale[ok])
    assert int((ks != 0).sum()) == 2                               # nothing else was written


def test_cache_append_fp8_latent_rows_match_oracle():
    """Latent rows into an FP8 cache: each row encoded like a key (oracle
    quantize_e4m3_rows on the bf16 values), codes and scales bit for bit, and
    the whole cache equal to the generator's FP8 latent cache."""
    cache, perm, rows, block = _paged_cache(seed=6)
    wl_rows = rows
    kv_new = inputs.randn((wl_rows, 576), 14, "append_kv8", DEV).to(torch.bfloat16)
    kv_new[3] = 0.0                                                # all-zero row: scale 1
    kv_new[5, 100] = 5e3                                           # an outlier row
    # every logical position of the three sequences, so the whole cache is written
    seq = torch.arange(3, dtype=torch.int32).repeat_interleave(5 * block)
    pos = torch.arange(5 * block, dtype=torch.int32).repeat(3)
    k_new = inputs.randn((wl_rows, 128), 15, "append_k8", DEV)
    k_cache = torch.empty((rows, 128), dtype=torch.uint8, device=DEV)
    k_scale = torch.empty((rows,), dtype=torch.float32, device=DEV)
    kv_cache = torch.full((rows, 576), 0x5A, dtype=torch.uint8, device=DEV)
    kv_scale = torch.full((rows,), -7.0, dtype=torch.float32, device=DEV)
    api.dsa_cache_append(cache.desc(), seq.to(DEV), pos.to(DEV), k_new, k_cache, k_scale, kv_new, kv_cache,
                         kv_scale=kv_scale)
    assert api.dsa_check_device_error() == api.DSA_OK
    phys = (perm[seq.long(), (pos // block).long()].to(torch.int64) * block + (pos % block)).numpy()
    codes, scale = O.quantize_e4m3_rows(kv_new.float().cpu().numpy())
    kvc, kvs = kv_cache.cpu().numpy(), kv_scale.cpu().numpy()
    assert np.array_equal(kvc[phys], codes)
    assert np.array_equal(kvs[phys].view(np.uint32), scale.view(np.uint32))
    assert scale[3] == 1.0 and np.all(codes[3] == 0)
    # the generator's encoding of the same rows (in physical order)
    order = torch.from_numpy(np.argsort(phys))
    c8, s8 = inputs.quantize_fp8_rows(kv_new[order.to(DEV)].float())
    assert torch.equal(kv_cache, c8) and torch.equal(kv_scale, s8)


def test_cache_append_rebuilds_the_generated_fp8_key_cache():
    """Appending the raw keys of a workload reproduces the FP8 key cache the
    generator built for it (same encoding, so the forward's inputs and a
    decode loop's appends agree)."""
    L = 640
    raw = inputs.randn((L, 128), 0, "k_idx", DEV)
    want_codes, want_scale = inputs.quantize_fp8_rows(raw)
    cache = api.Cache(1, L, L, None, 0)
    k_cache = torch.empty((L, 128), dtype=torch.uint8, device=DEV)
    k_scale = torch.empty((L,), dtype=torch.float32, device=DEV)
    pos = torch.arange(L, dtype=torch.int32, device=DEV)
    api.dsa_cache_append(cache.desc(), torch.zeros(L, dtype=torch.int32, device=DEV), pos, raw, k_cache, k_scale)
    assert api.dsa_check_device_error() == api.DSA_OK
    assert torch.equal(k_cache, want_codes) and torch.equal(k_scale, want_scale)
