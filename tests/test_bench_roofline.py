"""The benchmark's work counts and roofline arithmetic (CPU).  The pair
counts of the long prefill are pinned to their closed forms; the roofline
object must pick the kernel with the most device time and divide its
algorithmic work per launch by its average launch time."""
import math
import os
import sys
import types

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

PEAKS = {"hbm": 6000.0, "bf16": 1800.0, "bf16_sus": 1400.0, "src": "test"}


def _prefill(L=32768, k=2048):
    return types.SimpleNamespace(q_pos=torch.arange(L, dtype=torch.int32), topk=k)


def test_pair_counts_of_the_long_prefill():
    n_idx, n_attn = bench._pairs(_prefill())
    L, k = 32768, 2048
    # every causal pair of the queries with more than k keys (t + 1 > k)
    assert n_idx == L * (L + 1) // 2 - k * (k + 1) // 2 == 534_789_120
    assert n_attn == k * (k + 1) // 2 + (L - k) * k == 65_012_736      # min(t + 1, k) per query


def test_work_units_per_pair():
    assert bench.FLOP_PER_ATTN_PAIR == 2 * 128 * 576 + 2 * 128 * 512  # QK^T over 576 dims, PV over 512
    assert bench.FLOP_PER_IDX_PAIR == 2 * 64 * 128                    # 64 heads x 128 dims
    assert bench.BYTES_PER_IDX_KEY == 132 and bench.BYTES_PER_ATTN_KEY == 1152


def test_prefill_roofline_takes_the_dominant_kernel():
    wl = _prefill()
    steps = 5
    per_stage = {"indexer": [40, 40 * 0.85], "topk": [40, 40 * 0.24], "attention": [40, 40 * 2.46]}
    r = bench._roofline_prefill(wl, per_stage, steps, PEAKS)
    assert r["kernel"] == "attention" and r["bound"] == "tensor" and r["launches"] == 40
    # 8 launches per step: each does an eighth of the step's 65,012,736 pairs in 2.46 ms
    want = 65_012_736 / 8 * 278_528 / 2.46e-3 / 1e12
    assert math.isclose(r["achieved"], want, rel_tol=1e-12)
    # a kernel timed inside a sub-second step is held to the burst peak; the
    # sustained (power-capped) peak is reported beside it
    assert math.isclose(r["frac"], want / 1800.0, rel_tol=1e-12)
    assert math.isclose(r["frac_of_sustained"], want / 1400.0, rel_tol=1e-12)
    # an indexer-dominated step reports against twice the bf16 peak (FP8)
    per_stage["indexer"][1] = 40 * 5.0
    r = bench._roofline_prefill(wl, per_stage, steps, PEAKS)
    want = 534_789_120 / 8 * 16_384 / 5.0e-3 / 1e12
    assert r["kernel"] == "indexer" and math.isclose(r["achieved"], want, rel_tol=1e-12)
    assert math.isclose(r["peak"], 3600.0) and r["traffic"] is None


def test_decode_roofline_counts_the_key_bytes_streamed():
    # 64 sequences, one query each at position 65535: 65536 keys of 132 bytes per query
    wl = types.SimpleNamespace(q_pos=torch.full((64,), 65535, dtype=torch.int32), topk=2048)
    n_idx, n_attn = bench._pairs(wl)
    assert n_idx == 64 * 65536 and n_attn == 64 * 2048
    per_stage = {"indexer": [10, 10 * 0.146], "topk": [10, 10 * 0.034], "attention": [10, 10 * 0.061]}
    r = bench._roofline_decode(wl, per_stage, 10, PEAKS)
    want = 64 * 65536 * 132 / 0.146e-3 / 1e9                          # 553.6 MB per launch
    assert r["kernel"] == "indexer" and r["bound"] == "hbm"
    assert math.isclose(r["achieved"], want, rel_tol=1e-12) and math.isclose(r["frac"], want / 6000.0)


def test_decode_stage_fractions_count_each_stage_bytes():
    wl = types.SimpleNamespace(q_pos=torch.full((64,), 65535, dtype=torch.int32), topk=2048, num_q=64,
                               H=128, d_qk=576, d_v=512)
    per_stage = {"indexer": [10, 10 * 0.146], "topk": [10, 10 * 0.034], "attention": [10, 10 * 0.061]}
    r = bench._decode_stage_roofline(wl, per_stage, 10, PEAKS)
    assert r["indexer"]["bytes"] == 64 * 65536 * 132
    assert r["topk"]["bytes"] == 64 * 2048 * 8 + 64 * 2048 * 4           # k candidate keys read, index rows written
    assert r["attention"]["bytes"] == 64 * 2048 * 1152 + 64 * 128 * (576 + 512) * 2   # gather + q in + O out
    for name, ms in (("indexer", 0.146), ("topk", 0.034), ("attention", 0.061)):
        assert math.isclose(r[name]["ms"], ms)
        assert math.isclose(r[name]["frac"], r[name]["bytes"] / (ms / 1e3) / 1e9 / 6000.0)
