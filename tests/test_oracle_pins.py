"""Pins for the CPU oracle: each test ties the oracle to something other than
itself -- hand-computed fixtures, exact integer arithmetic, a library routine
on a case that reduces to it, brute force on tiny inputs, or an identity of
the mathematics -- chosen so that a dropped term, a wrong sign, a wrong index
or a transposed operand in the oracle fails at least one of them."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import dsa_oracle as O
from sparse_attention_long_11_b300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------- decoders

def test_e4m3_closed_form_values():
    # OCP FP8 E4M3: bias 7, 3 mantissa bits, subnormals below 2^-6, max 448, S.1111.111 = NaN
    expect = {0x00: 0.0, 0x38: 1.0, 0x40: 2.0, 0x3C: 1.5, 0x7E: 448.0, 0xFE: -448.0,
              0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x30: 0.5, 0xB8: -1.0}
    for code, v in expect.items():
        assert O.decode_e4m3(code) == v, hex(code)
    assert math.copysign(1.0, O.decode_e4m3(0x80)) == -1.0 and O.decode_e4m3(0x80) == 0.0
    assert np.isnan(O.decode_e4m3(0x7F)) and np.isnan(O.decode_e4m3(0xFF))
    pos = O.decode_e4m3(np.arange(0x00, 0x7F))
    assert np.all(np.diff(pos) > 0)          # strictly increasing over the finite positive codes
    assert np.array_equal(O.decode_e4m3(np.arange(0x80, 0xFF)), -pos)


def test_e4m3_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.decode_e4m3(codes.numpy())
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def test_e4m3_encoder_round_trip_and_ties():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = O.decode_e4m3(codes)
    assert np.array_equal(O.encode_e4m3(vals), codes)             # every finite code (incl. -0) round-trips
    pos = O.E4M3_TABLE[:0x7F]
    mids = (pos[:-1] + pos[1:]) / 2                                # exact midpoints of neighbouring codes
    got = O.encode_e4m3(mids)
    lo = np.arange(0x7E)
    want = np.where(lo % 2 == 0, lo, lo + 1)                       # ties to the even code
    assert np.array_equal(got, want.astype(np.uint8))
    assert np.array_equal(O.encode_e4m3([448.0, 449.0, 1e30, -1e30, -464.0]),
                          np.array([0x7E, 0x7E, 0x7E, 0xFE, 0xFE], dtype=np.uint8))   # saturation


def test_e4m3_encoder_matches_torch_float8_on_random_values():
    g = torch.Generator().manual_seed(11)
    x = (torch.randn(200000, generator=g) * torch.exp2(torch.randint(-12, 10, (200000,), generator=g).float()))
    x = x.clamp(-448, 448)                                         # torch's cast does not saturate
    want = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.encode_e4m3(x.numpy()), want)


def test_row_quantisation_scale_and_extremes():
    x = np.array([[0.5, -2.0, 1.0, 0.0], [0.0, 0.0, 0.0, 0.0], [-3.0, 1e-9, 2.0, -0.0]], dtype=np.float32)
    codes, scale = O.quantize_e4m3_rows(x)
    assert scale.dtype == np.float32
    assert scale[0] == np.float32(2.0) / np.float32(448.0) and scale[1] == 1.0
    assert codes[0, 1] == 0xFE and codes[2, 0] == 0xFE             # each row's largest magnitude -> -448
    assert np.all(codes[1] == 0) and codes[2, 3] == 0x80            # zero row; -0.0 keeps its sign
    # decoding reproduces every element within half a code step (relative 2^-4) or the subnormal step
    back = O.decode_e4m3(codes) * scale[:, None]
    step = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -9 * scale[:, None])
    assert np.all(np.abs(back - x) <= step)


def test_bf16_matches_torch():
    x = torch.randn(4096, dtype=torch.float32) * 100
    b = x.to(torch.bfloat16)
    bits = b.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.decode_bf16(bits), b.to(torch.float64).numpy())


def test_bf16_rounding_ties_and_torch():
    # hand cases: exact, below/above the halfway point, ties to the even pattern, sign
    one = np.float32(1.0)
    ulp = 2.0 ** -7                                             # bf16 spacing just above 1
    cases = {1.0: 1.0, 1.0 + 2 ** -9: 1.0, 1.0 + 2 ** -8 + 2 ** -20: 1.0 + ulp,
             1.0 + 2 ** -8: 1.0,                                # tie, 1.0 is even -> stays
             1.0 + 3 * 2 ** -8: 1.0 + 2 * ulp,                 # tie between 1+ulp (odd) and 1+2ulp (even)
             -(1.0 + 3 * 2 ** -8): -(1.0 + 2 * ulp), 0.0: 0.0}
    for x, want in cases.items():
        assert O.round_bf16(np.float32(x)) == want, x
    assert O.round_bf16(one) == 1.0
    # torch's float32 -> bfloat16 cast on random values and constructed ties
    g = torch.Generator().manual_seed(3)
    x = torch.randn(20000, generator=g, dtype=torch.float32) * 50
    ties = (x.view(torch.int32) & ~0xFFFF) | 0x8000
    for t in (x, ties.view(torch.float32)):
        assert np.array_equal(O.round_bf16(t.numpy()), t.to(torch.bfloat16).to(torch.float64).numpy())


def test_fp8_kv_dequantisation():
    codes = np.arange(256, dtype=np.uint8).reshape(4, 64)
    finite = ~np.isnan(O.decode_e4m3(codes))
    # scale 1 and powers of two: the product is exact and every e4m3 value is a bf16 value
    for sc in (1.0, 2.0 ** -5, 2.0 ** 7):
        got = O.dequantize_kv_e4m3(codes, np.full(4, sc, dtype=np.float32))
        assert np.array_equal(got[finite], O.decode_e4m3(codes)[finite] * sc)
    # signed zero and the subnormal step survive
    got = O.dequantize_kv_e4m3(np.array([[0x00, 0x80, 0x01, 0x7E]], dtype=np.uint8), np.array([3.0], np.float32))
    assert got[0, 0] == 0.0 and np.signbit(got[0, 1]) and got[0, 2] == 3.0 * 2.0 ** -9 and got[0, 3] == 1344.0
    # arbitrary scales: torch's float8 decode, a float32 multiply and its bfloat16 cast, bit for bit
    g = torch.Generator().manual_seed(5)
    c = torch.randint(0, 256, (300, 576), generator=g, dtype=torch.uint8)
    c[(c & 0x7F) == 0x7F] = 0x11                                # no NaN codes
    sc = torch.rand(300, generator=g, dtype=torch.float32) * 0.01 + 1e-4
    want = (c.view(torch.float8_e4m3fn).to(torch.float32) * sc[:, None]).to(torch.bfloat16).to(torch.float64)
    assert np.array_equal(O.dequantize_kv_e4m3(c.numpy(), sc.numpy()), want.numpy())
    # a quantised row comes back within the e4m3 step and the bf16 rounding of the row
    x = np.random.default_rng(0).standard_normal((8, 576)).astype(np.float32)
    q, s8 = O.quantize_e4m3_rows(x)
    back = O.dequantize_kv_e4m3(q, s8)
    assert np.all(np.abs(back - x) <= np.abs(x) * (2.0 ** -4 + 2.0 ** -8) + 2.0 ** -9 * s8[:, None])


# --------------------------------------------------------------------------- indexer

def test_indexer_hand_cases():
    for c in _load("indexer_hand.json")["cases"]:
        k = np.array(c["k"], dtype=np.float64)
        got = O.index_scores(np.array(c["q"], float), np.array(c["w"]), k, k.shape[0] - 1,
                             None if c["q_scale"] is None else np.array(c["q_scale"]),
                             None if c["k_scale"] is None else np.array(c["k_scale"]))
        assert np.array_equal(got, np.array(c["expected"])), c["note"]


def _fp8_case(seed, n=40, H=8, d=128):
    q, qs = inputs.quantize_fp8_rows(inputs.randn((H, d), seed, "pq"))
    k, ks = inputs.quantize_fp8_rows(inputs.randn((n, d), seed, "pk"))
    w = inputs.rand((H,), seed, "pw").numpy().astype(np.float64)
    return q.numpy(), qs.numpy().astype(np.float64), k.numpy(), ks.numpy().astype(np.float64), w


def test_indexer_fp8_dot_is_exact_integer_arithmetic():
    # every e4m3 value times 2^9 is an integer, so <q,k> * 2^18 is an exact integer sum
    q8, _, k8, _, _ = _fp8_case(1)
    qi = np.rint(O.decode_e4m3(q8) * 2 ** 9).astype(np.int64)
    ki = np.rint(O.decode_e4m3(k8) * 2 ** 9).astype(np.int64)
    exact = (ki @ qi.T)                                 # [n, H] integers
    for j in range(q8.shape[0]):
        w = np.zeros(q8.shape[0]); w[j] = 1.0           # one-hot weight picks ReLU(dot_j)
        got = O.index_scores(O.decode_e4m3(q8), w, O.decode_e4m3(k8), k8.shape[0] - 1)
        ref = np.array([max(int(v), 0) for v in exact[:, j]], dtype=np.float64) * 2.0 ** -18
        assert np.array_equal(got, ref)


def test_indexer_relu_identity_and_linearity():
    # ReLU(x) - ReLU(-x) = x, so I(q) - I(-q) = sum_j w_j sq_j sk_s <q_j, k_s> (one matmul)
    q8, qs, k8, ks, w = _fp8_case(2)
    qv, kv = O.decode_e4m3(q8), O.decode_e4m3(k8)
    n = kv.shape[0]
    lin = ((kv @ qv.T) * qs[None, :] * ks[:, None]) @ w
    diff = O.index_scores(qv, w, kv, n - 1, qs, ks) - O.index_scores(-qv, w, kv, n - 1, qs, ks)
    np.testing.assert_allclose(diff, lin, rtol=1e-12, atol=1e-12)
    # w >= 0 -> I >= 0;  w = 0 -> 0;  2w -> exactly 2I
    base = O.index_scores(qv, w, kv, n - 1, qs, ks)
    assert np.all(base >= 0)
    assert np.all(O.index_scores(qv, 0 * w, kv, n - 1, qs, ks) == 0)
    assert np.array_equal(O.index_scores(qv, 2 * w, kv, n - 1, qs, ks), 2 * base)
    # causal bound: pos p returns exactly p+1 scores equal to the prefix of the full row
    assert np.array_equal(O.index_scores(qv, w, kv, 9, qs, ks), base[:10])


def test_indexer_single_head_is_plain_dot():
    rng = np.random.default_rng(0)
    q = np.abs(rng.standard_normal((1, 16)))
    k = np.abs(rng.standard_normal((5, 16)))
    got = O.index_scores(q, np.array([1.0]), k, 4)
    np.testing.assert_allclose(got, [float(np.dot(q[0], r)) for r in k], rtol=1e-15)


# --------------------------------------------------------------------------- top-k

def test_topk_hand_cases():
    for c in _load("topk_hand.json")["cases"]:
        got = O.topk_select(np.array(c["scores"], dtype=np.float64), c["k"])
        assert got.tolist() == c["expected"], c["note"]


def _unique_valid_subset(scores, k):
    """Brute force: the only k-subset whose every member outranks every
    non-member under (score desc, position asc)."""
    n = len(scores)
    m = min(k, n)
    found = []
    for sub in itertools.combinations(range(n), m):
        rest = [s for s in range(n) if s not in sub]
        ok = all((scores[a] > scores[b]) or (scores[a] == scores[b] and a < b)
                 for a in sub for b in rest)
        if ok:
            found.append(list(sub))
    assert len(found) == 1
    return found[0] + [-1] * (k - m)


def test_topk_brute_force_small():
    rng = np.random.default_rng(3)
    for trial in range(60):
        n = int(rng.integers(1, 10))
        k = int(rng.integers(1, 11))
        scores = rng.integers(-2, 3, size=n).astype(np.float64)   # many ties
        if trial % 3 == 0:
            scores = rng.standard_normal(n)
        assert O.topk_select(scores, k).tolist() == _unique_valid_subset(scores.tolist(), k)


def test_topk_matches_torch_topk_on_distinct_scores():
    x = torch.randperm(5000, generator=torch.Generator().manual_seed(5)).to(torch.float64)
    got = O.topk_select(x.numpy(), 700)
    ref = torch.topk(x, 700).indices.sort().values.numpy()
    assert np.array_equal(got, ref)


def test_topk_all_equal_takes_lowest_positions():
    assert np.array_equal(O.topk_select(np.ones(100), 17), np.arange(17))


# --------------------------------------------------------------------------- attention

def test_attention_hand_cases():
    for c in _load("attention_hand.json")["cases"]:
        o, lse = O.sparse_attention(np.array(c["q"]), np.array(c["kv"]), c["scale"], c["d_v"])
        np.testing.assert_allclose(o, c["expected_O"], rtol=0, atol=1e-15)
        np.testing.assert_allclose(lse, c["expected_LSE"], rtol=0, atol=1e-15)


def test_attention_special_cases():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((6, 24))
    kv = rng.standard_normal((9, 24))
    # one selected row -> O is exactly that row's value part, LSE its logit
    o, lse = O.sparse_attention(q, kv[3:4], 0.7, 16)
    assert np.array_equal(o, np.repeat(kv[3:4, :16], 6, axis=0))
    np.testing.assert_allclose(lse, 0.7 * q @ kv[3], rtol=1e-15)
    # q = 0 -> uniform weights: O = mean of the selected value rows, LSE = ln n
    o, lse = O.sparse_attention(np.zeros((2, 24)), kv, 0.3, 20)
    np.testing.assert_allclose(o, np.repeat(kv[:, :20].mean(0, keepdims=True), 2, 0), atol=1e-15)
    np.testing.assert_allclose(lse, np.log(9.0), rtol=1e-15)
    # order of the selected rows does not matter; the softmax weights sum to one
    o1, l1 = O.sparse_attention(q, kv, 0.2, 24)
    perm = rng.permutation(9)
    o2, l2 = O.sparse_attention(q, kv[perm], 0.2, 24)
    np.testing.assert_allclose(o1, o2, atol=1e-14)
    np.testing.assert_allclose(l1, l2, atol=1e-14)
    p = np.exp(0.2 * q @ kv.T - l1[:, None])
    np.testing.assert_allclose(p.sum(1), 1.0, atol=1e-14)
    np.testing.assert_allclose(p @ kv, o1, atol=1e-14)     # O is the p-weighted row sum
    # no selected rows: O = 0, LSE = -inf
    o, lse = O.sparse_attention(q, kv[:0], 0.2, 24)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def _sdpa_causal(q, kv, scale, d_v):
    """torch scaled_dot_product_attention (float64, CPU) with the shared KV row
    broadcast to every head: the textbook dense causal softmax attention."""
    qt = torch.from_numpy(q).permute(1, 0, 2).unsqueeze(0)            # [1, H, T, d]
    H = q.shape[1]
    k = torch.from_numpy(kv).unsqueeze(0).unsqueeze(0).expand(1, H, -1, -1)
    v = k[..., :d_v]
    o = torch.nn.functional.scaled_dot_product_attention(qt, k, v, is_causal=True, scale=scale)
    return o[0].permute(1, 0, 2).numpy()


def test_dense_mqa_matches_torch_sdpa():
    rng = np.random.default_rng(6)
    T, H, d, dv = 37, 3, 20, 12
    q = rng.standard_normal((T, H, d))
    kv = rng.standard_normal((T, d))
    o, _ = O.dense_causal_mqa(q, kv, np.arange(T), 0.4, dv)
    np.testing.assert_allclose(o, _sdpa_causal(q, kv, 0.4, dv), atol=1e-12)


def test_dsa_with_k_at_least_L_is_dense_causal_mqa():
    # when every causal key is selected, DSA must equal dense causal MQA
    wl = inputs.make_tiny(seed=0, L=96, topk=96)
    from oracle.workload_view import OracleView
    v = OracleView(wl)
    q = wl.q.numpy().astype(np.float64)
    kv = wl.kv.numpy().astype(np.float64)
    ref = _sdpa_causal(q, kv, wl.softmax_scale, wl.d_v)
    for i in range(wl.num_q):
        _, idx, o, _ = v.run(i)
        assert np.array_equal(idx[:i + 1], np.arange(i + 1)) and np.all(idx[i + 1:] == -1)
        np.testing.assert_allclose(o, ref[i], atol=1e-12)


def test_dsa_rows_before_k_equal_dense():
    # with k = 32, every query t < 32 has t+1 <= k candidates -> dense
    wl = inputs.make_tiny(seed=1, L=64, topk=32)
    from oracle.workload_view import OracleView
    v = OracleView(wl)
    ref = _sdpa_causal(wl.q.numpy().astype(np.float64), wl.kv.numpy().astype(np.float64),
                       wl.softmax_scale, wl.d_v)
    for i in range(32):
        _, _, o, _ = v.run(i)
        np.testing.assert_allclose(o, ref[i], atol=1e-12)
    # later rows select exactly k distinct causal positions
    for i in range(32, 64):
        _, idx, _, _ = v.run(i)
        assert len(set(idx.tolist())) == 32 and idx.min() >= 0 and idx.max() <= i


def _hand_paged_workload():
    """A paged cache written out by hand: block size 4, three sequences of 6,
    9 and 3 positions, block table [[4, 1], [0, 5, 2], [3, 0]] (the last 0 is
    padding past sequence 2's one block).  Row r of every cache tensor holds
    the value r, so a decoded logical cache shows which physical row it read."""
    bt = torch.tensor([[4, 1, 0], [0, 5, 2], [3, 0, 0]], dtype=torch.int32)
    rows = 6 * 4
    col = torch.arange(rows, dtype=torch.float32)[:, None]
    q_seq = torch.tensor([0, 1, 2], dtype=torch.int32)
    q_pos = torch.tensor([5, 8, 2], dtype=torch.int32)
    return inputs.Workload(
        name="hand_paged", seed=0, idx_dtype="f32", H_I=1, d_I=4,
        q_idx=torch.ones((3, 1, 4)), q_scale=None, w=torch.ones((3, 1)),
        k_idx=col.repeat(1, 4), k_scale=None, topk=4, attn_dtype="f32", H=8, d_qk=4, d_v=4,
        q=torch.zeros((3, 8, 4)), kv=col.repeat(1, 4) + 0.5, softmax_scale=0.5,
        q_seq=q_seq, q_pos=q_pos, seq_lens=[6, 9, 3], seq_stride=0,
        block_table=bt, block_size=4, chunks=[(0, 3)])


def test_paged_row_map_walked_by_hand():
    # row(b, s) = block_table[b][s // 4] * 4 + s % 4, each value typed out
    wl = _hand_paged_workload()
    want = {
        0: [16, 17, 18, 19, 4, 5],                       # blocks 4, 1
        1: [0, 1, 2, 3, 20, 21, 22, 23, 8],              # blocks 0, 5, 2
        2: [12, 13, 14],                                 # block 3
    }
    for b, rows in want.items():
        assert wl.logical_rows(b, len(rows)).tolist() == rows, b
    from oracle.workload_view import OracleView
    view = OracleView(wl)
    for b, rows in want.items():
        k_vals, k_scale, kv = view.seq_cache(b, len(rows))
        assert k_scale is None
        assert k_vals[:, 0].tolist() == [float(r) for r in rows], b
        assert kv[:, 0].tolist() == [r + 0.5 for r in rows], b


def test_paged_view_reads_logical_rows():
    # the mixed workload's block table maps its sequences onto disjoint
    # physical blocks that together are a permutation of the pool
    wl = inputs.make_mixed(seed=0, batch=3, lo=200, hi=300, prefill=40, decode=4, block=16, topk=16)
    nblk = [(c + 15) // 16 for c in wl.seq_lens]
    used = torch.cat([wl.block_table[b, :n] for b, n in enumerate(nblk)])
    assert sorted(used.tolist()) == list(range(sum(nblk)))
    assert wl.num_rows == sum(nblk) * 16
    rows = torch.cat([wl.logical_rows(b, c) for b, c in enumerate(wl.seq_lens)])
    assert rows.unique().numel() == rows.numel()            # no two logical rows share storage
    assert int(rows.max()) < wl.num_rows


# --------------------------------------------------------------------------- indexer training (KL alignment)

def _kl_case(seed, H=6, d=16, n=40, kk=24, fp8=False):
    rng = np.random.default_rng(seed)
    if fp8:
        q, qs = O.quantize_e4m3_rows(rng.standard_normal((H, d)).astype(np.float32))
        kr, ks = O.quantize_e4m3_rows(rng.standard_normal((n, d)).astype(np.float32))
        q, kr = O.decode_e4m3(q), O.decode_e4m3(kr)
    else:
        q, qs, kr, ks = rng.standard_normal((H, d)), None, rng.standard_normal((n, d)), None
    w = rng.standard_normal(H)
    sel = np.sort(rng.choice(n, kk - 3, replace=False))
    sel = np.concatenate([sel, [-1, -1, -1]])
    p = rng.random(kk) ** 3
    p[sel < 0] = 0
    p /= p.sum()
    return q, qs, w, kr, ks, sel, p


@pytest.mark.parametrize("fp8", [False, True])
def test_indexer_kl_backward_matches_autograd(fp8):
    q, qs, w, kr, ks, sel, p = _kl_case(1 + fp8, fp8=fp8)
    r = O.indexer_kl_backward(q, w, kr, sel, p, qs, ks)
    qd = q * (qs[:, None] if qs is not None else 1.0)
    kd = kr * (ks[:, None] if ks is not None else 1.0)
    qt = torch.tensor(qd, requires_grad=True)
    wt = torch.tensor(w, requires_grad=True)
    kt = torch.tensor(kd, requires_grad=True)
    v = sel >= 0
    x = qt @ kt[torch.tensor(sel[v])].T
    lp = torch.log_softmax(wt @ torch.relu(x), 0)
    pt = torch.tensor(p[v])
    loss = (pt * (torch.log(pt) - lp)).sum()
    loss.backward()
    assert abs(loss.item() - r["loss"]) < 1e-12
    np.testing.assert_allclose(r["dw"], wt.grad.numpy(), rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(r["dq"], qt.grad.numpy(), rtol=1e-10, atol=1e-13)
    dk = np.zeros_like(kd)
    for row, s in enumerate(sel):
        if s >= 0:
            dk[s] += r["dk"][row]
    np.testing.assert_allclose(dk, kt.grad.numpy(), rtol=1e-10, atol=1e-13)
    assert np.all(r["dk"][~v] == 0) and np.all(r["g"][~v] == 0)


def test_indexer_kl_loss_and_finite_differences():
    q, _, w, kr, _, sel, p = _kl_case(3)
    v = sel >= 0
    r = O.indexer_kl_backward(q, w, kr, sel, p)
    assert abs(O.indexer_kl_loss(q, w, kr[sel[v]], p[v]) - r["loss"]) < 1e-12
    h = 1e-6
    for j in range(len(w)):
        wp, wm = w.copy(), w.copy()
        wp[j] += h
        wm[j] -= h
        fd = (O.indexer_kl_loss(q, wp, kr[sel[v]], p[v]) - O.indexer_kl_loss(q, wm, kr[sel[v]], p[v])) / (2 * h)
        assert abs(fd - r["dw"][j]) < 1e-6 * max(1.0, abs(fd))
    for (j, c) in [(0, 3), (2, 7), (5, 15)]:
        qp, qm = q.copy(), q.copy()
        qp[j, c] += h
        qm[j, c] -= h
        fd = (O.indexer_kl_loss(qp, w, kr[sel[v]], p[v]) - O.indexer_kl_loss(qm, w, kr[sel[v]], p[v])) / (2 * h)
        assert abs(fd - r["dq"][j, c]) < 1e-6 * max(1.0, abs(fd))


def test_indexer_kl_special_cases():
    q, _, w, kr, _, sel, p = _kl_case(4)
    v = sel >= 0
    # p = softmax(I): zero loss and zero gradients
    I = w @ np.maximum(q @ kr[sel[v]].T, 0)
    pi = np.zeros(len(sel))
    pi[v] = np.exp(I - I.max()) / np.exp(I - I.max()).sum()
    r = O.indexer_kl_backward(q, w, kr, sel, pi)
    assert abs(r["loss"]) < 1e-12 and np.abs(r["dw"]).max() < 1e-12 and np.abs(r["dq"]).max() < 1e-12
    # one candidate: pi = p = 1
    one = np.array([5, -1, -1])
    r = O.indexer_kl_backward(q, w, kr, one, np.array([1.0, 0, 0]))
    assert r["loss"] == 0 and np.all(r["dw"] == 0) and np.all(r["dq"] == 0) and np.all(r["dk"] == 0)
    # w = 0: pi uniform, no gradient reaches q or k, dw_j = sum (1/n - p_s) ReLU(x_js)
    r = O.indexer_kl_backward(q, np.zeros_like(w), kr, sel, p)
    n = int(v.sum())
    assert np.all(r["dq"] == 0) and np.all(r["dk"] == 0)
    np.testing.assert_allclose(r["dw"], np.maximum(q @ kr[sel[v]].T, 0) @ (1.0 / n - p[v]), rtol=1e-12)
    # an exactly-zero code dot is not a positive one, whatever the scales (ReLU'(0) = 0)
    qz, kz = np.array([[1.0, 1.0, 0.0]]), np.array([[1.0, -1.0, 0.5], [1.0, 1.0, 0.0]])
    r = O.indexer_kl_backward(qz, np.array([1.0]), kz, np.array([0, 1]), np.array([0.5, 0.5]),
                              np.array([0.37]), np.array([0.11, 0.13]))
    assert np.all(r["dk"][0] == 0) and np.any(r["dk"][1] != 0)
    # KL >= 0
    for s in range(5):
        qq, _, ww, kk_, _, ss, pp = _kl_case(10 + s)
        assert O.indexer_kl_backward(qq, ww, kk_, ss, pp)["loss"] >= 0


# --------------------------------------------------------------------------- per-head (prefill) attention mode

def _latent_mha(seed, n, H=4, dl=24, dr=8, dn=6, dv=5):
    """Latent rows c (dl latent + dr rope), per-head up-projections W_K, W_V,
    the per-head keys and values they give, and a query."""
    rng = np.random.default_rng(seed)
    c = rng.standard_normal((n, dl + dr))
    WK = rng.standard_normal((H, dn, dl))
    WV = rng.standard_normal((H, dv, dl))
    qn, qr = rng.standard_normal((H, dn)), rng.standard_normal((H, dr))
    k_nope = np.einsum("hdl,nl->nhd", WK, c[:, :dl])
    v = np.einsum("hdl,nl->nhd", WV, c[:, :dl])
    return c, WK, WV, qn, qr, k_nope, c[:, dl:], v


def test_mha_mode_equals_absorbed_latent_mqa():
    """The two attention modes are one attention: with per-head keys and
    values that are up-projections of latent rows (k_nope = W_K c,
    v = W_V c, the rope part shared), per-head attention equals the latent MQA
    of sparse_attention with the absorbed query (W_K^T q_nope, q_rope), its
    output up-projected by W_V, and the two LSEs agree."""
    dl = 24
    c, WK, WV, qn, qr, k_nope, k_rope, v = _latent_mha(41, n=37, dl=dl)
    o, lse = O.sparse_attention_mha(np.concatenate([qn, qr], 1), k_nope, k_rope, v, 0.3)
    q_abs = np.concatenate([np.einsum("hdl,hd->hl", WK, qn), qr], 1)
    o_lat, lse_lat = O.sparse_attention(q_abs, c, 0.3, dl)           # the value: the latent part
    np.testing.assert_allclose(lse, lse_lat, rtol=0, atol=1e-11)
    np.testing.assert_allclose(o, np.einsum("hdl,hl->hd", WV, o_lat), rtol=0, atol=1e-11)


def test_mha_mode_dense_causal_matches_torch_sdpa():
    rng = np.random.default_rng(42)
    T, H, dn, dr, dv = 13, 3, 6, 4, 5
    q = rng.standard_normal((T, H, dn + dr))
    k_nope, k_rope, v = rng.standard_normal((T, H, dn)), rng.standard_normal((T, dr)), rng.standard_normal((T, H, dv))
    kh = np.concatenate([k_nope, np.broadcast_to(k_rope[:, None, :], (T, H, dr))], 2)   # each head's full key
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q).permute(1, 0, 2), torch.tensor(kh).permute(1, 0, 2), torch.tensor(v).permute(1, 0, 2),
        is_causal=True, scale=0.45).permute(1, 0, 2).numpy()
    for t in range(T):
        o, _ = O.sparse_attention_mha(q[t], k_nope[:t + 1], k_rope[:t + 1], v[:t + 1], 0.45)
        np.testing.assert_allclose(o, ref[t], rtol=0, atol=1e-12)


def test_mha_mode_special_cases():
    _, _, _, qn, qr, k_nope, k_rope, v = _latent_mha(43, n=9)
    q = np.concatenate([qn, qr], 1)
    o, lse = O.sparse_attention_mha(q, k_nope[4:5], k_rope[4:5], v[4:5], 0.7)     # one key: its value row
    np.testing.assert_allclose(o, v[4], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, 0.7 * (np.einsum("hd,hd->h", qn, k_nope[4]) + qr @ k_rope[4]), atol=1e-12)
    o0, l0 = O.sparse_attention_mha(q, k_nope[:0], k_rope[:0], v[:0], 0.7)        # no key
    assert np.all(o0 == 0) and np.all(np.isneginf(l0))
    perm = np.random.default_rng(0).permutation(9)                                   # order of the keys is irrelevant
    o1, l1 = O.sparse_attention_mha(q, k_nope, k_rope, v, 0.7)
    o2, l2 = O.sparse_attention_mha(q, k_nope[perm], k_rope[perm], v[perm], 0.7)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)
