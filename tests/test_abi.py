"""The C ABI without a GPU: the library loads, exports every entry point the
header declares, and its host-side validation rejects bad arguments before
touching the device."""
import ctypes
import os
import re

import pytest

from sparse_attention_long_11_b300 import api

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "dsa.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(dsa_\w+)\s*\(", src, flags=re.M)))


def test_library_exports_every_declared_symbol():
    names = _declared()
    assert "dsa_forward" in names and "dsa_topk" in names and len(names) >= 8
    L = api.lib()
    for n in names:
        assert hasattr(L, n), n
        assert n in api._SIGS, f"binding lacks {n}"


def test_status_strings_and_version():
    for s in range(7):
        assert api.status_string(s).startswith("DSA_")
    assert api.status_string(99) == "unknown dsa_status"
    assert api.dsa_version() >= 100


def _fake(addr=0x10000):
    return ctypes.c_void_p(addr)


def _ix(dtype=api.DSA_FP8_E4M3, heads=64, dim=128, scales=True, addr=0x10000):
    s = addr if scales else None
    return api.IndexerInputs(dtype, heads, dim, addr, s, addr, addr, s)


def _at(dtype=api.DSA_BF16, heads=128, d_qk=576, d_v=512, addr=0x10000, kv_scale=None):
    return api.AttnInputs(dtype, heads, d_qk, d_v, addr, addr, 0.04, kv_scale)


def test_workspace_size_validation():
    L = api.lib()
    qd = api.QueryDesc(16, 0x10000, 0x10000, 4096)
    ws = L.dsa_forward_workspace_size(ctypes.byref(qd), ctypes.byref(_ix()), 2048, ctypes.byref(_at()))
    assert ws >= 16 * 4096 * 4 and ws % 256 == 0
    # k out of range, unsupported shapes, bad dtypes -> 0
    assert L.dsa_forward_workspace_size(ctypes.byref(qd), ctypes.byref(_ix()), 8193, ctypes.byref(_at())) == 0
    assert L.dsa_forward_workspace_size(ctypes.byref(qd), ctypes.byref(_ix(heads=32)), 2048, ctypes.byref(_at())) == 0
    assert L.dsa_forward_workspace_size(ctypes.byref(qd), ctypes.byref(_ix()), 2048, ctypes.byref(_at(d_v=256))) == 0
    # staged scores are bounded (1 GiB) however many queries there are, and hold at least one row
    big = api.QueryDesc(1 << 20, 0x10000, 0x10000, 131072)
    assert 131072 * 4 <= L.dsa_forward_workspace_size(ctypes.byref(big), ctypes.byref(_ix()), 2048,
                                                       ctypes.byref(_at())) <= 1 << 30
    # 4 queries at a 2^22 context: one stage of all four rows, with a fallback score row for each
    huge = api.QueryDesc(4, 0x10000, 0x10000, 1 << 22)
    ws_huge = L.dsa_forward_workspace_size(ctypes.byref(huge), ctypes.byref(_ix()), 2048, ctypes.byref(_at()))
    assert ws_huge == L.dsa_forward_stage_workspace_size(ctypes.byref(huge), ctypes.byref(_ix()), 2048,
                                                         ctypes.byref(_at()), 4)
    assert ws_huge >= 4 << 24
    # per-stage sizes: more rows per stage need more bytes; below one row nothing
    st = lambda q, r, ix=None: L.dsa_forward_stage_workspace_size(ctypes.byref(q), ctypes.byref(ix or _ix()), 2048,
                                                                  ctypes.byref(_at()), r)
    assert 0 < st(qd, 1) < st(qd, 8) < st(qd, 16) == st(qd, 100)           # capped at the batch
    assert st(qd, 0) == 0 and st(qd, -3) == 0
    # the FP8 path keeps a candidate list per row, far less than a score row at long contexts
    long_q = api.QueryDesc(4096, 0x10000, 0x10000, 131072)
    assert st(long_q, 4096) - st(long_q, 2048) < 2048 * 131072 * 4 // 4
    # fp32 operands stage whole score rows
    f32 = _ix(dtype=api.DSA_F32, heads=4, dim=64, scales=False)
    assert st(qd, 3, f32) == 3 * 4096 * 4


@pytest.mark.parametrize("num_q,max_kv,k", [(4096, 32768, 2048), (4096, 131072, 2048), (4096, 4096, 2048),
                                             (64, 65536, 2048), (1000, 20000, 8192), (7, 3000, 100)])
def test_recommended_workspace_runs_one_stage(num_q, max_kv, k):
    """dsa_forward_workspace_size() holds the whole batch in one stage (below the 1 GiB cap), and a
    stage size's own workspace runs no more (equal) stages than stages of that many rows would."""
    qd = api.QueryDesc(num_q, 0x10000, 0x10000, max_kv)
    ix, at = _ix(), _at()
    ws = api.dsa_forward_workspace_size(qd, ix, k, at)
    assert ws > 0
    assert api.dsa_forward_stage_rows(qd, ix, k, at, ws) == num_q
    for r in sorted({1, 2, 3, num_q // 3 + 1, num_q - 1}):
        if 1 <= r <= num_q:
            rows = api.dsa_forward_stage_rows(qd, ix, k, at, api.dsa_forward_stage_workspace_size(qd, ix, k, at, r))
            assert rows > 0 and -(-num_q // rows) <= -(-num_q // r), (r, rows)   # no more stages than r-row ones
    least = api.dsa_forward_stage_workspace_size(qd, ix, k, at, 1)
    assert api.dsa_forward_stage_rows(qd, ix, k, at, least - 256) == 0
    # fp32 operands stage whole score rows: stages are equal and as large as the bytes allow
    f32 = _ix(dtype=api.DSA_F32, heads=4, dim=64, scales=False)
    row = ((max_kv + 3) // 4) * 16
    assert api.dsa_forward_stage_rows(qd, f32, k, at, 3 * row) == -(-num_q // -(-num_q // min(3, num_q)))


def test_host_validation_rejects_before_launch():
    L = api.lib()
    cd = api.CacheDesc(1, 4096, 4096, None, 0, 0)
    qd = api.QueryDesc(16, 0x10000, 0x10000, 4096)
    f = L.dsa_forward
    args = lambda q=qd, c=cd, ix=_ix(), k=2048, at=_at(), idx=0x10000, ws=0x10000, wsb=1 << 30: (
        ctypes.byref(q), ctypes.byref(c), ctypes.byref(ix), k, ctypes.byref(at), idx, 0x10000, 0x10000, ws, wsb, None)
    assert f(*args(k=0)) == api.DSA_ERR_INVALID_ARG
    assert f(*args(k=8193)) == api.DSA_ERR_INVALID_ARG
    assert f(*args(idx=None)) == api.DSA_ERR_INVALID_ARG
    assert f(*args(ix=_ix(scales=False))) == api.DSA_ERR_INVALID_ARG           # fp8 without scales
    assert f(*args(ix=_ix(addr=0x10004))) == api.DSA_ERR_INVALID_ARG           # misaligned operand
    assert f(*args(ix=_ix(dtype=api.DSA_BF16))) == api.DSA_ERR_UNSUPPORTED
    assert f(*args(at=_at(heads=64))) == api.DSA_ERR_UNSUPPORTED
    neg = _at()
    neg.softmax_scale = -0.04
    assert f(*args(at=neg)) == api.DSA_ERR_INVALID_ARG                        # tensor-core attention: scale > 0
    # FP8 latent cache: the per-row scales are required, 4-byte aligned, and only with that dtype
    assert f(*args(at=_at(dtype=api.DSA_FP8_E4M3))) == api.DSA_ERR_INVALID_ARG
    assert f(*args(at=_at(dtype=api.DSA_FP8_E4M3, kv_scale=0x10002))) == api.DSA_ERR_INVALID_ARG
    assert f(*args(at=_at(kv_scale=0x10000))) == api.DSA_ERR_INVALID_ARG
    assert f(*args(at=_at(dtype=api.DSA_FP8_E4M3, kv_scale=0x10000, d_v=256))) == api.DSA_ERR_UNSUPPORTED
    assert f(*args(ws=None)) == api.DSA_ERR_WORKSPACE
    assert f(*args(ws=0x10010)) == api.DSA_ERR_WORKSPACE                      # not 256-byte aligned
    assert f(*args(wsb=1024)) == api.DSA_ERR_WORKSPACE
    least = L.dsa_forward_stage_workspace_size(ctypes.byref(qd), ctypes.byref(_ix()), 2048, ctypes.byref(_at()), 1)
    assert f(*args(wsb=4096 * 4)) == api.DSA_ERR_WORKSPACE                    # one score row is not a stage
    assert least > 4096 * 4
    assert f(*args(wsb=least - 256)) == api.DSA_ERR_WORKSPACE                 # less than one stage of one row
    assert f(*args(q=api.QueryDesc(16, 0x10000, 0x10000, 0))) == api.DSA_ERR_INVALID_ARG
    assert f(*args(c=api.CacheDesc(2, 4096, 100, None, 0, 0))) == api.DSA_ERR_INVALID_ARG   # overlapping seqs
    assert f(*args(c=api.CacheDesc(1, 4096, 0, 0x10000, 64, 2))) == api.DSA_ERR_INVALID_ARG  # table too short
    # an empty batch is a no-op that never touches the device
    assert f(*args(q=api.QueryDesc(0, None, None, 0))) == api.DSA_OK
    # stage entry points
    assert L.dsa_topk(ctypes.byref(qd), 0x10000, 100, 2048, 0x10000, None) == api.DSA_ERR_INVALID_ARG  # ld < max_kv
    assert L.dsa_topk(ctypes.byref(qd), None, 4096, 2048, 0x10000, None) == api.DSA_ERR_INVALID_ARG
    assert L.dsa_index_scores(ctypes.byref(qd), ctypes.byref(cd), ctypes.byref(_ix()), 0x10000, 4094,
                              None) == api.DSA_ERR_INVALID_ARG
    assert L.dsa_sparse_attn(ctypes.byref(qd), ctypes.byref(cd), ctypes.byref(_at(dtype=7)), 0x10000, 2048,
                             0x10000, 0x10000, None) == api.DSA_ERR_UNSUPPORTED


def test_cache_append_validation_rejects_before_launch():
    L = api.lib()
    cd = api.CacheDesc(1, 4096, 4096, None, 0, 0)
    A = 0x10000
    f = lambda n=4, kdt=api.DSA_BF16, kn=A, dim=128, kc=A, ks=A, kvn=A, dqk=576, kvc=A, kvs=None, c=cd: \
        L.dsa_cache_append(ctypes.byref(c), n, A, A, kdt, kn, dim, kc, ks, kvn, dqk, kvc, kvs, None)
    assert f(n=0) == api.DSA_OK                                   # nothing to append: no launch
    assert f(n=-1) == api.DSA_ERR_INVALID_ARG
    assert f(dim=64) == api.DSA_ERR_UNSUPPORTED
    assert f(kdt=api.DSA_FP8_E4M3) == api.DSA_ERR_UNSUPPORTED
    assert f(kn=A + 8) == api.DSA_ERR_INVALID_ARG                 # key rows must be 16-byte aligned
    assert f(kc=None) == api.DSA_ERR_INVALID_ARG
    assert f(kvc=None) == api.DSA_ERR_INVALID_ARG                 # latent rows without a latent cache
    assert f(dqk=100) == api.DSA_ERR_UNSUPPORTED                  # 200-byte rows: not a 16-byte multiple
    assert f(c=api.CacheDesc(1, 4096, 0, A, 64, 0)) == api.DSA_ERR_INVALID_ARG   # empty block table
    # FP8 latent cache: scales only with latent rows, 4-byte aligned, rows of whole 16-byte chunks
    assert f(kvn=None, kvc=None, kvs=A) == api.DSA_ERR_INVALID_ARG
    assert f(kvs=A + 2) == api.DSA_ERR_INVALID_ARG
    assert f(kvs=A, dqk=72) == api.DSA_ERR_UNSUPPORTED


def test_indexer_kl_backward_validation_rejects_before_launch():
    L = api.lib()
    cd = api.CacheDesc(1, 4096, 4096, None, 0, 0)
    qd = api.QueryDesc(16, 0x10000, 0x10000, 4096)
    A = 0x10000
    f = lambda q=qd, ix=_ix(), idx=A, k=2048, p=A, loss=A, g=None, dw=A, dq=A, dk=A: L.dsa_indexer_kl_backward(
        ctypes.byref(q), ctypes.byref(cd), ctypes.byref(ix), idx, k, p, loss, g, dw, dq, dk, None)
    assert f(q=api.QueryDesc(0, None, None, 0)) == api.DSA_OK          # empty batch: no launch
    assert f(k=0) == api.DSA_ERR_INVALID_ARG and f(k=8193) == api.DSA_ERR_INVALID_ARG
    assert f(idx=None) == api.DSA_ERR_INVALID_ARG and f(dk=None) == api.DSA_ERR_INVALID_ARG
    assert f(dq=A + 4) == api.DSA_ERR_INVALID_ARG                      # dq and dk take float4 stores/atomics
    assert f(dk=A + 8) == api.DSA_ERR_INVALID_ARG
    assert f(ix=_ix(dtype=api.DSA_F32, scales=False, heads=80)) == api.DSA_ERR_UNSUPPORTED


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(api, "_lib", None)
    monkeypatch.setattr(api, "LIB_PATH", str(tmp_path / "libdsa.so"))
    with pytest.raises(RuntimeError, match="missing"):
        api.lib()


def test_wait_limit_entry_point_validates_on_the_host():
    L = api.lib()
    qd = api.QueryDesc(16, 0x10000, 0x10000, 4096)
    cd = api.CacheDesc(1, 4096, 4096, None, 0, 0)
    for limit in (0, -5):
        st = L.dsa_index_scores_wait_limit(ctypes.byref(qd), ctypes.byref(cd), ctypes.byref(_ix()), _fake(),
                                           4096, limit, None)
        assert st == api.DSA_ERR_INVALID_ARG
