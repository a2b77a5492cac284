"""CPU oracle for the DeepSeek Sparse Attention (DSA) hot path.

TEST INFRASTRUCTURE ONLY.  This module is the slow, plain, float64 statement
of what the GPU library computes.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import it; the library itself never does,
and it never imports the library.

Sources (web pages about DeepSeek-V3.2):
  * "DeepSeek-V3.2: Pushing the Frontier of Open Large Language Models"
    summary card, section "How DSA Works": a lightning indexer computes cheap
    FP8 relevance scores between a query and all keys, a top-k step keeps the
    2048 most relevant tokens, and full attention runs only on those tokens.
  * "DeepSeek researchers announce DeepSeek-V3.2 and DeepSeek-V3.2-Speciale ..."
    (news article), section on sparse attention with near-linear long-context
    cost: the indexer runs a few low-precision heads on every token pair; the
    fine-grained selector keeps the top-k key/value positions per query; the
    main path runs multi-query / multi-head latent attention on that sparse
    set.  Section on continued pre-training: the selector keeps 2048 entries
    per query.
  * "Deepseek V3.2 Frontier" summary, section "Implementation": a sketch
    score -> top-k -> gather -> softmax.  Its use of the indexer score as the
    attention logit is NOT followed (the news article's section says the main
    path runs MQA/MLA attention over the selected set).

The pages give no formula; this library fixes the indexer as
    I[t,s] = sum_j w[t,j] * ReLU(sq[t,j] * sk[s] * <q8[t,j,:], k8[s,:]>)
with FP8 e4m3 codes q8/k8 and positive per-row fp32 scales sq/sk (or plain
fp32 vectors and no scales), keys s <= t (causal, inclusive);
top-k = the min(k, t+1) largest I[t,s], ties to the lower s, returned in
ascending s and padded with -1; attention
    O[t,h,:] = sum_{s in sel} softmax_s(tau * <q[t,h,:], kv[s,:]>) * kv[s,:d_v]
plus LSE[t,h] = log sum_s exp(tau * <q, kv_s>) (natural log).  For training,
the indexer's alignment loss KL(p || softmax(I)) over a query's candidate
set and its gradients (indexer_kl_backward).

Everything is computed in float64 from exactly decoded inputs, except the
key-cache encoding (quantize_e4m3_rows): the FP8 keys of the summary card's
"cheap FP8 relevance scores" are written once per token as e4m3 codes with a
per-row scale amax/448, and the codes that write produces are decided by its
float32 scale and division, which the oracle therefore takes in float32.

FP8 latent KV cache (an optional storage format of the attention cache; the
pages name no KV format, so this library reuses the key-cache encoding for
it): each 576-wide latent row is stored as e4m3 codes with one fp32 scale,
and the attention reads row s as bf16(scale_s * code_s), the product taken in
float32 and rounded once to bfloat16 (dequantize_kv_e4m3).  The attention
itself is then the bf16 one above, on those values.
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# Exact decoders for the input encodings
# ---------------------------------------------------------------------------


def _e4m3_value(code: int) -> float:
    """OCP 8-bit float E4M3 ("fn" variant): 1 sign, 4 exponent (bias 7),
    3 mantissa bits; exponent field 0 is subnormal (m/8 * 2^-6); S.1111.111
    is NaN; there are no infinities, so S.1111.000-110 are normal numbers up
    to 448."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)


def decode_e4m3(codes) -> np.ndarray:
    """uint8 e4m3 codes -> float64 values (exact)."""
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


# Positive finite codes 0x00..0x7E in increasing order of value (the code is
# the index: e4m3 codes are monotonic in magnitude).
_E4M3_POS = E4M3_TABLE[:0x7F]


def encode_e4m3(y) -> np.ndarray:
    """Float values -> OCP e4m3 ("fn") codes: round to the nearest
    representable value, ties to the code with an even last mantissa bit,
    magnitudes above 448 saturated to 448; the sign bit is kept (-0.0 ->
    0x80).  The inputs are taken exactly as given (float32 values are exact
    in float64)."""
    y = np.asarray(y, dtype=np.float64)
    a = np.minimum(np.abs(y), 448.0)
    hi = np.searchsorted(_E4M3_POS, a, side="left")          # first code with value >= a
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _E4M3_POS[lo]
    d_hi = _E4M3_POS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a == _E4M3_POS[hi], hi, code)             # exactly representable
    return (code | np.where(np.signbit(y), 0x80, 0)).astype(np.uint8)


def quantize_e4m3_rows(x) -> tuple:
    """Indexer key-cache encoding of float32 rows (x [n, d]): per row
    scale = amax(|row|) / 448 (1 for an all-zero row) and codes =
    encode_e4m3(row / scale), the scale and the division taken in float32
    -- the precision of the kernel that writes the cache, which decides the
    codes.  Returns (uint8 codes [n, d], float32 scales [n])."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.abs(x).max(axis=1)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    y = (x / scale[:, None]).astype(np.float32)
    return encode_e4m3(y), scale


def round_bf16(x) -> np.ndarray:
    """float32 values -> the nearest bfloat16 value (ties to the even bit
    pattern), as float64.  bf16 keeps the top 16 bits of a binary32, so the
    rounding adds half a unit of the dropped 16 bits, plus one when the kept
    part is odd, and truncates.  Inputs are finite."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) & np.uint64(0xFFFF0000)
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def dequantize_kv_e4m3(codes, scale) -> np.ndarray:
    """FP8 latent rows -> the bf16 values the attention reads:
    bf16(float32(scale[r]) * float32(e4m3 value of codes[r, d])).
    codes [n, d] uint8, scale [n] float32; returns float64 [n, d]."""
    v = decode_e4m3(codes).astype(np.float32)                    # exact: e4m3 values fit float32
    prod = (np.asarray(scale, dtype=np.float32)[:, None] * v).astype(np.float32)
    return round_bf16(prod)


def decode_bf16(bits) -> np.ndarray:
    """uint16 bfloat16 bit patterns -> float64 values (exact: bf16 is the top
    half of an IEEE binary32)."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# Stage 1: lightning indexer
# ---------------------------------------------------------------------------


def index_scores(q_vals, w, k_vals, pos, q_scale=None, k_scale=None) -> np.ndarray:
    """Indexer scores of ONE query against keys 0..pos.

    q_vals [H_I, d_I] and k_vals [>pos, d_I] are decoded float64 values;
    q_scale [H_I] and k_scale [>pos] the positive per-row dequantisation
    scales (None = 1).  Returns I[s] for s = 0..pos (float64, length pos+1):
        I[s] = sum_j w[j] * max(0, sq[j] * sk[s] * <q[j], k[s]>)
    The inner product of two e4m3 rows is exact in float64 (every product has
    at most 8 significant bits and the partial sums stay below 2^53 units of
    the smallest product), so the only roundings are the scale products, the
    ReLU-weighted head sum and nothing else.
    """
    n = int(pos) + 1
    k = np.asarray(k_vals[:n], dtype=np.float64)
    q = np.asarray(q_vals, dtype=np.float64)
    dots = k @ q.T                                   # [n, H_I]: <q[j], k[s]>
    if q_scale is not None:
        dots = dots * np.asarray(q_scale, dtype=np.float64)[None, :]
    if k_scale is not None:
        dots = dots * np.asarray(k_scale[:n], dtype=np.float64)[:, None]
    # head sum row by row (a per-row reduction, so a score does not depend on
    # how many other keys are scored in the same call)
    return (np.maximum(dots, 0.0) * np.asarray(w, dtype=np.float64)[None, :]).sum(axis=1)


# ---------------------------------------------------------------------------
# Stage 2: per-query top-k selection
# ---------------------------------------------------------------------------


def topk_select(scores, k: int) -> np.ndarray:
    """Top-k of one score row over candidates 0..len-1.

    Candidates are ranked by (score descending, position ascending), so among
    equal scores the lower position wins (+0 and -0 compare equal).  The first
    min(k, n) of that ranking are returned in ascending position order,
    padded with -1 to length k (int32).
    """
    s = np.asarray(scores, dtype=np.float64)
    n = s.shape[0]
    order = np.lexsort((np.arange(n), -s))           # primary: -score, secondary: position
    keep = np.sort(order[:min(k, n)])
    out = np.full(k, -1, dtype=np.int32)
    out[:keep.shape[0]] = keep
    return out


# ---------------------------------------------------------------------------
# Stage 3: attention over the selected entries (MQA over one shared KV row)
# ---------------------------------------------------------------------------


def sparse_attention(q, kv_rows, scale: float, d_v: int):
    """Softmax attention of H query heads over n selected KV rows.

    q [H, d_qk] and kv_rows [n, d_qk] float64; the value of a row is its first
    d_v entries.  Returns (O [H, d_v], LSE [H]).  With n = 0, O = 0 and
    LSE = -inf.
    """
    q = np.asarray(q, dtype=np.float64)
    kv = np.asarray(kv_rows, dtype=np.float64)
    H = q.shape[0]
    if kv.shape[0] == 0:
        return np.zeros((H, d_v)), np.full(H, -np.inf)
    logits = scale * (q @ kv.T)                      # [H, n]
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    l = p.sum(axis=1, keepdims=True)
    o = (p @ kv[:, :d_v]) / l
    return o, (m + np.log(l))[:, 0]


def dense_causal_mqa(q, kv, q_pos, scale: float, d_v: int):
    """Dense causal MQA: query i (position q_pos[i]) attends to KV rows
    0..q_pos[i].  q [T, H, d_qk], kv [S, d_qk].  Returns (O [T,H,d_v], LSE [T,H])."""
    T, H, _ = q.shape
    O = np.zeros((T, H, d_v))
    LSE = np.zeros((T, H))
    for i in range(T):
        p = int(q_pos[i])
        O[i], LSE[i] = sparse_attention(q[i], kv[:p + 1], scale, d_v)
    return O, LSE


# ---------------------------------------------------------------------------
# Per-head attention over the selected entries (the prefill attention mode)
# ---------------------------------------------------------------------------


def sparse_attention_mha(q, k_nope, k_rope, v, scale: float):
    """Softmax attention of H query heads over n selected keys, each head with
    its own key and value rows: the per-head (non-absorbed) form of
    multi-head latent attention.  Susan Zhang's thread on the DeepSeek-V3.2
    write-up names separate attention modes for disaggregated prefill and
    decode; this is the prefill one, the latent MQA of sparse_attention the
    decode one.  A head's key is its own d_nope-wide part followed by the
    d_rope-wide part that all heads share.

    q [H, d_nope + d_rope], k_nope [n, H, d_nope], k_rope [n, d_rope],
    v [n, H, d_v] float64.  Returns (O [H, d_v], LSE [H]); n = 0 gives
    O = 0 and LSE = -inf.
    """
    q = np.asarray(q, dtype=np.float64)
    kn = np.asarray(k_nope, dtype=np.float64)
    kr = np.asarray(k_rope, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    H = q.shape[0]
    if kn.shape[0] == 0:
        return np.zeros((H, v.shape[2])), np.full(H, -np.inf)
    dn = kn.shape[2]
    logits = scale * (np.einsum("hd,nhd->hn", q[:, :dn], kn) + q[:, dn:] @ kr.T)   # [H, n]
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    l = p.sum(axis=1, keepdims=True)
    o = np.einsum("hn,nhd->hd", p, v) / l
    return o, (m + np.log(l))[:, 0]


# ---------------------------------------------------------------------------
# The whole hot path for a set of queries
# ---------------------------------------------------------------------------


def dsa_query(q_idx_vals, q_scale, w, k_vals, k_scale, pos, topk, q_attn, kv_vals, scale, d_v):
    """indexer -> top-k -> sparse attention for ONE query at position pos.

    All arrays hold decoded float64 values of one sequence in logical order
    (row s = position s).  Returns (scores [pos+1], idx [topk], O [H,d_v], LSE [H]).
    """
    sc = index_scores(q_idx_vals, w, k_vals, pos, q_scale, k_scale)
    idx = topk_select(sc, topk)
    sel = idx[idx >= 0]
    o, lse = sparse_attention(q_attn, kv_vals[sel], scale, d_v)
    return sc, idx, o, lse


# ---------------------------------------------------------------------------
# Indexer training: the alignment (KL) loss and its gradients
# ---------------------------------------------------------------------------


def indexer_kl_loss(q, w, k_sel, p) -> float:
    """KL(p || softmax(I)) for ONE query over its candidate set, straight from
    the definitions (used to pin the gradients by finite differences).
    q [H, d] and k_sel [n, d] dequantised values, w [H], p [n] (sums to 1)."""
    x = np.asarray(q, dtype=np.float64) @ np.asarray(k_sel, dtype=np.float64).T     # [H, n]
    I = np.asarray(w, dtype=np.float64) @ np.maximum(x, 0.0)                       # [n]
    log_pi = I - I.max() - np.log(np.exp(I - I.max()).sum())
    p = np.asarray(p, dtype=np.float64)
    nz = p > 0
    return float((p[nz] * (np.log(p[nz]) - log_pi[nz])).sum())


def indexer_kl_backward(q_vals, w, k_rows, sel, p, q_scale=None, k_scale=None) -> dict:
    """Indexer alignment loss of ONE query and its gradients.

    The news article's continued-pre-training section: the indexer is trained
    with a Kullback-Leibler loss to match the main attention's distribution --
    over all keys in the dense warm-up, over the selected set only in the
    sparse phase, where the indexer's gradients come from that loss alone.
    With the candidate set S (the valid entries of sel), a target
    distribution p over S, the dequantised operands q_j = sq_j * q_vals[j]
    and k_s = sk_s * k_rows[s], and x_js = <q_j, k_s>:
        I_s  = sum_j w_j ReLU(x_js)
        pi   = softmax over S of I
        loss = sum_{s in S} p_s (log p_s - log pi_s)            (0 log 0 = 0)
        g_s  = d loss / d I_s = pi_s - p_s
        dw_j = sum_s g_s ReLU(x_js)
        dq_j = sum_s g_s w_j [x_js > 0] k_s
        dk_s = g_s sum_j w_j [x_js > 0] q_j
    (ReLU'(0) = 0).  The gradients are with respect to the dequantised q, w
    and k.

    q_vals [H, d], w [H], k_rows [n, d] (logical rows 0..n-1 of the
    sequence), sel [k] positions with -1 padding, p [k] aligned with sel
    (ignored where sel = -1); q_scale [H] and k_scale [n] or None.  Returns a
    dict with loss, g [k], dw [H], dq [H, d], dk [k, d] (row r belongs to
    sel[r]; zero at padding) and mag_dw, mag_dq, mag_dk: the same sums taken
    over absolute values with |g_s| widened by 1e-4 (pi_s + p_s), the scale of
    the rounding a float32 evaluation of g can carry."""
    q8 = np.asarray(q_vals, dtype=np.float64)
    sq = np.ones(q8.shape[0]) if q_scale is None else np.asarray(q_scale, dtype=np.float64)
    q = q8 * sq[:, None]
    w = np.asarray(w, dtype=np.float64)
    sel = np.asarray(sel)
    valid = sel >= 0
    k8 = np.asarray(k_rows, dtype=np.float64)[sel[valid]]
    sk = np.ones(k8.shape[0]) if k_scale is None else np.asarray(k_scale, dtype=np.float64)[sel[valid]]
    ks = k8 * sk[:, None]
    pv = np.asarray(p, dtype=np.float64)[valid]
    H, d = q.shape
    kk = sel.shape[0]
    out = {"g": np.zeros(kk), "dk": np.zeros((kk, d)), "mag_dk": np.zeros((kk, d))}
    if ks.shape[0] == 0:
        out.update(loss=0.0, dw=np.zeros(H), dq=np.zeros((H, d)), mag_dw=np.zeros(H), mag_dq=np.zeros((H, d)))
        return out
    # the dot of the (decoded) operands first, then the scales, as in
    # ReLU(sq * sk * <q8, k8>): for e4m3 codes that dot is exact in float64,
    # so the sign deciding [x > 0] is exact (a dot of the scaled operands
    # would round, and can turn an exact 0 into +-1e-16)
    raw = q8 @ k8.T                               # [H, n]
    x = raw * sq[:, None] * sk[None, :]
    r = np.maximum(x, 0.0)
    m = (raw > 0).astype(np.float64)
    I = w @ r
    e = np.exp(I - I.max())
    pi = e / e.sum()
    log_pi = I - I.max() - np.log(e.sum())
    nz = pv > 0
    loss = float((pv[nz] * (np.log(pv[nz]) - log_pi[nz])).sum())
    g = pi - pv
    ga = np.abs(g) + 1e-4 * (pi + pv)
    wm = w[:, None] * m                           # [H, n]
    out["loss"] = loss
    out["g"][valid] = g
    out["dw"] = r @ g
    out["mag_dw"] = r @ ga
    out["dq"] = (wm * g[None, :]) @ ks
    out["mag_dq"] = (np.abs(wm) * ga[None, :]) @ np.abs(ks)
    out["dk"][valid] = g[:, None] * (wm.T @ q)
    out["mag_dk"][valid] = ga[:, None] * (np.abs(wm).T @ np.abs(q))
    return out
