"""Thin ctypes binding over libdsa.so (C ABI in include/dsa.h).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  Tensors are torch CUDA tensors (torch supplies
device memory and the current stream); each function has the name of the C
entry point it calls and raises ``DSAError`` on a non-OK status.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdsa.so")

DSA_OK, DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_CUDA, DSA_ERR_TIMEOUT, DSA_ERR_BOUNDS, \
    DSA_ERR_WORKSPACE = range(7)
DSA_F32, DSA_BF16, DSA_FP8_E4M3 = 0, 1, 2


class DSAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


class QueryDesc(ctypes.Structure):
    _fields_ = [("num_q", ctypes.c_int32), ("q_seq", ctypes.c_void_p), ("q_pos", ctypes.c_void_p),
                ("max_kv", ctypes.c_int32)]


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("num_rows", ctypes.c_int64), ("seq_stride", ctypes.c_int64),
                ("block_table", ctypes.c_void_p), ("block_size", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32)]


class IndexerInputs(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("heads", ctypes.c_int32), ("dim", ctypes.c_int32),
                ("q", ctypes.c_void_p), ("q_scale", ctypes.c_void_p), ("w", ctypes.c_void_p),
                ("k", ctypes.c_void_p), ("k_scale", ctypes.c_void_p)]


class AttnInputs(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("heads", ctypes.c_int32), ("d_qk", ctypes.c_int32),
                ("d_v", ctypes.c_int32), ("q", ctypes.c_void_p), ("kv", ctypes.c_void_p),
                ("softmax_scale", ctypes.c_float), ("kv_scale", ctypes.c_void_p)]


class MhaInputs(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("heads", ctypes.c_int32), ("d_nope", ctypes.c_int32),
                ("d_rope", ctypes.c_int32), ("d_v", ctypes.c_int32), ("q", ctypes.c_void_p),
                ("k_nope", ctypes.c_void_p), ("k_rope", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("softmax_scale", ctypes.c_float)]


_P = ctypes.POINTER
_SIGS = {
    "dsa_index_scores": (ctypes.c_int, [_P(QueryDesc), _P(CacheDesc), _P(IndexerInputs), ctypes.c_void_p,
                                        ctypes.c_int64, ctypes.c_void_p]),
    "dsa_index_scores_wait_limit": (ctypes.c_int, [_P(QueryDesc), _P(CacheDesc), _P(IndexerInputs), ctypes.c_void_p,
                                                   ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]),
    "dsa_topk": (ctypes.c_int, [_P(QueryDesc), ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p,
                                ctypes.c_void_p]),
    "dsa_sparse_attn": (ctypes.c_int, [_P(QueryDesc), _P(CacheDesc), _P(AttnInputs), ctypes.c_void_p,
                                       ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "dsa_sparse_attn_mha": (ctypes.c_int, [_P(QueryDesc), _P(CacheDesc), _P(MhaInputs), ctypes.c_void_p,
                                           ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "dsa_forward_workspace_size": (ctypes.c_size_t, [_P(QueryDesc), _P(IndexerInputs), ctypes.c_int32,
                                                     _P(AttnInputs)]),
    "dsa_forward_stage_workspace_size": (ctypes.c_size_t, [_P(QueryDesc), _P(IndexerInputs), ctypes.c_int32,
                                                           _P(AttnInputs), ctypes.c_int64]),
    "dsa_forward_stage_rows": (ctypes.c_int64, [_P(QueryDesc), _P(IndexerInputs), ctypes.c_int32,
                                                _P(AttnInputs), ctypes.c_size_t]),
    "dsa_forward": (ctypes.c_int, [_P(QueryDesc), _P(CacheDesc), _P(IndexerInputs), ctypes.c_int32,
                                   _P(AttnInputs), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "dsa_forward_noalloc": (ctypes.c_int, [_P(QueryDesc), _P(CacheDesc), _P(IndexerInputs), ctypes.c_int32,
                                           _P(AttnInputs), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_void_p]),
    "dsa_cache_append": (ctypes.c_int, [_P(CacheDesc), ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_int, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_void_p]),
    "dsa_kv_dequant": (ctypes.c_int, [ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_void_p]),
    "dsa_indexer_kl_backward": (ctypes.c_int, [_P(QueryDesc), _P(CacheDesc), _P(IndexerInputs), ctypes.c_void_p,
                                               ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "dsa_check_device_error": (ctypes.c_int, [ctypes.c_void_p]),
    "dsa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "dsa_last_error_detail": (ctypes.c_char_p, []),
    "dsa_version": (ctypes.c_int32, []),
    "dsa_profile_start": (ctypes.c_int, [ctypes.c_int32]),
    "dsa_profile_stop": (ctypes.c_int32, []),
    "dsa_profile_read": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]),
    "dsa_launch_count": (ctypes.c_int64, []),
}
DSA_STAGE_INDEXER, DSA_STAGE_TOPK, DSA_STAGE_ATTN, DSA_STAGE_APPEND, DSA_STAGE_INDEXER_BWD = 1, 2, 3, 4, 5
STAGE_NAMES = {1: "indexer", 2: "topk", 3: "attention", 4: "cache_append", 5: "indexer_bwd"}

_lib = None


def lib() -> ctypes.CDLL:
    """Loads libdsa.so once.  Raises if it has not been built: there is no
    fallback implementation."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m sparse_attention_long_11_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().dsa_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != DSA_OK:
        detail = lib().dsa_last_error_detail().decode() if status == DSA_ERR_CUDA else ""
        raise DSAError(status, where + (f" [{detail}]" if detail else ""))


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


# --------------------------------------------------------------------------- descriptors

@dataclasses.dataclass
class Batch:
    """Device-side query batch plus its host-side bound (see dsa_query_desc)."""
    q_seq: torch.Tensor   # int32 [num_q]
    q_pos: torch.Tensor   # int32 [num_q]
    max_kv: int

    def desc(self, r0: int = 0, r1: Optional[int] = None) -> QueryDesc:
        r1 = self.q_pos.shape[0] if r1 is None else r1
        return QueryDesc(r1 - r0, _ptr(self.q_seq[r0:r1]) if r1 > r0 else None,
                         _ptr(self.q_pos[r0:r1]) if r1 > r0 else None, self.max_kv)


@dataclasses.dataclass
class Cache:
    num_seqs: int
    num_rows: int
    seq_stride: int = 0
    block_table: Optional[torch.Tensor] = None  # int32 [num_seqs, max_blocks]
    block_size: int = 0

    def desc(self) -> CacheDesc:
        bt = self.block_table
        return CacheDesc(self.num_seqs, self.num_rows, self.seq_stride, _ptr(bt), self.block_size,
                         0 if bt is None else bt.shape[1])


def indexer_inputs(dtype: int, q, q_scale, w, k, k_scale) -> IndexerInputs:
    return IndexerInputs(dtype, q.shape[-2], q.shape[-1], _ptr(q), _ptr(q_scale), _ptr(w), _ptr(k), _ptr(k_scale))


def attn_inputs(dtype: int, q, kv, d_v: int, softmax_scale: float, kv_scale=None) -> AttnInputs:
    """DSA_FP8_E4M3: bf16 q, uint8 e4m3 kv codes and their fp32 kv_scale rows."""
    return AttnInputs(dtype, q.shape[-2], q.shape[-1], d_v, _ptr(q), _ptr(kv), softmax_scale,
                      None if kv_scale is None else _ptr(kv_scale))


# --------------------------------------------------------------------------- entry points

def dsa_index_scores(batch: QueryDesc, cache: CacheDesc, ix: IndexerInputs, scores: torch.Tensor,
                     stream=None) -> None:
    _check(lib().dsa_index_scores(ctypes.byref(batch), ctypes.byref(cache), ctypes.byref(ix), _ptr(scores),
                                  scores.stride(0), _stream(stream)), "dsa_index_scores")


def dsa_index_scores_wait_limit(batch: QueryDesc, cache: CacheDesc, ix: IndexerInputs, scores: torch.Tensor,
                                wait_limit_cycles: int, stream=None) -> None:
    """dsa_index_scores with every device-side wait bounded by wait_limit_cycles
    SM clocks (a test aid for the timeout path)."""
    _check(lib().dsa_index_scores_wait_limit(ctypes.byref(batch), ctypes.byref(cache), ctypes.byref(ix),
                                             _ptr(scores), scores.stride(0), int(wait_limit_cycles),
                                             _stream(stream)), "dsa_index_scores_wait_limit")


def dsa_topk(batch: QueryDesc, scores: torch.Tensor, k: int, idx: torch.Tensor, stream=None) -> None:
    _check(lib().dsa_topk(ctypes.byref(batch), _ptr(scores), scores.stride(0), k, _ptr(idx), _stream(stream)),
           "dsa_topk")


def dsa_sparse_attn(batch: QueryDesc, cache: CacheDesc, at: AttnInputs, idx: torch.Tensor, k: int,
                    out: torch.Tensor, lse: torch.Tensor, stream=None) -> None:
    _check(lib().dsa_sparse_attn(ctypes.byref(batch), ctypes.byref(cache), ctypes.byref(at), _ptr(idx), k,
                                 _ptr(out), _ptr(lse), _stream(stream)), "dsa_sparse_attn")


def mha_inputs(q, k_nope, k_rope, v, softmax_scale: float) -> MhaInputs:
    """Per-head attention operands (bf16): q [num_q, H, 192], k_nope [rows, H, 128],
    k_rope [rows, 64], v [rows, H, 128]."""
    return MhaInputs(DSA_BF16, q.shape[1], k_nope.shape[-1], k_rope.shape[-1], v.shape[-1], _ptr(q), _ptr(k_nope),
                     _ptr(k_rope), _ptr(v), softmax_scale)


def dsa_sparse_attn_mha(batch: QueryDesc, cache: CacheDesc, at: MhaInputs, idx: torch.Tensor, k: int,
                        out: torch.Tensor, lse: torch.Tensor, stream=None) -> None:
    """Per-head (non-absorbed) sparse attention: the prefill attention mode."""
    _check(lib().dsa_sparse_attn_mha(ctypes.byref(batch), ctypes.byref(cache), ctypes.byref(at), _ptr(idx), k,
                                     _ptr(out), _ptr(lse), _stream(stream)), "dsa_sparse_attn_mha")


def dsa_forward_workspace_size(batch: QueryDesc, ix: IndexerInputs, k: int, at: AttnInputs) -> int:
    return int(lib().dsa_forward_workspace_size(ctypes.byref(batch), ctypes.byref(ix), k, ctypes.byref(at)))


def dsa_forward_stage_workspace_size(batch: QueryDesc, ix: IndexerInputs, k: int, at: AttnInputs,
                                     stage_rows: int) -> int:
    return int(lib().dsa_forward_stage_workspace_size(ctypes.byref(batch), ctypes.byref(ix), k, ctypes.byref(at),
                                                      int(stage_rows)))


def dsa_forward_stage_rows(batch: QueryDesc, ix: IndexerInputs, k: int, at: AttnInputs, workspace_bytes: int) -> int:
    """Query rows per stage that dsa_forward runs with this much workspace (0: too little)."""
    return int(lib().dsa_forward_stage_rows(ctypes.byref(batch), ctypes.byref(ix), k, ctypes.byref(at),
                                            int(workspace_bytes)))


def dsa_forward(batch: QueryDesc, cache: CacheDesc, ix: IndexerInputs, k: int, at: AttnInputs,
                idx: torch.Tensor, out: torch.Tensor, lse: torch.Tensor, workspace: torch.Tensor,
                stream=None) -> None:
    _check(lib().dsa_forward(ctypes.byref(batch), ctypes.byref(cache), ctypes.byref(ix), k, ctypes.byref(at),
                             _ptr(idx), _ptr(out), _ptr(lse), _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream(stream)), "dsa_forward")


NOALLOC_MAX_KV = 2097152


def dsa_cache_append(cache: CacheDesc, tok_seq: torch.Tensor, tok_pos: torch.Tensor, k_new: torch.Tensor,
                     k_cache: torch.Tensor, k_scale: torch.Tensor, kv_new: Optional[torch.Tensor] = None,
                     kv_cache: Optional[torch.Tensor] = None, stream=None,
                     kv_scale: Optional[torch.Tensor] = None) -> None:
    """Writes new tokens into the caches: key rows (bf16 or fp32, width 128)
    encoded as e4m3 codes with a per-row scale, and optionally latent rows
    (copied into a bf16 cache, or encoded the same way into an FP8 cache
    when kv_scale is given)."""
    if k_new.dtype == torch.bfloat16:
        kdt = DSA_BF16
    elif k_new.dtype == torch.float32:
        kdt = DSA_F32
    else:
        raise TypeError("k_new must be bfloat16 or float32")
    d_qk = kv_new.shape[-1] if kv_new is not None else 0
    _check(lib().dsa_cache_append(ctypes.byref(cache), int(tok_seq.numel()), _ptr(tok_seq), _ptr(tok_pos), kdt,
                                  _ptr(k_new), int(k_new.shape[-1]), _ptr(k_cache), _ptr(k_scale),
                                  None if kv_new is None else _ptr(kv_new), d_qk,
                                  None if kv_cache is None else _ptr(kv_cache),
                                  None if kv_scale is None else _ptr(kv_scale), _stream(stream)),
           "dsa_cache_append")


def dsa_kv_dequant(kv: torch.Tensor, kv_scale: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    """The bf16 rows an FP8 latent cache stands for: out = bf16(kv_scale * code)
    per row (kv uint8 [num_rows, 576], kv_scale fp32 [num_rows], out bf16
    [num_rows, 576])."""
    n = int(kv.shape[0])
    if kv.dtype != torch.uint8 or kv_scale.dtype != torch.float32 or out.dtype != torch.bfloat16:
        raise TypeError("dsa_kv_dequant: kv uint8, kv_scale float32, out bfloat16")
    if tuple(out.shape) != tuple(kv.shape) or kv_scale.numel() != n:
        raise ValueError("dsa_kv_dequant: shapes")
    _check(lib().dsa_kv_dequant(n, _ptr(kv), _ptr(kv_scale), _ptr(out), _stream(stream)), "dsa_kv_dequant")


def dsa_indexer_kl_backward(batch: QueryDesc, cache: CacheDesc, ix: IndexerInputs, idx: torch.Tensor, k: int,
                            p: torch.Tensor, loss: torch.Tensor, dw: torch.Tensor, dq: torch.Tensor,
                            dk: torch.Tensor, grad_scores: Optional[torch.Tensor] = None, stream=None) -> None:
    """Indexer alignment loss KL(p || softmax(I)) over each query's candidate
    entries (idx, -1 padded) and its gradients; dk is accumulated into."""
    _check(lib().dsa_indexer_kl_backward(ctypes.byref(batch), ctypes.byref(cache), ctypes.byref(ix), _ptr(idx), k,
                                         _ptr(p), _ptr(loss), None if grad_scores is None else _ptr(grad_scores),
                                         _ptr(dw), _ptr(dq), _ptr(dk), _stream(stream)),
           "dsa_indexer_kl_backward")


def dsa_forward_noalloc(batch: QueryDesc, cache: CacheDesc, ix: IndexerInputs, k: int, at: AttnInputs,
                        idx: torch.Tensor, out: torch.Tensor, lse: torch.Tensor, stream=None) -> None:
    """dsa_forward without a workspace, for callers that cannot allocate device
    memory: the library keeps its scratch in a fixed device array (calls that
    overlap on the GPU race on it; max_kv <= NOALLOC_MAX_KV)."""
    _check(lib().dsa_forward_noalloc(ctypes.byref(batch), ctypes.byref(cache), ctypes.byref(ix), k,
                                     ctypes.byref(at), _ptr(idx), _ptr(out), _ptr(lse), _stream(stream)),
           "dsa_forward_noalloc")


def dsa_check_device_error(stream=None) -> int:
    return int(lib().dsa_check_device_error(_stream(stream)))


def dsa_version() -> int:
    return int(lib().dsa_version())


def dsa_profile_start(capacity: int) -> None:
    _check(lib().dsa_profile_start(capacity), "dsa_profile_start")


def dsa_profile_stop() -> int:
    return int(lib().dsa_profile_stop())


def dsa_profile_read(cap: int):
    """[(stage, ms)] of the launches recorded by the last profile."""
    st = (ctypes.c_int32 * cap)()
    ms = (ctypes.c_float * cap)()
    n = ctypes.c_int32(0)
    _check(lib().dsa_profile_read(st, ms, cap, ctypes.byref(n)), "dsa_profile_read")
    return [(int(st[i]), float(ms[i])) for i in range(n.value)]


def dsa_launch_count() -> int:
    return int(lib().dsa_launch_count())


# --------------------------------------------------------------------------- workload helpers

class Problem:
    """Descriptors of one generated workload (tensors must be on the GPU),
    built once and reused across calls."""

    def __init__(self, wl):
        self.wl = wl
        self.batch = Batch(wl.q_seq, wl.q_pos, wl.max_kv)
        self.cache = Cache(wl.num_seqs, wl.num_rows, wl.seq_stride, wl.block_table, wl.block_size)
        idt = DSA_FP8_E4M3 if wl.idx_dtype == "fp8" else DSA_F32
        adt = {"bf16": DSA_BF16, "fp8kv": DSA_FP8_E4M3}.get(wl.attn_dtype, DSA_F32)
        self.ix = indexer_inputs(idt, wl.q_idx, wl.q_scale, wl.w, wl.k_idx, wl.k_scale)
        self.at = attn_inputs(adt, wl.q, wl.kv, wl.d_v, wl.softmax_scale, wl.kv_scale)
        self.idx_dtype, self.attn_dtype = idt, adt

    def rows(self, r0: int, r1: int):
        """(batch desc, indexer inputs, attention inputs) for query rows [r0, r1)."""
        wl = self.wl
        ix = indexer_inputs(self.idx_dtype, wl.q_idx[r0:r1], None if wl.q_scale is None else wl.q_scale[r0:r1],
                            wl.w[r0:r1], wl.k_idx, wl.k_scale)
        at = attn_inputs(self.attn_dtype, wl.q[r0:r1], wl.kv, wl.d_v, wl.softmax_scale, wl.kv_scale)
        return self.batch.desc(r0, r1), ix, at

    def out_dtype(self):
        return torch.float32 if self.attn_dtype == DSA_F32 else torch.bfloat16
