"""Benchmark of the DSA hot path (lightning indexer -> top-k -> sparse MQA
attention) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one pass of the whole hot path over the long-prefill workload:
L = 32768 tokens of one sequence, processed as 8 chunks of 4096 queries
against the full causal prefix (one dsa_forward call per chunk).  Synthetic,
seeded inputs of the DeepSeek-V3.2 shapes: FP8 indexer with 64 heads x 128,
k = 2048, 128 attention heads over one 576-wide bf16 latent KV row.  The
decode workload (64 sequences x 65536 cached rows, one query each) is timed in
the same run and reported under "decode".

Prints ONE JSON line on rank 0.  Under torchrun each rank runs an
independent replica on its own GPU (weak scaling, no collective on the data
path); timing is the max over ranks.

--impl reference times the CPU oracle (float64 numpy, the machine's host cores)
on a bounded sample of the same workload and prints the same line with
"impl": "reference".
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_attention_long_11_b300 import api, inputs  # noqa: E402

METRIC = "DSA tokens/s (prefill 32K; decode B=64@64K ctx) and % of FP8/BF16/HBM roofline"
FLOP_PER_ATTN_PAIR = 2 * 128 * (576 + 512)        # QK^T + PV per selected (query, key), 128 heads
FLOP_PER_IDX_PAIR = 2 * 64 * 128                  # per causal (query, key) indexer pair
BYTES_PER_IDX_KEY = 128 + 4                       # FP8 key row + its scale
BYTES_PER_ATTN_KEY = 576 * 2                      # gathered bf16 latent row
BYTES_PER_ATTN_KEY_FP8 = 576 + 4                  # gathered FP8 latent row and its scale


def _traffic(entry: str, kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or None
    when no capture exists or the kernel's sources changed since it was taken."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        d = json.load(open(p))[entry]
    except (OSError, KeyError, ValueError):
        return None
    if d.get("kernel", "").split("_")[0] != kernel.split("_")[0]:
        return None
    for rel, h in d["sources_sha256"].items():
        try:
            if hashlib.sha256(open(os.path.join(ROOT, rel), "rb").read()).hexdigest() != h:
                return None
        except OSError:
            return None
    return d["bytes_per_launch"]


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"], src="measured")
    return dict(hbm=6400.0, bf16=1800.0, bf16_sus=1400.0, src="fallback")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return ws, rank, local


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(tokens_per_rank: int, ms_local: float, ws: int):
    """Whole-job throughput of N independent replicas: every rank processed
    `tokens_per_rank` tokens; the job took the slowest rank's time.
    Returns (tokens/s over all ranks, ms per step of the slowest rank)."""
    ms = _max_over_ranks(ms_local, ws)
    return tokens_per_rank * ws / (ms / 1e3), ms


class Runner:
    """Outputs, workspace and one full step of dsa_forward over a workload."""

    def __init__(self, wl):
        self.wl = wl
        self.prob = api.Problem(wl)
        dev = wl.q.device
        self.idx = torch.empty((wl.num_q, wl.topk), dtype=torch.int32, device=dev)
        self.out = torch.empty((wl.num_q, wl.H, wl.d_v), dtype=self.prob.out_dtype(), device=dev)
        self.lse = torch.empty((wl.num_q, wl.H), dtype=torch.float32, device=dev)
        self.calls = []
        for a, b in wl.chunks:
            qd, ix, at = self.prob.rows(a, b)
            self.calls.append((a, b, qd, ix, at))
        wsb = max(api.dsa_forward_workspace_size(qd, ix, wl.topk, at) for _, _, qd, ix, at in self.calls)
        self.ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        self.cache = self.prob.cache.desc()

    def step(self):
        for ci in range(len(self.calls)):
            self.chunk(ci)

    def chunk(self, ci: int, stream=None):
        """dsa_forward over call ci (one chunk of query rows)."""
        a, b, qd, ix, at = self.calls[ci]
        api.dsa_forward(qd, self.cache, ix, self.wl.topk, at, self.idx[a:b], self.out[a:b], self.lse[a:b], self.ws,
                        stream=stream)


def _pairs(wl):
    """Algorithmic work of one step: (indexer pairs, selected attention pairs).
    A query at position t with t + 1 <= k selects all its t + 1 keys, so only
    queries with t + 1 > k need indexer scores: the indexer's work is their
    causal (query, key) pairs; attention has min(t + 1, k) pairs a query."""
    n = wl.q_pos.to(torch.int64) + 1
    return int(torch.where(n > wl.topk, n, torch.zeros_like(n)).sum()), int(torch.clamp(n, max=wl.topk).sum())


def _time_steps(r: Runner, steps: int, warmup: int, ws: int, gpu: int, profile: bool = True):
    """Times `steps` steps after `warmup` untimed ones, with CUDA events on the
    launching stream and nvidia-smi clocks sampled during the timed region.
    With `profile`, every launch is also bracketed by library events (per-stage
    device time); the loop time is then measured with that bookkeeping in it.
    Returns (ms per step, {stage: [launches, total ms]}, launches, clocks)."""
    for _ in range(warmup):
        r.step()
    torch.cuda.synchronize()
    cap = 0
    if profile:
        cap = max(8192, steps * len(r.calls) * 8)
        api.dsa_profile_start(cap)
    n0 = api.dsa_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu) as clk:
        _barrier(ws)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(steps):
            r.step()
        e1.record()
        torch.cuda.synchronize()
        _barrier(ws)
    launches = api.dsa_launch_count() - n0
    per_stage = {}
    if profile:
        api.dsa_profile_stop()
        for s_, t in api.dsa_profile_read(cap):
            d = per_stage.setdefault(api.STAGE_NAMES[s_], [0, 0.0])
            d[0] += 1
            d[1] += t
    st = api.dsa_check_device_error()
    if st != api.DSA_OK:
        raise RuntimeError(f"device error during bench: {api.status_string(st)}")
    ms = e0.elapsed_time(e1) / steps
    return ms, per_stage, launches, clk.summary()


def _roofline_prefill(wl, per_stage, steps, peaks):
    """Dominant kernel of the prefill step (by device time) against its roofline."""
    n_idx, n_attn = _pairs(wl)
    dom = max(per_stage, key=lambda s: per_stage[s][1])
    cnt, tot = per_stage[dom]
    avg_s = tot / cnt / 1e3
    per_launch_units = {"indexer": n_idx * steps / cnt, "attention": n_attn * steps / cnt,
                        "topk": n_idx * steps / cnt}[dom]
    if dom == "attention":
        achieved = per_launch_units * FLOP_PER_ATTN_PAIR / avg_s / 1e12
        return {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peaks["bf16"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16"],
                "frac_of_sustained": achieved / peaks["bf16_sus"],
                "traffic": _traffic("prefill_attention", "attn"),
                "peak_src": f"{peaks['src']} bf16 burst (kernel timed in a sub-second step); "
                            f"frac_of_sustained against {peaks['bf16_sus']}",
                "avg_launch_ms": tot / cnt, "launches": cnt}
    if dom == "indexer":
        # FP8 peak = measured bf16 peak x the nominal fp8/bf16 ratio (2)
        pk = 2 * peaks["bf16"]
        achieved = per_launch_units * FLOP_PER_IDX_PAIR / avg_s / 1e12
        return {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": pk, "unit": "TFLOP/s",
                "frac": achieved / pk, "frac_of_sustained": achieved / (2 * peaks["bf16_sus"]), "traffic": None,
                "peak_src": f"{peaks['src']} bf16 burst x2 (fp8/bf16 nominal ratio)",
                "avg_launch_ms": tot / cnt, "launches": cnt}
    achieved = per_launch_units * 4 / avg_s / 1e9
    return {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm"], "unit": "GB/s",
            "frac": achieved / peaks["hbm"], "traffic": None, "peak_src": f"{peaks['src']} hbm",
            "avg_launch_ms": tot / cnt, "launches": cnt}


def _roofline_decode(wl, per_stage, steps, peaks):
    n_idx, n_attn = _pairs(wl)
    dom = max(per_stage, key=lambda s: per_stage[s][1])
    cnt, tot = per_stage[dom]
    avg_s = tot / cnt / 1e3
    if dom == "indexer":
        byts = n_idx * BYTES_PER_IDX_KEY * steps / cnt
    elif dom == "attention":
        byts = n_attn * BYTES_PER_ATTN_KEY * steps / cnt
    else:
        byts = n_idx * 4 * steps / cnt
    achieved = byts / avg_s / 1e9
    return {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm"], "unit": "GB/s",
            "frac": achieved / peaks["hbm"], "traffic": _traffic("decode_indexer", dom) if dom == "indexer" else None,
            "peak_src": f"{peaks['src']} hbm burst",
            "avg_launch_ms": tot / cnt, "launches": cnt}


def _decode_stage_roofline(wl, per_stage, steps, peaks):
    """HBM fraction of every decode stage: algorithmic bytes per launch (indexer:
    the FP8 key rows and scales of every scored pair; top-k: the k candidate
    keys a selecting query needs at the least, and the index rows written;
    attention: the gathered latent rows plus q read and O written) over its
    average launch time."""
    n_idx, n_attn = _pairs(wl)
    n_sel = int((wl.q_pos.to(torch.int64) + 1 > wl.topk).sum())   # queries that select from more than k keys
    byts = {"indexer": n_idx * BYTES_PER_IDX_KEY,
            # the streamed selection reads at least k candidates (8-byte keys) of
            # each selecting query and writes every index row
            "topk": n_sel * wl.topk * 8 + wl.num_q * wl.topk * 4,
            "attention": n_attn * BYTES_PER_ATTN_KEY + wl.num_q * wl.H * (wl.d_qk + wl.d_v) * 2}
    out = {}
    for name, (cnt, tot) in per_stage.items():
        if name not in byts:
            continue
        ms = tot / steps
        gbs = byts[name] / (ms / 1e3) / 1e9
        out[name] = {"bytes": byts[name], "ms": ms, "achieved_gbs": gbs, "frac": gbs / peaks["hbm"]}
    return out


def _time_append(wl, r: Runner, steps: int, warmup: int):
    """The decode loop's cache write: one new token per sequence (bf16 key of
    width 128 encoded to e4m3 + scale, and its 576-wide bf16 latent row,
    copied, or encoded to e4m3 + scale for an FP8 latent cache), written at
    each sequence's last position.  Timed with CUDA events after the decode
    steps (it rewrites those rows)."""
    dev = wl.q.device
    n = wl.num_seqs
    k_new = inputs.randn((n, 128), 1, "append_k", dev).to(torch.bfloat16)
    kv_new = inputs.randn((n, 576), 1, "append_kv", dev).to(torch.bfloat16)
    seq = torch.arange(n, dtype=torch.int32, device=dev)
    pos = torch.tensor(wl.seq_lens, dtype=torch.int32, device=dev) - 1
    cache = r.prob.cache.desc()

    def one():
        api.dsa_cache_append(cache, seq, pos, k_new, wl.k_idx, wl.k_scale, kv_new, wl.kv, kv_scale=wl.kv_scale)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    api.dsa_profile_start(steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        one()
    e1.record()
    torch.cuda.synchronize()
    api.dsa_profile_stop()
    recs = api.dsa_profile_read(steps)
    st = api.dsa_check_device_error()
    if st != api.DSA_OK:
        raise RuntimeError(f"device error during cache append: {api.status_string(st)}")
    loop_ms = e0.elapsed_time(e1) / steps          # includes the host call between launches
    ms = sum(t for _, t in recs) / max(1, len(recs))   # the kernel alone, from the launch events
    kv_row = 576 + 4 if wl.kv_scale is not None else 576 * 2
    byts = n * ((128 * 2 + 576 * 2) + (128 + 4 + kv_row))   # read new rows, write cache rows
    return {"tokens": n, "ms": ms, "loop_ms_per_call": loop_ms, "bytes": byts,
            "achieved_gbs": byts / (ms / 1e3) / 1e9,
            "note": "latency-bound: one 128-thread block per 4 tokens; ms from the launch's own events"}




def _time_kl_backward(r: Runner, steps: int, warmup: int, peaks):
    """The indexer's training step (alignment loss + gradients) over the last
    4096-query call of the prefill, on the entries the forward selected and
    seeded synthetic targets.  One launch per step, timed with CUDA events."""
    wl = r.wl
    a, b = wl.chunks[-1]
    qd, ix, _ = r.prob.rows(a, b)
    idx = r.idx[a:b]
    k = wl.topk
    p = inputs.kl_targets(idx, seed=1)
    n = b - a
    loss = torch.empty(n, dtype=torch.float32, device=idx.device)
    g = torch.empty((n, k), dtype=torch.float32, device=idx.device)
    dw = torch.empty((n, wl.H_I), dtype=torch.float32, device=idx.device)
    dq = torch.empty((n, wl.H_I, wl.d_I), dtype=torch.float32, device=idx.device)
    dk = torch.zeros((wl.num_rows, wl.d_I), dtype=torch.float32, device=idx.device)
    cache = r.prob.cache.desc()

    def one():
        api.dsa_indexer_kl_backward(qd, cache, ix, idx, k, p, loss, dw, dq, dk, g)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        one()
    e1.record()
    torch.cuda.synchronize()
    st = api.dsa_check_device_error()
    if st != api.DSA_OK:
        raise RuntimeError(f"device error during the indexer backward: {api.status_string(st)}")
    ms = e0.elapsed_time(e1) / steps
    pairs = int((idx >= 0).sum().item())
    flop = pairs * 3 * 2 * wl.H_I * wl.d_I          # head dots, dq, dk: one 64 x 128 contraction each
    tf = flop / (ms / 1e3) / 1e12
    return {"workload": f"queries {a}..{b - 1} of the L={wl.max_kv} prefill, k={k}, synthetic targets",
            "value": n / (ms / 1e3), "unit": "tokens/s", "ms": ms, "pairs": pairs,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16"], "unit": "TFLOP/s",
                         "frac": tf / peaks["bf16"],
                         "peak_src": f"{peaks['src']} bf16 burst (the three contractions run as fp16 MMAs, "
                                     f"the same rate)"}}


def _time_mha_mode(r: Runner, peaks, nq: int = 512, steps: int = 5, warmup: int = 3):
    """The per-head (non-absorbed) prefill attention mode against the latent
    MQA mode on the same selections: the last nq queries of the prefill, the
    entries the forward selected for them, per-head keys and values of 128
    (rope part 64 shared) for 128 heads.  Each selected pair moves 65,664
    bytes of rows in the per-head mode and 1,152 in the latent one."""
    wl = r.wl
    L = wl.max_kv
    a, b = wl.num_q - nq, wl.num_q
    mh = inputs.make_mha_prefill(seed=0, device=wl.q.device, L=L, heads=128, q_rows=(L - nq, L))
    idx = r.idx[a:b].contiguous()
    bdesc = api.Batch(mh.q_seq, mh.q_pos, L).desc()
    cache = api.Cache(1, L, L).desc()
    out = torch.empty((nq, 128, 128), dtype=torch.bfloat16, device=wl.q.device)
    lse = torch.empty((nq, 128), dtype=torch.float32, device=wl.q.device)
    at = api.mha_inputs(mh.q, mh.k_nope, mh.k_rope, mh.v, mh.softmax_scale)
    qd, _, atl = r.prob.rows(a, b)
    out_l = torch.empty((nq, 128, 512), dtype=torch.bfloat16, device=wl.q.device)
    lse_l = torch.empty((nq, 128), dtype=torch.float32, device=wl.q.device)

    def timed(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    ms_mha = timed(lambda: api.dsa_sparse_attn_mha(bdesc, cache, at, idx, wl.topk, out, lse))
    ms_lat = timed(lambda: api.dsa_sparse_attn(qd, r.cache, atl, idx, wl.topk, out_l, lse_l))
    st = api.dsa_check_device_error()
    if st != api.DSA_OK:
        raise RuntimeError(f"device error in the per-head mode: {api.status_string(st)}")
    pairs = int((idx >= 0).sum().item())
    per_pair = 128 * (128 + 128) * 2 + 64 * 2
    gbs = pairs * per_pair / (ms_mha / 1e3) / 1e9
    del mh, out, lse, out_l, lse_l
    torch.cuda.empty_cache()
    return {"workload": f"queries {L - nq}..{L - 1} of the L={L} prefill on the forward's selections, 128 heads, "
                        f"per-head keys/values 128 + shared rope 64 (bf16)",
            "pairs": pairs, "bytes_per_pair": per_pair, "latent_bytes_per_pair": BYTES_PER_ATTN_KEY,
            "ms": ms_mha, "latent_ms": ms_lat, "ratio": ms_mha / ms_lat,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm"], "peak_src": f"{peaks['src']} hbm"}}


def _e2e(wl, steps: int):
    """Same metric through the public API with host buffers.  Every step
    copies the step's inputs from pinned host memory, runs dsa_forward chunk
    by chunk and copies the outputs back; a chunk's input copy, compute and
    output copy run on three streams, so the copies of one chunk overlap the
    compute of its neighbours (the host link, not the GPU, bounds this
    number).  Steps are separated by a device synchronisation.
    Returns (tokens/s, h2d bytes, d2h bytes, ms per step)."""
    row_names = ["q_idx", "q_scale", "w", "q", "q_seq", "q_pos"]   # one entry per query row
    cache_names = ["k_idx", "k_scale", "kv"]
    host = {n: getattr(wl, n).to("cpu").pin_memory() for n in row_names + cache_names}
    r = Runner(wl)
    dev_t = {n: getattr(wl, n) for n in row_names + cache_names}
    out_h = torch.empty(r.out.shape, dtype=r.out.dtype).pin_memory()
    lse_h = torch.empty(r.lse.shape, dtype=r.lse.dtype).pin_memory()
    idx_h = torch.empty(r.idx.shape, dtype=r.idx.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in (out_h, lse_h, idx_h))
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def one():
        with torch.cuda.stream(s_in):
            for n in cache_names:
                dev_t[n].copy_(host[n], non_blocking=True)
        for ci, (a, b) in enumerate(wl.chunks):
            with torch.cuda.stream(s_in):
                for n in row_names:
                    dev_t[n][a:b].copy_(host[n][a:b], non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
            s_cmp.wait_event(ev_in)
            r.chunk(ci, s_cmp)
            ev_done = torch.cuda.Event()
            ev_done.record(s_cmp)
            s_out.wait_event(ev_done)
            with torch.cuda.stream(s_out):
                out_h[a:b].copy_(r.out[a:b], non_blocking=True)
                lse_h[a:b].copy_(r.lse[a:b], non_blocking=True)
                idx_h[a:b].copy_(r.idx[a:b], non_blocking=True)

    one()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
        torch.cuda.synchronize()
    ms = (time.perf_counter() - t0) * 1e3 / steps
    del host, out_h, lse_h, idx_h
    return wl.num_q / (ms / 1e3), h2d, d2h, ms


class OracleSampler:
    """The CPU oracle (full path: indexer, top-k, attention) over a stratified
    sample of the workload's queries: 256 evenly spaced query rows, visited in
    a seeded random order so that any prefix of the visit is an unbiased
    sample of the positions (early queries are cheaper than late ones).
    Successive calls continue where the last one stopped."""

    def __init__(self, wl, points: int = 256, seed: int = 0):
        from oracle.workload_view import OracleView
        self.view = OracleView(wl)
        self.pos = wl.q_pos.to("cpu").numpy()
        pts = np.linspace(0, wl.num_q - 1, min(wl.num_q, points)).astype(int)
        self.order = pts[np.random.default_rng(seed).permutation(len(pts))]
        self.next = 0
        self.visited = []

    def run(self, budget_s: float, max_q: int = 1 << 30):
        """Runs queries until budget_s is spent (at least one); returns (queries, seconds)."""
        t0 = time.perf_counter()
        done = 0
        while done < max_q:
            i = int(self.order[self.next % len(self.order)])
            self.next += 1
            self.view.run(i)
            self.visited.append(int(self.pos[i]))
            done += 1
            if time.perf_counter() - t0 > budget_s:
                break
        return done, time.perf_counter() - t0

    def describe(self) -> str:
        v = np.asarray(self.visited)
        distinct = len(set(self.visited))
        return (f"{len(v)} query visits ({distinct} distinct of {len(self.order)} evenly spaced rows, seeded random "
                f"order), positions {v.min()}..{v.max()}, mean {v.mean():.0f}")


def _blas_threads() -> int:
    """Threads the oracle's BLAS uses (numpy matmul), else the usable cores."""
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        n = max([d.get("num_threads", 0) for d in info if d.get("user_api") == "blas"] + [0])
        if n:
            return n
    except ImportError:
        pass
    return len(os.sched_getaffinity(0))


def run_reference(args, ws, rank):
    if rank != 0:
        return
    wl = inputs.make_long(seed=0, device="cuda" if torch.cuda.is_available() else "cpu")
    budget = 4.0
    warm = OracleSampler(wl, seed=1)
    for _ in range(args.warmup):
        warm.run(0.5, max_q=1)
    samp = OracleSampler(wl, seed=0)
    done_tot, t_tot = 0, 0.0
    for _ in range(args.steps):
        d, t = samp.run(budget)
        done_tot += d
        t_tot += t
    val = done_tot / t_tot
    cores = _blas_threads()
    sample = (f"{samp.describe()} of the L=32768 prefill over {args.steps} steps "
              f"(~{budget:.0f} s of oracle work per step)")
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_tot / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": "long prefill L=32768 (8 chunks x 4096), k=2048",
                                            "sample": sample},
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=2)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-k-sweep", action="store_true")
    ap.add_argument("--no-128k", action="store_true")
    ap.add_argument("--no-fp8-kv", action="store_true")
    ap.add_argument("--no-kl-backward", action="store_true")
    ap.add_argument("--no-mixed", action="store_true")
    ap.add_argument("--no-mha", action="store_true")
    args = ap.parse_args()
    ws, rank, local = _dist()
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    peaks = _peaks()
    api.lib()

    # ---------------- long prefill (the reported workload)
    wl = inputs.make_long(seed=0, device=dev)
    r = Runner(wl)
    ms, per_stage, launches, clocks = _time_steps(r, args.steps, args.warmup, ws, local)
    value, ms = aggregate(wl.num_q, ms, ws)
    roof = _roofline_prefill(wl, per_stage, args.steps, peaks)
    stages = {k: {"launches": v[0], "ms_per_step": v[1] / args.steps} for k, v in per_stage.items()}
    # the indexer's training step on the selections of the last call (after the timed region)
    kl_bwd = None if args.no_kl_backward else _time_kl_backward(r, 3, 2, peaks)
    mha_mode = None if args.no_mha else _time_mha_mode(r, peaks)
    del r
    torch.cuda.empty_cache()
    e2e_val, h2d, d2h, e2e_ms = _e2e(wl, args.e2e_steps)
    e2e_val = e2e_val * ws

    cpu = None
    if rank == 0 and ws == 1:
        samp = OracleSampler(wl, seed=0)
        done, dt = samp.run(args.cpu_budget, max_q=len(samp.order))
        cpu = {"value": done / dt, "unit": "tokens/s", "cores": _blas_threads(), "kind": "oracle",
               "sample": f"{samp.describe()} of the L=32768 prefill, full oracle path (indexer, top-k, "
                         f"attention) in {dt:.1f} s"}
    prefill_fp8_kv = None
    if not args.no_fp8_kv:
        # the same prefill over an FP8 latent cache (not part of the headline value)
        r8 = Runner(inputs.with_fp8_kv(wl))
        ms8, st8, _, _ = _time_steps(r8, 2, args.warmup, ws, local)
        ms8 = _max_over_ranks(ms8, ws)
        prefill_fp8_kv = {"value": wl.num_q * ws / (ms8 / 1e3), "unit": "tokens/s", "ms_per_step": ms8,
                          "stages": {n: round(v[1] / 2, 3) for n, v in st8.items()}}
        del r8
        torch.cuda.empty_cache()
    k_sweep = None
    if not args.no_k_sweep:
        # the same prefill and inputs with other top-k sizes (not part of the headline value)
        k_sweep = {}
        for kk in (1024, 4096, 8192):
            rk = Runner(dataclasses.replace(wl, topk=kk))
            kms, kst, _, _ = _time_steps(rk, 2, args.warmup, ws, local)
            kms = _max_over_ranks(kms, ws)
            k_sweep[str(kk)] = {"value": wl.num_q * ws / (kms / 1e3), "unit": "tokens/s", "ms_per_step": kms,
                                "stages": {n: round(v[1] / 2, 3) for n, v in kst.items()}}
            del rk
            torch.cuda.empty_cache()
    del wl
    torch.cuda.empty_cache()

    # ---------------- 128K prefill (not part of the headline value): where the indexer leads
    long128k = None
    if not args.no_128k:
        wx = inputs.make_prefill(seed=0, device=dev, L=131072, chunk=4096, name="long128k")
        rx = Runner(wx)
        xms, xst, _, _ = _time_steps(rx, 2, args.warmup, ws, local)
        xms = _max_over_ranks(xms, ws)
        n_idx, n_attn = _pairs(wx)
        ims, ams = xst["indexer"][1] / 2, xst["attention"][1] / 2
        long128k = {"workload": "single-sequence causal prefill L=131072 in 32 calls of 4096 queries, k=2048",
                    "value": wx.num_q * ws / (xms / 1e3), "unit": "tokens/s", "ms_per_step": xms,
                    "stages": {n: round(v[1] / 2, 3) for n, v in xst.items()},
                    "indexer_tflops": n_idx * FLOP_PER_IDX_PAIR / (ims / 1e3) / 1e12,
                    "attention_tflops": n_attn * FLOP_PER_ATTN_PAIR / (ams / 1e3) / 1e12}
        del rx, wx
        torch.cuda.empty_cache()

    # ---------------- decode batch (second half of the metric)
    decode = None
    if not args.no_decode:
        wd = inputs.make_decode(seed=0, device=dev)
        rd = Runner(wd)
        # per-stage device times from a short run with per-launch events
        nprof = 20
        _, dstage, _, _ = _time_steps(rd, nprof, args.warmup, ws, local, profile=True)
        # the decode value: at least one second of back-to-back steps without
        # per-launch bookkeeping, so that the clock sampler sees the load
        est, _, _, _ = _time_steps(rd, 20, 1, ws, local, profile=False)
        nd = max(args.steps, int(math.ceil(1200.0 / max(est, 1e-3))))
        dms, _, dl, dclk = _time_steps(rd, nd, 1, ws, local, profile=False)
        dval, dms = aggregate(wd.num_q, dms, ws)
        decode = {"workload": "decode B=64, ctx 65536 each, k=2048", "value": dval,
                  "unit": "tokens/s", "ms_per_step": dms, "steps": nd, "gpu_launches": dl,
                  "stages": {k: {"launches": v[0], "ms_per_step": v[1] / nprof} for k, v in dstage.items()},
                  "stage_roofline": _decode_stage_roofline(wd, dstage, nprof, peaks),
                  "roofline": _roofline_decode(wd, dstage, nprof, peaks), "clocks": dclk}
        decode["cache_append"] = _time_append(wd, rd, max(args.steps, 10), args.warmup)
        del rd
        if not args.no_fp8_kv:
            # the same batch over an FP8 latent cache (e4m3 codes + one fp32 scale per row)
            w8 = inputs.with_fp8_kv(wd)
            r8 = Runner(w8)
            ms8, st8, _, _ = _time_steps(r8, nprof, args.warmup, ws, local)
            v8, ms8 = aggregate(w8.num_q, ms8, ws)
            _, n_attn = _pairs(w8)
            a_ms = st8["attention"][1] / nprof
            decode["fp8_kv"] = {"value": v8, "unit": "tokens/s", "ms_per_step": ms8,
                                "stages": {n: round(v[1] / nprof, 4) for n, v in st8.items()},
                                "attention_gather_gbs": n_attn * BYTES_PER_ATTN_KEY_FP8 / (a_ms / 1e3) / 1e9}
            decode["fp8_kv"]["cache_append"] = _time_append(w8, r8, max(args.steps, 10), args.warmup)
            del r8, w8
        del wd
        torch.cuda.empty_cache()

    # ---------------- mixed paged batch (not part of the headline value)
    mixed = None
    if not args.no_mixed:
        wm = inputs.make_mixed(seed=0, device=dev)
        rm = Runner(wm)
        mms, mst, _, mclk = _time_steps(rm, 2, args.warmup, ws, local)
        mms = _max_over_ranks(mms, ws)
        n_idx, n_attn = _pairs(wm)
        ims, ams = mst["indexer"][1] / 2, mst["attention"][1] / 2
        at_tf = n_attn * FLOP_PER_ATTN_PAIR / (ams / 1e3) / 1e12
        mixed = {"workload": f"mixed paged batch: 8 sequences of {min(wm.seq_lens)}..{max(wm.seq_lens)} cached "
                             f"rows (block 64, permuted pool), per sequence 8192 prefill + 32 decode queries, "
                             f"k=2048, one call",
                 "value": wm.num_q * ws / (mms / 1e3), "unit": "tokens/s", "ms_per_step": mms,
                 "queries": wm.num_q, "indexer_pairs": n_idx, "attention_pairs": n_attn,
                 "stages": {n: round(v[1] / 2, 3) for n, v in mst.items()},
                 "indexer_tflops": n_idx * FLOP_PER_IDX_PAIR / (ims / 1e3) / 1e12,
                 "roofline": {"kernel": "attention", "bound": "tensor", "achieved": at_tf, "peak": peaks["bf16"],
                              "unit": "TFLOP/s", "frac": at_tf / peaks["bf16"],
                              "peak_src": f"{peaks['src']} bf16 burst"},
                 "clocks": mclk}
        del rm, wm
        torch.cuda.empty_cache()

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "fp8+bf16 (fp32 accumulate)", "data": "synthetic",
                "config": {"workload": "long prefill L=32768, 8 chunks x 4096 queries, causal, k=2048; "
                                       "indexer FP8 64x128; attention 128 heads, d_qk 576, d_v 512, bf16",
                           "global_batch": 1, "seq_len": 32768, "parallelism": f"replicas x{ws}",
                           "l2": "inputs larger than L2 (q alone is 4.8 GB)"},
                "roofline": roof, "stages": stages, "gpu_launches": launches, "clocks": clocks,
                "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
                "cpu_baseline": cpu, "decode": decode, "k_sweep": k_sweep,
                "prefill_128k": long128k, "prefill_fp8_kv": prefill_fp8_kv, "indexer_kl_backward": kl_bwd,
                "mixed": mixed, "prefill_mha_mode": mha_mode}
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
