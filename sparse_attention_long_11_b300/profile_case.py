"""Runs one DSA workload through dsa_forward a few times, for profilers.

    python -m sparse_attention_long_11_b300.profile_case --workload prefill --reps 2

Workloads: tiny, prefill (L=4096), long (L=32768, 8 chunks), decode
(64 x 65536), mixed (8 paged sequences).  --fp8-kv stores the latent cache
as FP8 (e4m3 codes and a scale per row).  With --kl-backward it runs, after
the forward repetitions, the indexer's training step (dsa_indexer_kl_backward)
on the selected entries with seeded synthetic targets, --reps times.
Exits non-zero on a device error.
"""
import argparse
import sys

import torch

from . import api, inputs


def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="prefill", choices=inputs.CONFIG_NAMES)
    ap.add_argument("--reps", type=int, default=2)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--q-rows", default=None,
                    help="a:b -- keep only query positions [a, b) of the prefill workloads (all keys stay cached)")
    ap.add_argument("--kl-backward", action="store_true",
                    help="then run the indexer backward on the forward's selections, --reps times")
    ap.add_argument("--decode-batch", type=int, default=64,
                    help="sequences of the decode workload (65536 cached rows each)")
    ap.add_argument("--fp8-kv", action="store_true", help="the latent cache stored as FP8")
    a = ap.parse_args()
    if a.q_rows and a.workload in ("prefill", "long"):
        r0, r1 = (int(x) for x in a.q_rows.split(":"))
        L = 4096 if a.workload == "prefill" else 32768
        wl = inputs.make_prefill(seed=a.seed, device="cuda", L=L, name=a.workload, q_rows=(r0, r1))
    elif a.workload == "decode":
        wl = inputs.make_decode(seed=a.seed, device="cuda", batch=a.decode_batch)
    else:
        wl = inputs.make_config(inputs.CONFIG_NAMES.index(a.workload), seed=a.seed, device="cuda")
    if a.fp8_kv:
        wl = inputs.with_fp8_kv(wl)
    prob = api.Problem(wl)
    idx = torch.empty((wl.num_q, wl.topk), dtype=torch.int32, device="cuda")
    out = torch.empty((wl.num_q, wl.H, wl.d_v), dtype=prob.out_dtype(), device="cuda")
    lse = torch.empty((wl.num_q, wl.H), dtype=torch.float32, device="cuda")
    calls = [(a_, b_) + prob.rows(a_, b_) for a_, b_ in wl.chunks]
    wsb = max(api.dsa_forward_workspace_size(qd, ix, wl.topk, at) for _, _, qd, ix, at in calls)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    cache = prob.cache.desc()
    for _ in range(a.reps):
        for r0, r1, qd, ix, at in calls:
            api.dsa_forward(qd, cache, ix, wl.topk, at, idx[r0:r1], out[r0:r1], lse[r0:r1], ws)
    if a.kl_backward:
        p = inputs.kl_targets(idx, seed=1)
        loss = torch.empty(wl.num_q, dtype=torch.float32, device="cuda")
        dw = torch.empty((wl.num_q, wl.H_I), dtype=torch.float32, device="cuda")
        dq = torch.empty((wl.num_q, wl.H_I, wl.d_I), dtype=torch.float32, device="cuda")
        dk = torch.zeros((wl.num_rows, wl.d_I), dtype=torch.float32, device="cuda")
        for _ in range(a.reps):
            api.dsa_indexer_kl_backward(prob.batch.desc(), cache, prob.ix, idx, wl.topk, p, loss, dw, dq, dk)
    st = api.dsa_check_device_error()
    print(f"{a.workload}: {wl.num_q} queries x {a.reps} reps, launches={api.dsa_launch_count()}, "
          f"status={api.status_string(st)}")
    return 0 if st == api.DSA_OK else 1


if __name__ == "__main__":
    sys.exit(main())
