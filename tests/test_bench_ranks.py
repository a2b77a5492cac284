"""Host logic of the multi-replica benchmark (N > 1): every rank runs an
independent replica, the job time is the slowest rank's, and the reported
throughput is all ranks' tokens over that time.  Runs as two gloo ranks on
the CPU; no GPU and no data-path collective are involved."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, ws: int, port: int, q):
    os.environ["CUDA_VISIBLE_DEVICES"] = ""    # gloo ranks on the host, even where a GPU exists
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, local = bench._dist()            # gloo: no CUDA in this process
    assert (w, r, local) == (ws, rank, rank)
    ms_local = [40.0, 50.0][rank]          # rank 1 is the slow one
    value, ms = bench.aggregate(32768, ms_local, ws)
    bench._barrier(ws)
    q.put((rank, value, ms))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_replicas_report_all_tokens_over_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(100)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, value, ms in res:
        assert ms == 50.0                              # max over ranks
        assert value == pytest.approx(2 * 32768 / 0.050)   # both ranks' tokens / slowest time


def test_single_rank_is_plain_throughput():
    sys.path.insert(0, ROOT)
    import bench
    value, ms = bench.aggregate(64, 0.5, 1)
    assert ms == 0.5 and value == pytest.approx(64 / 0.0005)


def test_oracle_sampler_visits_every_stratified_point_in_a_seeded_order():
    import bench
    from sparse_attention_long_11_b300 import inputs
    wl = inputs.make_tiny(seed=0, L=64, topk=16)
    a, b = bench.OracleSampler(wl, points=16, seed=3), bench.OracleSampler(wl, points=16, seed=3)
    assert list(a.order) == list(b.order) and sorted(a.order) == sorted(set(a.order))
    assert list(a.order) != sorted(a.order)                  # not ascending: any prefix mixes early and late rows
    n1, _ = a.run(1e9, max_q=5)
    n2, _ = a.run(1e9, max_q=11)                              # continues where the first call stopped
    assert (n1, n2) == (5, 11)
    assert sorted(a.visited) == sorted(int(wl.q_pos[i]) for i in a.order)
