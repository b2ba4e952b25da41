"""bench.py's replica coordination for N > 1 (one process per GPU, independent
replicas): a host barrier and the max of the per-rank times, over gloo. Run
here with two CPU ranks; no GPU and no data of the computation is involved."""
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import os
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_env()
    rep = bench.Replicas(w, r)
    rep.barrier()
    slowest = rep.max(10.0 + 5.0 * r)      # per-rank step time, ms
    rep.barrier()
    rep.close()
    q.put((r, w, local, slowest))


def test_two_rank_replicas_report_the_slowest_rank():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1]
    assert all(o[1] == 2 for o in out)
    assert all(o[3] == 15.0 for o in out)
