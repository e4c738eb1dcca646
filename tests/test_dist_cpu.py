"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): each rank is
an independent replica; the job's time is the maximum over ranks and its
bytes the sum, with a barrier around the timed region."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench

    r, w, _ = bench.dist_setup()
    assert (r, w) == (rank, world)
    bench.barrier(w)
    t = bench.allreduce_max(1.0 + rank, w)          # rank 1 is the slow one
    b = bench.allreduce_sum(100.0 * (rank + 1), w)  # bytes of both replicas
    wl = bench.workload_for("mha_bf16", rank)
    q.put((rank, t, b, wl.seed))
    import torch.distributed as dist

    dist.destroy_process_group()


def test_replicas_aggregate_max_time_and_summed_bytes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[1] for x in res] == [2.0, 2.0]
    assert [x[2] for x in res] == [300.0, 300.0]
    assert res[0][3] != res[1][3]  # replicas draw different inputs
