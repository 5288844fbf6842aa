"""The bench's multi-rank host logic on CPU: two gloo ranks get disjoint row
windows of the seeded stream and agree on the max-over-ranks time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, w, local = bench.dist_env()
    t = bench.reduce_max(float(rank + 1) * 1.5, w, torch.device("cpu"))
    bench.barrier(w)
    q.put((r, w, bench.rank_rows(r), t))
    dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1] and all(r[1] == 2 for r in res)
    starts = [r[2] for r in res]
    assert starts == [0, 4096]           # disjoint 4096-row windows, weak scaling
    assert all(r[3] == 3.0 for r in res)  # max over ranks


def test_bench_arguments():
    import bench
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and a.impl == "ours"
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "1"])
