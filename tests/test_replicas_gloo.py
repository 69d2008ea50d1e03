"""Multi-GPU path of the bench on CPU: N independent replicas, no data
exchange; the job's throughput is all ranks' pairs over the slowest rank's
time. Run as two gloo ranks (no GPU)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r "took" 10*(r+1) ms and scored 1000*(r+1) pairs
    value, ms_max, total = bench.aggregate(10.0 * (rank + 1), 1000.0 * (rank + 1), world,
                                           device="cpu")
    out[rank] = (value, ms_max, total)
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_aggregate_with_max_time():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(world):
        value, ms_max, total = out[r]
        assert ms_max == 20.0                    # slowest rank
        assert total == 3000.0                   # all ranks' pairs
        assert value == pytest.approx(3000.0 / 0.020)
