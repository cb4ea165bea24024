"""The bench's multi-rank bookkeeping on CPU: two gloo ranks, each timing its own chunk; the job's time is the slowest
rank's and the job's throughput counts every rank's pairs (weak scaling, no collective on the data path)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    elapsed = [3.0, 5.0][rank]                 # rank 1 is the slow one
    out[rank] = bench.max_over_ranks(elapsed, dist, "cpu")
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_over_ranks():
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        assert dict(out) == {0: 5.0, 1: 5.0}
