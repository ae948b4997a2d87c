"""The multi-GPU path of bench.py is replicas only: each rank runs the same
layer step on its own GPU with no data-path collective, and the timings are
combined on the host (barrier, then the maximum over ranks).  This runs that
host logic as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank)})
    import bench
    d = bench.Dist()
    d.barrier()
    out[rank] = d.max(10.0 + rank)      # e.g. each rank's ms per step
    d.barrier()
    d.close()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_take_the_max():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(100)
            assert p.exitcode == 0
        assert dict(out) == {0: 11.0, 1: 11.0}
