"""The multi-GPU path is replicas only: each rank decodes its own batch and no collective touches
the data path. The benchmark's whole-job aggregation (slowest rank's time, sum of tokens) is
checked here with two gloo ranks on CPU."""
import os
import socket

import torch.multiprocessing as mp


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank: int, world: int, port: int, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms, toks = bench.aggregate(10.0 + 5.0 * rank, 100.0 * (rank + 1), "cpu")
    out[rank] = (ms, toks)
    dist.destroy_process_group()


def test_replica_aggregation_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        assert out[0] == out[1] == (15.0, 300.0)
