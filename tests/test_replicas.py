"""The multi-GPU form is replicas only: N independent copies of the decode step, no
data-path collective.  The host logic that combines them (the slowest rank's time
bounds the job, the value sums the ranks' units) runs here on world-size-2 gloo
ranks on the CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [40.0, 55.0][rank]   # the second rank is slower
    total, value = bench.replica_rate(local_ms, 1000, dist, device="cpu")
    out[rank] = (total, value)
    dist.destroy_process_group()


def test_replica_rate_two_gloo_ranks():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        total, value = res[rank]
        assert total == 55.0                       # every rank sees the slowest time
        assert value == pytest.approx(2 * 1000 / 0.055)


def test_replica_rate_single_process():
    import bench
    total, value = bench.replica_rate(50.0, 1000)
    assert total == 50.0 and value == pytest.approx(1000 / 0.05)
