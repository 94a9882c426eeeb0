"""The N>1 benchmark path on CPU: two gloo ranks, each a replica with its own timing; the
whole-job figure uses the slowest rank's time and all ranks' work (no data-path collective)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = 100.0 + 25.0 * rank                     # rank 1 is the slow one
    slowest = bench.max_over_ranks(local_ms, dist)
    out[rank] = (slowest, bench.whole_job_tflops(world, slowest, steps=4))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_replicas_take_slowest_rank(world):
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(world, port, out), nprocs=world, start_method="spawn")
        res = dict(out)
    import bench
    assert res[0][0] == res[1][0] == 125.0
    assert res[0][1] == pytest.approx(world * bench.GEMM_FLOPS / (125.0 / 4 * 1e-3) / 1e12)
    assert bench.max_over_ranks(3.5) == 3.5              # world of one: no collective
