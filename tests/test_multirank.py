"""The multi-GPU benchmark path on CPU: two gloo ranks, each with its own
batch, aggregate work by sum and time by max (weak scaling, no data-path
collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    work, ms = bench.aggregate(1e12 * (rank + 1), 2.0 + rank, world)
    out[rank] = (work, ms)
    dist.barrier()
    dist.destroy_process_group()


def test_aggregate_two_ranks():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        work, ms = out[r]
        assert work == pytest.approx(3e12)
        assert ms == pytest.approx(3.0)


def test_single_rank_passthrough():
    import bench
    assert bench.aggregate(5.0, 7.0, 1) == (5.0, 7.0)


def test_work_accounting():
    import bench
    # causal bottom-right pairs: Lq = Lk = 4 -> 1+2+3+4
    assert bench.causal_pairs(4, 4) == 10
    # Lq > Lk: rows 0..1 see nothing, then 1, 2
    assert bench.causal_pairs(4, 2) == 3
    # headline workload: 68.75 GFLOP of unmasked work
    assert bench.dense_flops(4, 16, 2048, 2048, 128, True) == pytest.approx(68.753e9, rel=1e-3)
