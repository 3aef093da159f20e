"""The multi-GPU mode of bench.py is replicas only: each rank runs the whole
layer on its own tokens, the job time is the slowest rank's and the
throughput counts all ranks' tokens.  This checks that aggregation with two
gloo ranks on the CPU (no GPU, no data-path collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [7.5, 9.25][rank]                 # the second replica is slower
    ms, tok_s = bench.replica_throughput(local_ms, 16384, world)
    results[rank] = (ms, tok_s)
    dist.barrier()
    dist.destroy_process_group()


def test_replica_aggregation_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank, args=(world, port, results), nprocs=world, join=True)
        got = dict(results)
    for r in range(world):
        ms, tok_s = got[r]
        assert ms == 9.25                         # max over ranks
        assert tok_s == pytest.approx(2 * 16384 / 9.25e-3)


def test_single_rank_is_its_own_time():
    ms, tok_s = bench.replica_throughput(4.0, 1000, 1)
    assert ms == 4.0 and tok_s == pytest.approx(1000 / 4e-3)
