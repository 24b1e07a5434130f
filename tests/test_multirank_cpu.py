"""Two gloo ranks on CPU exercise the benchmark's multi-rank logic: each rank
runs its own replica (weak scaling), tokens are summed and the step time is the
maximum over ranks; no collective touches the data path."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    assert bench.dist_info() == (world, rank, rank)
    tokens, secs = bench.aggregate_ranks(100.0 * (rank + 1), 0.5 + rank)
    bench.barrier()
    out[rank] = (tokens, secs)
    dist.destroy_process_group()


def test_two_rank_aggregation_sums_tokens_and_takes_max_time():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        assert out[r] == (300.0, 1.5)


def test_single_rank_aggregation_is_identity():
    import bench
    assert bench.aggregate_ranks(7.0, 2.0) == (7.0, 2.0)


def test_replica_workloads_differ_per_rank():
    """Each rank draws its own replica (seed offset by rank) with the same shape."""
    from paged_kv_attention_25_gb300 import workloads as wl
    a = wl.tiny_mixed(seed=1)
    b = wl.tiny_mixed(seed=1 + 1000)
    assert a.q.shape == b.q.shape and not (a.q == b.q).all()
