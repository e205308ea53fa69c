"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): every rank
builds its own replica (distinct seeds, same shapes) and the reported timing
is the max over ranks.  No GPU needed."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from compressed_paged_kv_gb300 import workloads as W
    wl = W.WORKLOADS["tiny"]
    st = W.build_cache(wl, "cpu", seed=bench.replica_seed(wl, rank))
    vals = bench.reduce_max([1.0 + rank, 10.0 - rank], world)
    out[rank] = (vals, float(st.k_pools[0].float().sum()), tuple(st.block_tables.shape))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_and_max_reduction():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    (v0, s0, shape0), (v1, s1, shape1) = out[0], out[1]
    assert v0 == v1 == [2.0, 10.0]
    assert shape0 == shape1
    assert s0 != s1  # distinct replicas


def test_single_rank_reduce_is_identity():
    import bench
    assert bench.reduce_max([3.0, 4.5], 1) == [3.0, 4.5]
