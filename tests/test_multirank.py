"""The multi-rank path of bench.py on CPU: world-size-2 gloo process groups.

Each rank serves its own batch of requests (weak scaling, no collective on
the data path); the only exchange is the timing reduction, a max over ranks
after a barrier.  These tests run that host logic with gloo on CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, values, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        got = bench.max_over_ranks(values[rank], world, "cpu")
        out[rank] = got
        # the ranks' request batches differ: their seeds and inputs differ
        out[world + rank] = bench.rank_seed(rank)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("values", [(3.5, 1.25), (1.0, 7.0)])
def test_max_over_ranks_two_gloo_ranks(values):
    world = 2
    out = torch.zeros(2 * world, dtype=torch.float64).share_memory_()
    mp.spawn(_worker, args=(world, _free_port(), values, out), nprocs=world, join=True)
    assert out[0].item() == max(values) and out[1].item() == max(values)
    assert out[2].item() != out[3].item()


def test_max_over_ranks_single_rank_is_identity():
    assert bench.max_over_ranks(2.75, 1, "cpu") == 2.75


def test_rank_batches_are_distinct_requests():
    from deepseek_sparse_attention_index_gb300 import inputs as I
    a = I.decode_sweep(2, 512, seed=bench.rank_seed(0))
    b = I.decode_sweep(2, 512, seed=bench.rank_seed(1))
    assert not torch.equal(a.q, b.q)
    assert not torch.equal(a.indexer["k_idx"], b.indexer["k_idx"])
