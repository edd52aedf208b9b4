"""Multi-GPU is replicas only (no data-path collective): the bench's
aggregation over ranks, exercised with two gloo ranks on the CPU."""
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


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms, toks = bench.aggregate_over_ranks(10.0 + 5.0 * rank, 256, torch.device("cpu"))
    out[rank] = (ms, toks)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_takes_the_slowest_rank_and_all_tokens():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
    assert out[0] == (15.0, 512) and out[1] == (15.0, 512)


def test_single_process_aggregation_is_identity():
    import bench
    assert bench.aggregate_over_ranks(3.5, 7, torch.device("cpu")) == (3.5, 7)
