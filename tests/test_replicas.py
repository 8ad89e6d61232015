"""The bench's multi-GPU path is replicas only (one layer per rank, no data-path
collective): the step time is the max over ranks and the whole-job value divides by the
number of replicas.  Checked here with two gloo ranks on CPU."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local = 100.0 + 50.0 * rank          # rank 1 is the slower replica
    out[rank] = (bench.max_over_ranks(local), bench.replica_value(bench.max_over_ranks(local), world))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_replicas_take_the_max_and_divide_by_world():
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    port = _free_port()
    mp.start_processes(_rank, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert out[0] == out[1] == (150.0, 75.0)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.replica_value(12.5, 1) == 12.5
