"""The bench's multi-rank path on CPU: world_size-2 gloo ranks, max-over-ranks timing and the
whole-job throughput (independent replicas, no collective on the data path)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
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
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 2.0 + rank * 1.5          # rank 1 is the straggler
    m = bench.max_over_ranks(ms, torch.device("cpu"))
    out[rank] = (m, bench.job_tokens_per_s(64, world, m))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_timing_takes_the_slowest_rank():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn",
                       join=True)
    assert out[0] == out[1]
    ms, tps = out[0]
    assert ms == pytest.approx(3.5)
    assert tps == pytest.approx(64 * 2 / 3.5e-3)


def test_single_process_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(1.25, torch.device("cpu")) == 1.25
    assert bench.job_tokens_per_s(64, 1, 2.0) == pytest.approx(32000.0)
