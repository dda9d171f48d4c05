"""The multi-GPU path is replicas only (every (sequence, head) unit is
independent; there is no exchange step), so its one collective is the
benchmark's max-over-ranks timing.  Checked here with two gloo ranks on CPU."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [30.0, 50.0][rank]          # rank 1 is the straggler
    ms, value = bench.aggregate(local_ms, steps=10, tokens_per_step=1000, world=world, device="cpu")
    out[rank] = (ms, value)
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    for rank in range(world):
        ms, value = out[rank]
        assert ms == 5.0                     # 50 ms / 10 steps, the slowest rank
        assert abs(value - 2 * 1000 / 5e-3) < 1e-6  # tokens of both ranks over that time
