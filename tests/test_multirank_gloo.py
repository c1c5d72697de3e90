"""The multi-GPU path of bench.py is replicas only: every rank runs the whole
step on its own GPU, then the ranks agree on the slowest step time and rank 0
reports tokens of all ranks over that time. This checks that logic with two
gloo ranks on the CPU (no GPU, no data-path collective)."""
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
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, lr, ws = bench.dist_env()
    assert (r, lr, ws) == (rank, rank, world)
    # rank 1 is the slow one for the device timing, rank 0 for e2e
    local = [100.0 + 50.0 * rank, 30.0 - 10.0 * rank]
    got = bench.max_over_ranks(local, "cpu", world)
    out[rank] = got + [bench.job_throughput(16384, world, got[0] / 200)]
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_replicas_agree_on_the_slowest_rank(world):
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(world):
        total_ms, e2e_ms, value = out[r]
        assert total_ms == 150.0 and e2e_ms == 30.0
        # 2 replicas x 16384 tokens over 0.75 ms per step
        assert value == pytest.approx(2 * 16384 / 0.75e-3)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks([1.5, 2.5], "cpu", 1) == [1.5, 2.5]
    assert bench.job_throughput(128, 1, 0.5) == pytest.approx(256000.0)
