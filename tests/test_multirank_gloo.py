"""The benchmark's multi-rank bookkeeping on CPU with two gloo ranks: the
job is timed as its slowest rank and every rank runs the same per-GPU
workload (weak scaling), so the whole-job value scales with the rank count."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, local_ms, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK="0")
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        assert bench.dist_env() == (rank, world, 0)
        total = bench.max_over_ranks(local_ms[rank])
        out[rank] = (total, bench.job_tflops(world, 10, 1e12, total))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    world, port = 2, _free_port()
    local_ms = [120.0, 150.0]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, local_ms, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        total, value = res[rank]
        assert total == pytest.approx(150.0)
        # 2 ranks x 10 steps x 1 TFLOP in 0.150 s
        assert value == pytest.approx(2 * 10 * 1.0 / 0.150)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_tflops(1, 4, 2e12, 1000.0) == pytest.approx(8.0)
