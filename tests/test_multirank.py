"""The multi-GPU path of bench.py, on CPU with two gloo ranks: every rank
draws its own batch, the step time that counts is the maximum over ranks,
and the job's throughput is the sum over ranks (weak scaling, no collective
on the data path)."""
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
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from exact_attention_36_gb300.inputs import make_qkvdo

        bench.barrier(True)
        ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        ms_max = bench.max_over_ranks(ms, True)
        q, _, _, _ = make_qkvdo(1, 2, 64, 8, seed=rank)
        out[rank] = (ms_max, bench.job_tflops(world, 2e12, ms_max), float(q.float().sum()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_weak_scaling():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world,
                           start_method="spawn", join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0  # both ranks report the slowest rank's time
    assert res[0][1] == pytest.approx(2 * 2e12 / 15e-3 / 1e12)
    assert res[0][2] != res[1][2]  # each rank works on its own batch


def test_single_rank_paths_need_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, False) == 3.5
    assert bench.job_tflops(1, 1e12, 1000.0) == pytest.approx(1.0)
