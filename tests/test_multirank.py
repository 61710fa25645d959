"""The multi-GPU path of the benchmark is replicas only: every rank runs its
own batch, with no collective on the data path; the job's step time is the
slowest rank's and its throughput is the sum over replicas.  This checks that
host logic with two gloo ranks on the CPU."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from exact_attention_98_gb300.inputs import attention_inputs

        t = 3.0 + 2.0 * rank  # this rank's "step time"
        slowest = bench.max_over_ranks(t, "cpu")
        q = attention_inputs(1, 1, 8, 4, seed=bench.replica_seed(rank), with_dout=False)[0]
        gathered = [torch.empty_like(q) for _ in range(world)]
        dist.all_gather(gathered, q)
        distinct = not torch.equal(gathered[0], gathered[1])
        out[rank] = (slowest, distinct, bench.job_tflops(1e12, world, slowest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_replicas_and_max_time():
    world = 2
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    for rank in range(world):
        slowest, distinct, tflops = out[rank]
        assert slowest == 5.0  # max over ranks of 3 and 5
        assert distinct  # each replica draws its own batch
        assert tflops == pytest.approx(2 * 1e12 / 5e-3 / 1e12)


def test_single_process_max_is_identity():
    import bench

    assert bench.max_over_ranks(7.25) == 7.25
    assert bench.job_tflops(2e12, 1, 1.0) == pytest.approx(2000.0)


def test_reference_arm_only_on_rank_zero(monkeypatch, capsys):
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        gpus, steps, warmup = 2, 1, 1

    bench.reference_arm(Args())
    assert capsys.readouterr().out == ""
