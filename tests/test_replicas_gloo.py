"""Multi-process host logic of the benchmark's replica mode, on CPU with gloo.

The hot path shards into independent (batch, head, tile) units with no data
exchange, so N GPUs run N independent replicas; the only collective is the
max-over-ranks of the timed region. These tests run two gloo ranks on the CPU.
"""
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
    try:
        import bench
        import workloads
        w = workloads.WORKLOADS[bench.WORKLOAD]
        # rank r pretends its timed region took (10 + 5 r) ms for 4 steps
        ms_step, tflops = bench.replica_throughput(10.0 + 5.0 * rank, 4, 1e12, world)
        x = workloads.make_inputs(w.with_(B=1, H=1, Nq=8, Nk=8), with_dO=False,
                                  seed=bench.replica_seed(w, rank))
        out[rank] = (ms_step, tflops, float(x["q"].float().sum()))
    finally:
        dist.destroy_process_group()


def test_two_replicas_use_the_slowest_rank_and_all_ranks_work():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    assert set(res) == {0, 1}
    slow_ms = (10.0 + 5.0 * (world - 1)) / 4
    for r in range(world):
        ms_step, tflops, _ = res[r]
        assert ms_step == pytest.approx(slow_ms)
        assert tflops == pytest.approx(1e12 * world / (slow_ms * 1e-3) / 1e12)
    # replicas draw different inputs
    assert res[0][2] != res[1][2]


def test_single_process_throughput_needs_no_process_group():
    import bench
    ms_step, tflops = bench.replica_throughput(8.0, 4, 2e12, 1)
    assert ms_step == 2.0 and tflops == pytest.approx(1000.0)
