"""bench.py at N > 1 runs N independent replicas of the workload (no exchange between them); the
only cross-rank steps are the timing barrier and the max over ranks. This checks that host
logic with two gloo ranks on the CPU."""
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    # replica r took 10 + r ms for 5 steps of 1e12 flops each
    ms, tflops = bench.replica_throughput(1e12, 5, 10.0 + rank, world)
    out[rank] = (ms, tflops)
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_replicas_report_whole_job_throughput():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    world, port = 2, _free_port()
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    # every rank agrees on the slowest replica's time and on the whole-job throughput
    for r in range(world):
        ms, tflops = res[r]
        assert ms == 11.0
        assert tflops == pytest.approx(2 * 5 * 1e12 / 11e-3 / 1e12)


def test_single_process_needs_no_process_group():
    import bench

    assert bench.replica_throughput(2e12, 4, 8.0, 1) == (8.0, pytest.approx(1000.0))
