"""The N > 1 path of bench.py on CPU: ranks are independent replicas (the
GEMM has no exchange step), the job time is the slowest rank's, and the
whole-job value counts every rank's FLOPs.  world_size 2, gloo backend."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    out[rank] = bench.max_over_ranks(times[rank], dist)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    times = [12.5, 17.25]
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == 17.25


def test_whole_job_value_counts_every_replica():
    import bench
    # 2 ranks, 10 steps of 1 TFLOP each, slowest rank 20 ms in total
    assert bench.whole_job_tflops(1e12, 2, 10, 20.0) == pytest.approx(1000.0)
    assert bench.max_over_ranks(3.0, None) == 3.0


def test_reference_arm_prints_only_on_rank0(capsys, monkeypatch):
    import bench
    import gemm_inputs

    class A:
        gpus, steps, warmup = 2, 1, 0
    bench.run_reference(A(), gemm_inputs.WORKLOADS["square256_f16"], rank=1, world=2)
    assert capsys.readouterr().out == ""
