"""The multi-GPU form of the path is N independent replicas (no exchange step).  These CPU
tests run the benchmark's aggregation and the reference arm's rank handling as world-size-2
gloo process groups: the job time is the slowest rank's, the value counts every rank's work."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [10.0, 20.0][rank]
        value, total = bench.whole_job_value(local_ms, steps=5, flops_per_step=2e12, world=world,
                                             device="cpu")
        out[rank] = (value, total)
    finally:
        dist.destroy_process_group()


def test_whole_job_value_takes_slowest_rank_and_counts_all_work():
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    for rank in (0, 1):
        value, total = out[rank]
        assert total == 20.0  # the slowest rank's time
        # 2 ranks x 5 steps x 2 TFLOP in 20 ms = 1000 TFLOP/s
        assert value == pytest.approx(1000.0)


def test_single_rank_value_needs_no_process_group():
    value, total = bench.whole_job_value(4.0, steps=2, flops_per_step=1e12, world=1)
    assert total == 4.0 and value == pytest.approx(500.0)


def test_reference_arm_prints_on_rank_zero_only(capsys):
    class Args:
        steps, warmup, workload = 1, 3, "sgemm_256cube"

    assert bench.run_reference(Args(), rank=1, world=2) == 0
    assert capsys.readouterr().out == ""
    assert bench.run_reference(Args(), rank=0, world=2) == 0
    line = capsys.readouterr().out.strip()
    import json

    d = json.loads(line)
    assert d["impl"] == "reference" and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["n_gpus"] == 2
