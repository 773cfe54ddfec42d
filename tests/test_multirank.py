"""Multi-rank host logic of the benchmark on CPU: two gloo ranks.

The decode shards (batch, KV head) units across ranks with no data-path exchange, so
the only cross-rank step is the timing: every rank's time is reduced by max and the
whole-job rate counts the units of all ranks.  The reference arm runs on rank 0 only."""

import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [3.0, 5.0][rank]  # rank 1 is the slower one
        worst = bench.max_over_ranks(local_ms, dist, "cpu")
        rate = bench.job_rate(1000, world, worst)

        class Args:
            steps, warmup = 1, 0

        buf = io.StringIO()
        if rank == 1:  # the reference arm must do nothing and print nothing off rank 0
            with redirect_stdout(buf):
                bench.run_reference(Args, rank, world)
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"worst": worst, "rate": rate, "ref_stdout": buf.getvalue()}, f)
    finally:
        dist.destroy_process_group()


def test_two_rank_max_time_and_job_rate(tmp_path):
    import torch.multiprocessing as mp
    port = free_port()
    mp.start_processes(worker, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn", join=True)
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for g in got:
        assert g["worst"] == pytest.approx(5.0)          # max over ranks, on every rank
        assert g["rate"] == pytest.approx(2 * 1000 / 5e-3)  # units of both ranks / slowest time
    assert got[1]["ref_stdout"] == ""


def test_single_process_helpers_without_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5, None, "cpu") == 7.5
    assert bench.job_rate(10, 1, 2.0) == pytest.approx(5000.0)

