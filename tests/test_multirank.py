"""The benchmark's multi-rank path on CPU: two gloo ranks (one process each),
as the replicas run under torchrun on GPUs.  Each rank times its own replica;
the step time is the slowest rank's and the value counts every rank's bytes."""
import json
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [12.5, 20.0][rank]                  # each rank's own timed region, ms
        slowest = bench.slowest_rank_ms(mine, dist, "cpu")
        value = bench.whole_job_gbs(world, 1_000_000_000, slowest / 10)
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"slowest": slowest, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_rank, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    for r in range(2):
        got = json.load(open(tmp_path / f"rank{r}.json"))
        assert got["slowest"] == 20.0                       # max over ranks, seen by every rank
        assert abs(got["value"] - 2 * 1e9 / 2e-3 / 1e9) < 1e-6   # 2 ranks x 1 GB in 2 ms per step


def test_reference_arm_runs_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        steps, warmup, gpus = 1, 1, 2

    bench.run_reference(Args(), rank=1, world=2)   # the other ranks exit without work
    assert capsys.readouterr().out == ""
