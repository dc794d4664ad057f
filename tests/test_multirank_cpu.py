"""The replica path of bench.py with two ranks on CPU (gloo, 127.0.0.1): the
ranks agree on the slowest rank's time, the whole-job throughput counts every
rank's units, and the reference arm's non-zero ranks exit without work."""
import contextlib
import io
import json
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


def _rank(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        barrier, max_over_ranks = bench.rank_helpers(dist, torch.device("cpu"))
        barrier()
        slowest = max_over_ranks(10.0 + 3.0 * rank)   # rank 1 is the slower replica
        value = bench.job_throughput(world, 1000, slowest / 1e3)
        # the reference arm runs on rank 0 only: the others return without output
        printed = io.StringIO()
        with contextlib.redirect_stdout(printed):
            if rank != 0:
                bench.reference_arm(None)
        barrier()
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"slowest": slowest, "value": value, "printed": printed.getvalue()}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_replica(tmp_path):
    if not dist.is_gloo_available():
        pytest.skip("gloo backend not built")
    world, port = 2, _free_port()
    mp.start_processes(_rank, args=(world, port, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["slowest"] == 13.0
        assert r["value"] == pytest.approx(2 * 1000 / 0.013)
    assert res[1]["printed"] == ""


def test_single_process_helpers_are_no_ops():
    sys.path.insert(0, ROOT)
    import bench
    barrier, max_over_ranks = bench.rank_helpers(None, torch.device("cpu"))
    barrier()
    assert max_over_ranks(4.5) == 4.5
    assert bench.job_throughput(1, 100, 0.5) == 200.0
