"""Multi-rank host logic of the benchmark, on CPU with two gloo ranks.

Each rank runs its own batch (independent sequences, no data-path collective); the step
time reported is the slowest rank's, and the whole-job throughput counts every rank's
tokens. Only rank 0 prints the reference arm's line; the other ranks exit without work.
"""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, per_rank_ms, out_dir):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(per_rank_ms[rank], world, "cpu")
        tput = bench.job_throughput(4, world, ms)
        # the reference arm: rank 0 alone prints; other ranks return without work
        buf = io.StringIO()
        if rank != 0:
            with redirect_stdout(buf):
                bench.run_reference(type("A", (), {"warmup": 0, "steps": 1, "gpus": world})())
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as fh:
            json.dump({"ms": ms, "tput": tput, "printed": buf.getvalue()}, fh)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step(tmp_path):
    world = 2
    per_rank_ms = [0.25, 0.40]
    mp.start_processes(_rank_main, args=(world, _free_port(), per_rank_ms, str(tmp_path)),
                       nprocs=world, join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    for r in res:
        assert r["ms"] == pytest.approx(0.40)
        # 4 tokens per rank per step, 2 ranks, over the slowest rank's 0.40 ms
        assert r["tput"] == pytest.approx(8 / 0.40e-3)
    assert res[1]["printed"] == ""


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(0.123, 1) == 0.123
    assert bench.job_throughput(4, 1, 0.1) == pytest.approx(40000.0)
