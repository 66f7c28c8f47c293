"""The bench's multi-rank path on CPU: two gloo ranks on 127.0.0.1.

`bench.py --gpus N` under torchrun runs one independent replica of the
workload per rank (sequences are independent; nothing is exchanged on the data
path) and reports the whole job: all ranks' query tokens over the slowest
rank's step time.  These tests run that host logic with world size 2 without a
GPU: the max over ranks, the whole-job value, the per-rank replica seeds, and
the reference arm, which only rank 0 runs.
"""
import json
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        # rank r's own times: the max over ranks must be element-wise
        mine = [1.0 + rank, 5.0 - rank, 3.0]
        got = bench.max_over_ranks(dist, mine, "cpu")
        dist.barrier()
        res = {"max": got, "value": bench.whole_job_value(world, 4, got[0]), "seed": bench.replica_seed(2000, rank)}
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump(res, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_the_bench(tmp_path):
    import torch.multiprocessing as mp

    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["max"] == [2.0, 5.0, 3.0]  # the slowest rank's time, per entry
        # 2 ranks x 4 sequences per step, a step of 2.0 ms (the slowest rank)
        assert r["value"] == pytest.approx(world * 4 / 2.0e-3)
    # independent replicas: every rank draws its own workload
    assert res[0]["seed"] == 2000 and res[1]["seed"] != res[0]["seed"]


def test_single_process_needs_no_group():
    import bench

    assert bench.max_over_ranks(None, [1.5, 2]) == [1.5, 2.0]
    assert bench.whole_job_value(1, 1, 0.1) == pytest.approx(1e4)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
    assert bench.run_reference(bench.parse()) == 0
    assert capsys.readouterr().out == ""  # no line, no work: rank 0 prints the only one
