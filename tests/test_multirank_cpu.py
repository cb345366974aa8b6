"""The benchmark's multi-rank plumbing on CPU, two ranks over gloo.

`bench.py --gpus N` runs one replica per rank (every unit of work is
independent, so there is no data-path collective): the ranks only meet at
barriers around the timed region and in one all-reduce that takes the slowest
rank's time; rank 0 alone prints the line, and in the reference arm the other
ranks return without work.  These checks need no GPU.
"""
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench

    w, r, local = bench.dist_env()
    dist = bench.init_dist(w, local)
    bench.barrier(dist)
    slowest = bench.max_over_ranks(dist, 1.5 * (r + 1))

    class Args:
        steps, warmup, gpus = 1, 0, world

    ref = bench.run_reference(Args, r) if r != 0 else "rank 0 not run here"
    bench.barrier(dist)
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"world": w, "rank": r, "backend": "gloo", "slowest": slowest, "ref_is_none": ref is None}, f)


def test_two_ranks_gloo_barrier_and_max_over_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    for r in range(world):
        res = json.load(open(tmp_path / f"rank{r}.json"))
        assert res["world"] == world and res["rank"] == r
        assert res["slowest"] == pytest.approx(3.0)      # max over ranks of 1.5 * (rank + 1)
        if r != 0:
            assert res["ref_is_none"]                    # reference arm: only rank 0 works
