"""The multi-rank plumbing of bench.py on CPU: two gloo ranks on 127.0.0.1.

The hot path shards as independent replicas (no exchange step), so what N > 1 adds is the
launcher's environment, a barrier and the max over ranks of the timed region; rank 0 alone prints
(and alone runs the reference arm). These run here without a GPU.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, values, outdir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": "2",
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    world, r, local = bench.dist_setup()
    bench.barrier(world)
    m = bench.max_over_ranks(values[rank], world)
    bench.barrier(world)
    with open(os.path.join(outdir, f"rank{rank}.json"), "w") as f:
        json.dump({"world": world, "rank": r, "local": local, "max": m,
                   "backend": dist.get_backend()}, f)
    dist.destroy_process_group()


def test_two_gloo_ranks_barrier_and_max(tmp_path):
    import torch.multiprocessing as tmp
    values = [3.25, 7.5]
    tmp.spawn(_rank_main, args=(_free_port(), values, str(tmp_path)), nprocs=2, join=True)
    for rank in range(2):
        got = json.load(open(tmp_path / f"rank{rank}.json"))
        assert got["world"] == 2 and got["rank"] == rank and got["local"] == rank
        assert got["backend"] == "gloo"
        assert got["max"] == max(values)


def test_reference_arm_runs_on_rank0_only():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
