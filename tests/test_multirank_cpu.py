"""The benchmark's multi-rank path on CPU: two processes over gloo.

Each rank runs its own replica of the step (no exchange on the data path), so
the job's step time is the slowest rank's and the job's value is world x the
per-step bytes over that time.  The reference arm prints from rank 0 only.
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


def _rank_main(rank, world, port, out_path):
    import torch
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, local = bench.rank_env()
    ms = [0.030, 0.045][rank]                      # the ranks' own step times
    worst = bench.max_over_ranks(torch, ms, torch.device("cpu"), w)
    dist.barrier()
    dist.destroy_process_group()
    with open(out_path, "w") as f:
        json.dump({"rank": r, "world": w, "local": local, "worst": worst,
                   "value": bench.job_value(w, worst)}, f)


def test_two_ranks_take_the_slowest_step(tmp_path):
    port = _free_port()
    outs = [tmp_path / f"r{r}.json" for r in range(2)]
    code = ("import sys; sys.path.insert(0, %r); sys.path.insert(0, %r); "
            "import test_multirank_cpu as t; t._rank_main(int(sys.argv[1]), 2, %d, sys.argv[2])"
            % (ROOT, os.path.join(ROOT, "tests"), port))
    procs = [subprocess.Popen([sys.executable, "-c", code, str(r), str(outs[r])]) for r in range(2)]
    for p in procs:
        assert p.wait(timeout=120) == 0
    res = [json.loads(o.read_text()) for o in outs]
    import bench
    for r, d in enumerate(res):
        assert d["rank"] == r and d["world"] == 2 and d["local"] == r
        assert d["worst"] == pytest.approx(0.045)
        assert d["value"] == pytest.approx(2 * bench.LAYER_WEIGHT_BYTES / 0.045e-3 / 1e9)


def test_single_rank_needs_no_collective():
    import torch
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(torch, 0.021, torch.device("cpu"), 1) == 0.021
    assert bench.job_value(1, 0.021) == pytest.approx(bench.LAYER_WEIGHT_BYTES / 0.021e-3 / 1e9)


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
