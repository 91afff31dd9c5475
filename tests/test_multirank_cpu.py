"""The benchmark's multi-rank host logic on CPU with two gloo ranks: the job
time is the slowest rank's, the value counts every rank's units, and the
reference arm prints from rank 0 only.  (One process per GPU under torchrun
runs independent replicas of the path: there is no data-path collective to
test beyond this timing reduction.)"""
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


def _rank_main(rank, ws, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                            world_size=ws)
    local_ms = [3.0, 5.5][rank]
    ms = bench.max_over_ranks(local_ms, ws, "cpu")
    value = bench.job_throughput(4096, ws, ms)
    dist.barrier()
    dist.destroy_process_group()
    with open(out % rank, "w") as f:
        json.dump({"ms": ms, "value": value}, f)


def test_two_gloo_ranks_take_the_slowest_time(tmp_path):
    pytest.importorskip("torch")
    import torch.multiprocessing as mp
    port = _free_port()
    out = str(tmp_path / "rank%d.json")
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = [json.load(open(out % r)) for r in range(2)]
    for r in res:
        assert r["ms"] == 5.5                              # the slower rank's time
        assert abs(r["value"] - 2 * 4096 / 5.5e-3) < 1e-6  # both ranks' tokens


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, 1, "cpu") == 2.5
    assert bench.job_throughput(10, 1, 2.0) == 5000.0


def test_reference_arm_prints_from_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], capture_output=True, text=True,
                       env=env, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
