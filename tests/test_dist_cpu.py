"""Multi-process host logic of bench.py on CPU (gloo, world size 2).

The path shards as independent replicas (tokens are independent), so the only
cross-rank logic is the barrier around the timed region, the max over ranks of
the step time and rank 0 alone printing the JSON line.  No GPU is used.
"""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        mx = bench.max_over_ranks(10.0 + rank, world)
        args = bench.parse_args(["--steps", "2", "--warmup", "1", "--config", "tiny",
                                 "--impl", "reference", "--gpus", "2"])
        buf = io.StringIO()
        with redirect_stdout(buf):
            rc = bench.run_reference(args, world, rank)
        out_q.put((rank, mx, rc, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_max_and_only_rank0_prints():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in procs:
        rank, mx, rc, out = q.get(timeout=300)
        res[rank] = (mx, rc, out)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][0] == res[1][0] == 11.0
    assert res[0][1] == 0 and res[1][1] == 0
    line = json.loads(res[0][2].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert res[1][2].strip() == ""


def test_bench_spawns_its_own_ranks_when_no_launcher_did():
    """`bench.py --gpus 2` without torchrun starts two ranks itself; on CPU
    the reference arm runs (gloo): rank 0 prints one line for 2 GPUs."""
    import subprocess
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--config", "tiny", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["config"]["workload"] == "tiny"


def test_bench_refuses_more_gpus_than_visible():
    import subprocess
    env = {k: v for k, v in os.environ.items() if k != "WORLD_SIZE"}
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2",
                        "--config", "tiny"], capture_output=True, text=True, timeout=300,
                       env=env, cwd=ROOT)
    assert r.returncode == 1
    assert "needs 2 CUDA devices" in r.stdout
