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
        args = bench.argparse.Namespace(steps=2, warmup=1, config="tiny", impl="reference",
                                         dtype="bf16")
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
