"""The bench's multi-GPU host logic on the CPU: two ranks over gloo
(127.0.0.1).  Replicas only: each rank runs the whole workload, the job time
is the slowest rank's (one MAX all-reduce), the value is world x bytes over
that time; the reference arm runs on rank 0 alone."""

import io
import json
import multiprocessing as mp
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (world, rank, rank)
        t = bench.max_over_ranks(dist, 1.0 + 0.5 * rank)
        dist.barrier()
        buf = io.StringIO()
        with redirect_stdout(buf):
            rc = bench.main(["--impl", "reference", "--gpus", str(world), "--steps", "1", "--warmup", "0"])
        q.put((rank, t, rc, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_ranks_over_gloo():
    pytest.importorskip("torch")
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    for _ in range(world):
        r, t, rc, out = q.get(timeout=240)
        got[r] = (t, rc, out)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got[0][0] == got[1][0] == 1.5          # the slowest rank's time on every rank
    assert got[0][1] == got[1][1] == 0
    assert got[1][2] == ""                        # the reference arm prints on rank 0 only
    line = json.loads(got[0][2].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0


def test_whole_job_rate():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.whole_job_gbs(4, 10**9, 3, 2.0) == pytest.approx(6.0)
    assert bench.max_over_ranks(None, 3.25) == 3.25
