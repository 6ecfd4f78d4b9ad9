"""Host-side multi-rank logic of bench.py on CPU: world size 2 over gloo.

Every box runs one GPU, so the N > 1 path is replicas (weak scaling, no
collective on the data path). What a multi-rank run adds is host logic: the
maximum of the per-rank step time, the whole-job aggregate, and the reference
arm running on rank 0 only. Those are exercised here with real gloo ranks.
"""

import io
import json
import os
import socket
import subprocess
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_q):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    # each rank's own step time; the job reports the slowest
    ms = bench.combine_ranks(1.5 + rank, world)
    value = bench.job_throughput(1e9, world, ms)
    # the reference arm runs on rank 0 only: other ranks leave at once, silently
    buf = io.StringIO()
    rc = None
    if rank != 0:
        class A:  # the arm reads only these fields before returning
            steps, warmup = 1, 3

        with redirect_stdout(buf):
            rc = bench.reference_arm(A, rank, world)
    dist.barrier()
    dist.destroy_process_group()
    out_q.put((rank, ms, value, rc, buf.getvalue()))


def test_two_ranks_max_time_and_job_throughput():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value, rc, out in res:
        assert ms == 2.5  # max over ranks of 1.5 and 2.5
        assert abs(value - 2 * 1e9 / 2.5e-3) < 1e-3 * value
    assert res[1][3] == 0 and res[1][4] == ""


@pytest.mark.timeout(300)
def test_reference_arm_prints_one_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "3"], capture_output=True, text=True, timeout=280, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.strip().splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
