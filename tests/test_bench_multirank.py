"""bench.py's multi-rank logic on CPU: world_size-2 gloo process groups.

On GPUs each rank runs an independent replica of the GEMM (the path does not
shard), ranks meet at barriers around the timed region, the job time is the
slowest rank's, and rank 0 alone prints.  These tests run that logic with
the gloo backend and no GPU.
"""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, secs, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dist.barrier()
    m = bench.max_over_ranks(secs[rank])
    rate = bench.whole_job_rate(1000, 10, world, m)
    out.put((rank, m, rate))
    dist.barrier()
    dist.destroy_process_group()


def _free_port():
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_time_is_the_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    secs = [0.5, 2.0]
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, secs, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.0, 2.0]
    # 2 replicas x 10 steps x 1000 bytes in 2 s
    assert all(abs(r[2] - 2 * 10 * 1000 / 2.0 / 1e9) < 1e-15 for r in res)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.25) == 1.25


@pytest.mark.parametrize("rank,expect_line", [(1, False), (0, True)])
def test_reference_arm_prints_on_rank_zero_only(rank, expect_line):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    if not expect_line:
        assert lines == []
        return
    d = json.loads(lines[-1])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["unit"] == "GB/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["value"] > 0
