"""The N > 1 path of the benchmark on CPU: two gloo ranks.

The layer is token-parallel (replicas, no exchange), so the only cross-rank
steps are the barriers around the timed region, the max over ranks of the
step time and the whole-job value; these run here with gloo, and the
reference arm runs under torchrun with rank 0 alone printing its line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(ws),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    class A:
        pass
    got_ws, got_rank, _ = bench.dist_setup(A())
    assert (got_ws, got_rank) == (ws, rank) and dist.get_backend() == "gloo"
    bench.barrier(ws)
    ms = 10.0 + 5.0 * rank                        # rank 1 is the slow one
    ms_max = bench.reduce_max(ms, ws)
    value = bench.whole_job_value(ws, 1000, ms_max)
    bench.barrier(ws)
    out.put((rank, ms_max, value))
    dist.destroy_process_group()


@pytest.mark.skipif(torch.cuda.is_available(), reason="the gloo leg is the CPU path")
def test_two_gloo_ranks_max_time_and_whole_job_value():
    ws = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(ws))
    for rank, ms_max, value in res:
        assert ms_max == 15.0                     # every rank sees the slowest rank
        assert value == pytest.approx(2 * 1000 / 0.015)   # both ranks' tokens / slowest time


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--config", "tiny"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, OMP_NUM_THREADS="1"))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    assert lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2
