"""The N > 1 path on the CPU: two gloo ranks.

The path shards into independent replicas (every (b, kv head) unit is independent; no collective on the data path),
so multi-rank runs exchange only control-plane values: a barrier before and after the timed region and the maximum
of the per-rank times.  These tests run that exchange with world size 2 on the host, and the reference arm of
``bench.py`` under torchrun, where rank 0 alone prints the JSON line and the other rank exits 0 without work.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(ws), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    got_ws, got_rank, _ = bench.dist_setup()
    bench.dist_barrier(got_ws)
    # per-rank times differ; every rank must see the largest (the whole job is as slow as its slowest replica)
    t = bench.dist_max(10.0 + 5.0 * rank, got_ws)
    bench.dist_barrier(got_ws)
    results[rank] = (got_ws, got_rank, t)
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_max_time():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_rank_main, args=(2, free_port(), results), nprocs=2, join=True, start_method="spawn")
        res = dict(results)
    assert res[0] == (2, 0, 15.0)
    assert res[1] == (2, 1, 15.0)


@pytest.mark.timeout(600)
def test_reference_arm_under_torchrun_prints_once_from_rank_0():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(free_port()), "bench.py", "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "0"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
