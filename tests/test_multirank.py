"""The multi-rank host path on CPU: two gloo ranks (127.0.0.1).  Requests are independent,
so ranks run replicas with no collective on the data path; the only exchange is the
timing reduction (the slowest rank's time) and the whole-job rate built on it, and the
reference arm prints one line from rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, values, out_q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    from mla_latent_kv_17_gb300 import metrics
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m = metrics.max_over_ranks(values[rank], dist)
        rate = metrics.whole_job_rate(10.0, world, m)
        out_q.put((rank, m, rate))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    values = [3.5, 7.25]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, values, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[1] for g in got] == [7.25, 7.25]          # both ranks see the slowest time
    assert all(abs(g[2] - 10.0 * 2 / 7.25) < 1e-12 for g in got)


def test_single_process_needs_no_group():
    from mla_latent_kv_17_gb300 import metrics
    assert metrics.max_over_ranks(4.0) == 4.0
    assert metrics.whole_job_rate(6.0, 1, 2.0) == 3.0


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "3", "--ref-budget", "0.2",
           "--workload", "tiny_dense_b1_h16_l256"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
