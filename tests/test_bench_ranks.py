"""The multi-rank logic of bench.py on CPU: two gloo ranks (the data path shards by sequence
with no exchange, so only the timing reduction crosses ranks): the job time is the slowest
rank's and the throughput counts every rank's units."""

import os
import socket
import subprocess
import sys
import textwrap

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent("""
    import os, sys, json
    sys.path.insert(0, os.environ["KVQ_ROOT"])
    import bench
    rank, world, local = bench.dist_setup()
    ms_local = 100.0 * (rank + 1)          # rank 1 is the slow one
    ms, value = bench.aggregate(ms_local, 8 * 512, world, "cpu")
    bench.barrier(world)
    if rank == 0:
        print(json.dumps({"world": world, "ms": ms, "value": value}))
    import torch.distributed as dist
    dist.destroy_process_group()
""")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_weak_scaling(tmp_path):
    script = tmp_path / "ranks.py"
    script.write_text(SCRIPT)
    env = dict(os.environ, KVQ_ROOT=ROOT, KVQ_BENCH_BACKEND="gloo")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), str(script)]
    out = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=240)
    assert out.returncode == 0, out.stderr[-2000:]
    import json
    line = [ln for ln in out.stdout.splitlines() if ln.startswith("{")][-1]
    r = json.loads(line)
    assert r["world"] == 2
    assert r["ms"] == 200.0
    assert abs(r["value"] - 2 * 8 * 512 / 0.2) < 1e-6
