"""The bench's multi-rank path on the CPU (gloo, world size 2).

The hot path does not shard across GPUs: N GPUs run N independent replicas
(one process each, no collective on the data path).  What the N > 1 path
does need -- process-group setup from the launcher's environment, the
barrier around the timed region, the max over ranks of the elapsed time, and
a single JSON line from rank 0 -- is checked here with two CPU processes.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    w, r, local = bench.dist_setup()
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    m = bench.max_over_ranks(w, 1.5 * (r + 1), "cpu")   # per-rank "elapsed" values 1.5 and 3.0
    bench.barrier(w)
    q.put((r, w, local, m))
    dist.destroy_process_group()


def test_dist_helpers_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 2, 0, 3.0), (1, 2, 1, 3.0)]       # both ranks see the max


@pytest.mark.timeout(600)
def test_reference_arm_under_torchrun_two_ranks():
    """`bench.py --impl reference` launched like the driver launches N > 1: rank 0 alone
    runs the oracle sample and prints one JSON line; the other rank exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "1", "--workload", "tiny"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
