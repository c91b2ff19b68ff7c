"""Host-side logic of the bench harness on CPU: the replica timing reduction
over ranks (world size 2, gloo, 127.0.0.1) and the reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist = bench.init_dist(world, "gloo")
    bench.barrier(dist)
    t = bench.max_over_ranks(dist, 10.0 + rank)  # the slowest replica decides
    q.put((rank, t))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 11.0), (1, 11.0)]


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(None, 3.5) == 3.5


def test_reference_arm_line():
    """`bench.py --impl reference` times the oracle and prints the contract's line."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3", "--ref-tokens", "1"],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "cpu_baseline", "e2e"):
        assert k in line
    assert line["value"] > 0 and line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_step_sizing():
    """The reference arm's default sample keeps the whole run near its budget:
    16 tokens a step for a short run, down to 1 token for the default 2000 steps."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.ref_tokens_for(20, 3, 0.04) == 16
    assert bench.ref_tokens_for(2000, 20, 0.04) == 1
    n = bench.ref_tokens_for(200, 10, 0.04)
    assert 1 <= n <= 16 and (200 + 10) * n * 0.04 <= bench.REF_BUDGET_S
