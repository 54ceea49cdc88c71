"""Host-side pieces of bench.py: the multi-rank aggregation (2 gloo ranks on
CPU) and the reference arm (the oracle timed on the host cores)."""
import json
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t, u = bench.aggregate(10.0 + 5.0 * rank, 100.0 * (rank + 1), world)
        q.put((rank, t, u))
    finally:
        dist.destroy_process_group()


def test_aggregate_two_gloo_ranks():
    """Whole-job throughput = sum of the ranks' units / the slowest rank's time."""
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for _, t, u in res:
        assert t == 15.0 and u == 300.0


def test_reference_arm_prints_one_line():
    out = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
         "tiny", "--steps", "2", "--warmup", "1", "--ref-problems", "2"],
        capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_traffic_lookup_follows_source():
    sys.path.insert(0, ROOT)
    import bench
    t = bench.measured_traffic("llama8b_full", "gram_tc", 16384)
    assert t is None or t > 0
    assert bench.measured_traffic("llama8b_full", "no_such_kernel", 16) is None
    assert bench.measured_traffic("tiny", "gram_tc", 16) is None


def test_trace_interval_union():
    """The trace summary's busy time of a lane is the length of the union of
    its launches' intervals (overlapping and touching intervals merged)."""
    sys.path.insert(0, ROOT)
    import bench
    busy, merged = bench._busy([(0.0, 1.0), (0.5, 2.0), (3.0, 4.0), (4.0, 4.5), (6.0, 6.0)])
    assert merged == [[0.0, 2.0], [3.0, 4.5], [6.0, 6.0]]
    assert busy == pytest.approx(3.5)
    assert bench._busy([]) == (0, [])
