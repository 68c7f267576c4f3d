"""The benchmark's multi-rank host logic with two gloo ranks on the CPU:
process-group setup from the launcher's environment, the barrier, the
max-over-ranks timing reduction, replica aggregation, and the reference arm's
rank-0-only rule (other ranks exit 0 without work or output)."""
import io
import os
import socket
import sys
import contextlib

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_q):
    sys.path.insert(0, ROOT)
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch.distributed as dist

    import bench

    r, w, local = bench.dist_setup(world)
    bench.barrier(w)
    # every rank reports its own step time; the line uses the slowest rank
    t = bench.max_over_ranks(1.5 * (rank + 1), w)
    # replicas: each rank streams the same bytes, the job total is world x that
    per_rank_bytes = 1000.0
    total = w * per_rank_bytes / (t * 1e-3) / 1e9
    # the reference arm: rank != 0 returns 0 and prints nothing
    buf = io.StringIO()
    rc = None
    if rank != 0:
        with contextlib.redirect_stdout(buf):
            rc = bench.run_reference(type("A", (), {"steps": 1, "warmup": 0, "gpus": w})())
    bench.barrier(w)
    dist.destroy_process_group()
    out_q.put((r, w, local, t, total, rc, buf.getvalue()))


def test_two_gloo_ranks():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort()
    assert [r[0] for r in results] == [0, 1]
    for r, w, local, t, total, rc, out in results:
        assert w == 2 and local == r
        assert t == pytest.approx(3.0)  # the slower rank's time on both ranks
        assert total == pytest.approx(2 * 1000.0 / 3.0e-3 / 1e9)
    rank1 = results[1]
    assert rank1[5] == 0 and rank1[6] == ""
