"""The multi-rank path of bench.py on CPU: two gloo ranks on 127.0.0.1 (no GPU).

bench.py runs one replica per GPU (the operation has no exchange step between batches): the
only cross-rank steps are the barriers around the timed region and the max over ranks of the
step time; the job value is world x per-rank bytes / slowest step.  The reference arm prints
on rank 0 only.
"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        bench.barrier(w)
        step_ms = 1.0 + 0.5 * rank  # rank 1 is the slower one
        slowest = bench.reduce_max(step_ms, w)
        bench.barrier(w)
        q.put((r, local, slowest, bench.job_value(w, 1_000_000, slowest / 1e3)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step():
    torch = pytest.importorskip("torch")
    mp = torch.multiprocessing.get_context("spawn")
    q = mp.Queue()
    port = _free_port()
    procs = [mp.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.terminate()
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, (r, local, slowest, value) in enumerate(got):
        assert r == rank and local == rank
        assert slowest == 1.5
        assert value == pytest.approx(2 * 1_000_000 / 1.5e-3 / 1e9)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.25, 1) == 3.25
    assert bench.job_value(1, 2_000_000, 1e-3) == pytest.approx(2.0)


def test_reference_arm_prints_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), dict(workload="tiny", steps=2, warmup=3))()
    out = io.StringIO()
    with redirect_stdout(out):
        bench.run_reference(args)
    assert out.getvalue() == ""
