"""The N > 1 launch path of bench.py on CPU: two ranks over gloo (127.0.0.1).

Every rank runs the same work (replicas: the requests are independent units),
so the job's throughput is world x steps over the slowest rank's time; the
ranks meet at a barrier around the timed region and take the maximum of their
times.  The reference arm runs on rank 0 only; other ranks exit at once.
"""
import contextlib
import importlib.util
import io
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, ms_local, steps, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK="0")
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        r, w, _ = b.dist_env()
        b.barrier(w)
        ms = b.max_over_ranks(ms_local[rank], w)
        b.barrier(w)
        q.put((r, w, ms, b.job_rate(ms, steps, w)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_both_ranks_work():
    pytest.importorskip("torch")
    world, steps = 2, 20
    ms_local = [12.5, 17.25]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, ms_local, steps, q))
             for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    assert [o[0] for o in out] == [0, 1] and all(o[1] == world for o in out)
    assert all(o[2] == max(ms_local) for o in out)
    expected = world * steps / (max(ms_local) / 1e3)
    assert all(abs(o[3] - expected) < 1e-9 for o in out)


def test_one_rank_is_the_identity():
    b = _bench()
    assert b.max_over_ranks(3.5, 1) == 3.5
    b.barrier(1)
    assert b.job_rate(500.0, 10, 1) == 20.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    b = _bench()
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
    called = []
    monkeypatch.setattr(b, "reference_arm", lambda *a, **k: called.append(a))
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        assert b.main() == 0
    assert buf.getvalue() == "" and not called
