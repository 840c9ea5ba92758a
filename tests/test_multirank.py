"""The N > 1 path of the benchmark on CPU: two gloo ranks (no GPU).

Every (batch, layer, KV head) is independent, so the path shards with no data-path collective;
the only exchange is the timing: the job's time is the slowest rank's, and the whole-job
throughput counts every rank's tokens (weak scaling).  The reference arm runs on rank 0 only.
"""
import contextlib
import io
import os
import socket
import sys
import types

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # per-rank timings (ms): elapsed, e2e, decode; rank r is slower in the first one
        mine = [10.0 + rank, 20.0 - rank, 5.0 * (rank + 1)]
        q.put((rank, bench.dist_env(), bench.max_over_ranks(mine, torch.device("cpu"))))
    finally:
        dist.destroy_process_group()


def test_timings_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    by_rank = {r: (env, t) for r, env, t in got}
    for r in (0, 1):
        env, t = by_rank[r]
        assert env == (r, 2, r)
        assert t == [11.0, 20.0, 10.0], "every rank sees the slowest rank's times"


def test_job_throughput_is_weak_scaling():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.job_tokens_per_s(16, 400, 1, 1000.0)
    two = bench.job_tokens_per_s(16, 400, 2, 1000.0)
    assert one == pytest.approx(6400.0) and two == pytest.approx(2 * one)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    out = io.StringIO()
    args = types.SimpleNamespace(workload="streaming", steps=1, warmup=3)
    with contextlib.redirect_stdout(out):
        assert bench.run_reference(args) is None
    assert out.getvalue() == "", "a non-zero rank prints nothing and does no work"


def test_clock_samples_are_dated_by_their_own_timestamps():
    """Samples inside the timed region count; a region shorter than the sampling period takes
    the samples next to it; hardware slowdowns are reported."""
    sys.path.insert(0, ROOT)
    import bench
    import datetime
    c = bench.ClockSampler(0)
    base = datetime.datetime(2026, 1, 2, 3, 4, 5)

    def line(dt_s, sm, slow="Not Active"):
        ts = (base + datetime.timedelta(seconds=dt_s)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return f"{ts}, {sm}, 2070, 900.0, {slow}, Not Active, Not Active, Not Active\n"

    c.proc = types.SimpleNamespace(stdout=io.StringIO(
        line(0.0, 1500) + line(0.2, 2070) + line(0.4, 2070, "Active") + line(0.6, 1980)))
    c._read()
    t0 = base.timestamp()
    c.window(t0 + 0.1, t0 + 0.5)
    got = c.summary()
    assert got["samples"] == 2 and got["sm_mhz"] == 2070.0 and got["reasons"] == ["hw_slowdown"]
    c.window(t0 + 0.62, t0 + 0.7)            # no sample inside: the nearest ones
    got = c.summary()
    assert got["samples"] >= 1 and 1980.0 <= got["sm_mhz"] <= 2070.0
