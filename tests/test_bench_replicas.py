"""bench.py's N-replica host logic on CPU: two gloo ranks (no GPU).

Every replica times its own all-reduce; the job's time is the slowest
replica's and its throughput counts every replica's bytes.  Under torchrun
the reference arm runs on rank 0 only; other ranks leave without work.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 2.0 if rank == 0 else 5.0
        slowest = bench.max_over_ranks(local_ms, dist)
        out[rank] = (slowest, bench.job_gbs(1e9, slowest, world))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    slowest, gbs = res[0]
    assert slowest == 5.0
    assert gbs == pytest.approx(2 * 1e9 / 5e-3 / 1e9)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.job_gbs(64e6, 1.0, 1) == pytest.approx(64.0)


def test_reference_arm_runs_on_rank_zero_only(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "1")

    class Args:
        steps, warmup, gpus = 5, 3, 2

    bench.reference_arm(Args, bench.WORKLOADS["p8_64MiB_fp32_ring_ddp_mean"], "p8_64MiB_fp32_ring_ddp_mean")
    assert capsys.readouterr().out == ""


def test_fit_alpha_beta_recovers_a_line():
    pts = [(n, 3e-6 + n / 500e9) for n in (1 << k for k in range(3, 31))]
    alpha, beta = bench.fit_alpha_beta(pts)
    assert alpha == pytest.approx(3e-6, rel=1e-3)
    assert 1 / beta == pytest.approx(500e9, rel=1e-6)


def _failing_pair(rank, port, mode, timeout_s, q):
    """Rank 1 fails in `mode` ("exit": leaves before the barrier; "absent":
    never reaches it); rank 0 reports what its barrier did and how long it
    took."""
    import time

    os.environ["MASTER_PORT"] = str(port)
    os.environ.pop("MASTER_ADDR", None)
    if rank == 1:
        bench.init_replicas(2, rank, timeout_s=timeout_s)
        if mode == "exit":
            os._exit(3)
        time.sleep(timeout_s * 4)        # absent: the parent ends this process
        os._exit(0)
    t0 = time.monotonic()
    try:
        # an early exit of rank 1 may already fail the set-up; that too is
        # the failure seen, not a hang
        d = bench.init_replicas(2, rank, timeout_s=timeout_s)
        t0 = time.monotonic()
        d.barrier()
        q.put(("completed", time.monotonic() - t0))
    except Exception as exc:             # gloo reports a lost or silent peer as an error
        q.put((type(exc).__name__, time.monotonic() - t0))
    q.close()
    q.join_thread()                      # the result is sent before the process ends
    os._exit(0)


@pytest.mark.parametrize("mode", ["exit", "absent"])
def test_a_failed_replica_ends_the_others_barrier(mode):
    """Failure detection on the host: the surviving rank's barrier ends with
    an error -- at once when the peer exits, after the process group's
    timeout when it never arrives -- and never blocks."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port, timeout_s = _free_port(), 5
    procs = [ctx.Process(target=_failing_pair, args=(r, port, mode, timeout_s, q)) for r in (0, 1)]
    for p in procs:
        p.start()
    try:
        outcome, seconds = q.get(timeout=120)
    finally:
        for p in procs:
            p.join(timeout=1)
            if p.is_alive():
                p.kill()                 # this test's own child, by its handle
                p.join(timeout=10)
    assert outcome != "completed"
    if mode == "exit":
        assert seconds < timeout_s               # the lost connection is seen at once
    else:
        assert timeout_s * 0.5 <= seconds < timeout_s * 3
