"""The multi-GPU path of the benchmark runs independent replicas (the path
shards over query tokens with no exchange step): every rank times the same
step, the slowest rank's time counts, and the whole-job throughput is the
tokens of all ranks over that time.  This host logic is checked here with two
gloo ranks on the CPU; only rank 0 runs the reference arm."""
import io
import os
import socket
import contextlib

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r reports fwd 10 + r ms and bwd 30 - r ms
        got = bench.max_over_ranks([10.0 + rank, 30.0 - rank, 40.0], "cpu")
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_times_are_the_slowest_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(world):
        assert results[r] == [11.0, 30.0, 40.0]


def test_single_process_values_pass_through():
    assert bench.max_over_ranks([1.5, 2.5], "cpu") == [1.5, 2.5]


def test_whole_job_throughput_counts_every_replica():
    assert bench.replica_throughput(65536, 1, 303.7) == pytest.approx(65536 / 0.3037, rel=1e-12)
    assert bench.replica_throughput(65536, 4, 303.7) == pytest.approx(4 * 65536 / 0.3037, rel=1e-12)


def test_reference_arm_runs_on_rank_0_only(monkeypatch):
    monkeypatch.setenv("RANK", "1")

    class Args:
        config, ref_rows, warmup, steps, gpus = 1, 2, 0, 1, 2
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        assert bench.run_reference(Args()) is None
    assert buf.getvalue() == ""
