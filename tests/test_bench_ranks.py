"""The benchmark's multi-rank bookkeeping on CPU (gloo, world size 2).

With N GPUs the benchmark runs N independent replicas of the decode step (one
process per GPU; the layer does not shard across GPUs here), brackets the timed
region with barriers, takes the largest time over the ranks and reports the
whole-job rate (every rank's tokens over that time).  These tests run the same
helpers in two CPU processes.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as td  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    td.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.ranks_barrier(torch)
        my_time = 1.0 + 0.5 * rank  # rank 1 is the slower replica
        t = bench.max_over_ranks(torch, my_time)
        bench.ranks_barrier(torch)
        out[rank] = (t, bench.job_rate(world, 100, t))
    finally:
        td.destroy_process_group()


def test_max_over_ranks_and_job_rate_two_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0] == res[1] == (1.5, 2 * 100 / 1.5)


def test_helpers_without_process_group():
    import bench
    assert not td.is_initialized()
    bench.ranks_barrier(torch)  # no-op
    assert bench.max_over_ranks(torch, 2.5) == 2.5
    assert bench.job_rate(1, 10, 0.5) == 20.0


def test_traffic_hash_ignores_comments_only(tmp_path, monkeypatch):
    # the captured DRAM traffic is reported only while the decode sources match the
    # capture: a comment or blank-space edit keeps the hash, a code edit changes it
    import bench
    src = tmp_path / "k.cuh"
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "DECODE_SOURCES", ["k.cuh"])
    src.write_text("int f(int x) { return x + 1; }  // one\n")
    h0 = bench.decode_sources_sha1()
    src.write_text("/* doc */\nint f(int x)  {\n  return x + 1;\n}  // two\n")
    assert bench.decode_sources_sha1() == h0
    src.write_text("int f(int x) { return x + 2; }\n")
    assert bench.decode_sources_sha1() != h0
