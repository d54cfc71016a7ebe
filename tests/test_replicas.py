"""The N > 1 path of bench.py on CPU, as two gloo ranks.

The KDA path has no exchange step, so more GPUs run independent replicas:
each rank draws its own inputs, the timed region is closed by a barrier, the
job's time is the slowest rank's, the value counts every rank's tokens, and
only rank 0 prints (for the reference arm, rank 0 alone runs the oracle
sample).  These are the host-side pieces of that path; the GPU kernels are
the same on every rank.
"""
import contextlib
import io
import json
import os
import socket
import types

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(10.0 + rank, dist)
        rate = bench.job_rate(1000, world, ms)
        slots = bench.ki.slot_table(bench.replica_rng(rank), bench.B, bench.P).tolist()
        out = io.StringIO()
        with contextlib.redirect_stdout(out):
            bench.run_reference(types.SimpleNamespace(steps=1, warmup=0, gpus=world),
                                rank, world)
        dist.barrier()
        q.put((rank, ms, rate, slots, out.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_replica_logic():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(q.get(timeout=180) for _ in range(2))
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    (_, ms0, rate0, s0, out0), (_, ms1, rate1, s1, out1) = res
    assert ms0 == ms1 == 11.0                      # the slowest rank's time
    assert rate0 == rate1 == pytest.approx(2 * 1000 / 0.011)
    assert s0 != s1                                # independent replicas
    line = json.loads(out0.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert out1 == ""                              # rank 1 prints nothing


def test_single_rank_helpers_without_a_group():
    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.job_rate(500, 1, 2.0) == pytest.approx(250000.0)
    a = bench.ki.slot_table(bench.replica_rng(0), bench.B, bench.P)
    b = bench.ki.slot_table(bench.replica_rng(0), bench.B, bench.P)
    assert (a == b).all()                          # seeded: reproducible
