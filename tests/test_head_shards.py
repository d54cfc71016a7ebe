"""Head-sharded split of the path over ranks, as two gloo ranks on CPU.

Each rank owns a contiguous head range (recurrent_kda_state_gb300.sharding)
and serves those heads alone: its own state pool and ring, the token tensors'
columns of its heads.  Nothing crosses ranks on the path.  The checks are the
partition (every head exactly once, balanced) and that the ranks' results,
gathered along the head axis, are the one-rank results bit for bit -- run
here through the oracle's session, which stands in for each rank's library
calls on the CPU.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import kda_inputs as ki
import oracle
from recurrent_kda_state_gb300.sharding import gather_heads, head_range, shard_heads

B, H, D, P, T, STEPS = 3, 6, 8, 7, 4, 3


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _schedule():
    """The same seeded steps on every rank: prefill, then verify + commit."""
    rng = np.random.default_rng(4242)
    slots = ki.slot_table(rng, B, P)
    pre = ki.gen_tokens(rng, [5, 9, 3], H, D)
    steps = [(ki.gen_tokens(rng, [T] * B, H, D), ki.accepted_uniform(rng, B, T))
             for _ in range(STEPS)]
    return slots, pre, steps


def _serve(h0, h1):
    """Outputs and final pool of heads [h0, h1) through the session."""
    slots, pre, steps = _schedule()
    sub = lambda tok: dict({n: shard_heads(tok[n], h0, h1) for n in  # noqa: E731
                            ("q", "k", "v", "alpha", "beta")},
                           cu_seqlens=tok["cu_seqlens"])
    sess = oracle.OracleSession(P, h1 - h0, D, D)
    outs = [sess.prefill(sub(pre), slots, ckpt_every=4,
                         ckpt_slots=np.full((B, 1), -1))[0]]
    for tok, acc in steps:
        outs.append(sess.verify(sub(tok), slots))
        sess.commit(acc, slots)
    return np.concatenate(outs, axis=0), sess.pool


def _rank(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        h0, h1 = head_range(H, world, rank)
        o, pool = _serve(h0, h1)
        # ranks' head counts are equal here (H % world == 0): gather directly
        os_ = [torch.zeros_like(torch.from_numpy(o)) for _ in range(world)]
        ps_ = [torch.zeros_like(torch.from_numpy(pool)) for _ in range(world)]
        dist.all_gather(os_, torch.from_numpy(o))
        dist.all_gather(ps_, torch.from_numpy(pool))
        if rank == 0:
            q.put((gather_heads([t.numpy() for t in os_]),
                   gather_heads([t.numpy() for t in ps_])))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_head_range_partitions_every_head_once():
    for heads in (1, 6, 8, 32, 33, 7):
        for world in (1, 2, 3, 8):
            ranges = [head_range(heads, world, r) for r in range(world)]
            covered = [h for a, b in ranges for h in range(a, b)]
            assert covered == list(range(heads))
            sizes = [b - a for a, b in ranges]
            assert max(sizes) - min(sizes) <= 1
    assert head_range(32, 8, 3) == (12, 16)
    with pytest.raises(ValueError):
        head_range(8, 2, 2)


def test_shard_and_gather_are_inverse():
    x = np.arange(5 * 6 * 4).reshape(5, 6, 4)
    parts = [shard_heads(x, *head_range(6, 3, r)) for r in range(3)]
    assert all(p.flags["C_CONTIGUOUS"] for p in parts)
    assert np.array_equal(gather_heads(parts), x)
    t = torch.from_numpy(x.copy())
    tp = [shard_heads(t, *head_range(6, 4, r)) for r in range(4)]
    assert all(p.is_contiguous() for p in tp)
    assert torch.equal(gather_heads(tp), t)


def test_two_gloo_ranks_head_shards_equal_one_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        o_all, pool_all = q.get(timeout=180)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    o_ref, pool_ref = _serve(0, H)
    assert np.array_equal(o_all, o_ref)
    assert np.array_equal(pool_all, pool_ref)
