"""The direct per-position snapshot design (the ablation baseline that
ReplaySSM replaces) against the fp64 oracle and against ReplaySSM itself.

Snapshot t of a sequence is, by definition, the committed state after its
first t + 1 drafted tokens, so the oracle's commit of t + 1 tokens is the
expected value.  Both designs advance the state with the same step routine,
so the state a snapshot commit installs must equal, bit for bit, the state a
ReplaySSM commit of the same count rebuilds.
"""
import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle
from kda_gpu import (assert_outputs, assert_states, device_batch,
                     from_gpu_states, i32, to_gpu_states)
from recurrent_kda_state_gb300 import kda as K

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_error_word():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    K.kda_get_device_error()
    yield


def _random_states(rng, P, H, d, std=0.3):
    """Initial pool in the oracle orientation [P][H][d_k][d_v]."""
    return rng.standard_normal((P, H, d, d)) * std


def _tt(dtype):
    return torch.bfloat16 if dtype == "bf16" else torch.float32


@pytest.mark.parametrize("d,dtype,max_T", [(128, "bf16", 8), (128, "bf16", 16),
                                           (32, "f32", 5), (16, "f32", 4)])
def test_snapshots_outputs_and_commit_vs_oracle(d, dtype, max_T):
    """Several steps of verify-with-snapshots + snapshot commit with ragged
    draft counts (0 and max_T included): outputs, every written snapshot and
    the committed pool against the oracle; unwritten snapshot entries and
    slots outside the table keep their bytes."""
    rng = np.random.default_rng(300 + d + max_T)
    B, H, P = 6, 4, 11
    slots_np = ki.slot_table(rng, B, P)
    slots = i32(slots_np)
    S0 = _random_states(rng, P, H, d)
    pool = K.StatePool(to_gpu_states(S0).cuda())
    sess = oracle.OracleSession(P, H, d, d, init=S0)
    snaps = K.snapshot_buffer(B, max_T, pool)
    others = [s for s in range(P) if s not in set(slots_np.tolist())]
    keep = pool.data[others].clone()
    for step in range(3):
        lens = [max_T, 0, 1, max_T - 1, 2, max_T // 2 + 1]
        if step % 2:
            lens = lens[::-1]
        tok = ki.round_to(ki.gen_tokens(rng, lens, H, d), dtype)
        a = np.array([rng.integers(0, n + 1) for n in lens], dtype=np.int32)
        a[lens.index(max_T)] = max_T
        snaps.view(torch.int32).fill_(0x7fc00001)   # sentinel NaN
        tb = device_batch(tok, dtype)
        before = sess.pool[slots_np].copy()
        K.kda_verify_snapshot(tb, max_T, pool, slots, snaps)
        o_ref = sess.verify(tok, slots_np)
        assert_outputs(tb.o.cpu().numpy(), o_ref)
        cu = tok["cu_seqlens"]
        for i, n in enumerate(lens):
            seg = {k: tok[k][cu[i]:cu[i + 1]] for k in ("q", "k", "v", "alpha", "beta")}
            cu1 = np.array([0, n], dtype=np.int32)
            for t in range(n):
                want = oracle.commit(cu1, seg["q"], seg["k"], seg["v"], seg["alpha"],
                                     seg["beta"], np.array([t + 1], dtype=np.int32),
                                     before[i][None])[0]
                assert_states(from_gpu_states(snaps[i, t]), want)
            untouched = snaps[i, n:].view(torch.int32)
            assert bool((untouched == 0x7fc00001).all())
        K.kda_commit_snapshot(i32(a), slots, pool, snaps)
        sess.commit(a, slots_np)
        for s_ in slots_np:
            assert_states(from_gpu_states(pool.data[s_]), sess.pool[s_])
    torch.cuda.synchronize()
    assert pool.data[others].view(torch.int32).equal(keep.view(torch.int32))
    assert K.kda_get_device_error() == 0


@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (64, "f32")])
def test_snapshot_commit_is_bit_identical_to_replay_commit(d, dtype):
    """Same states and drafts, every accepted count 0..T: the snapshot the
    direct design commits equals the state the ReplaySSM ring rebuilds, bit
    for bit; the two designs' outputs agree within the output tolerance."""
    rng = np.random.default_rng(41 + d)
    T, H, P = 8, 4, 20
    B = T + 1
    slots_np = ki.slot_table(rng, B, P)
    slots = i32(slots_np)
    start = to_gpu_states(_random_states(rng, P, H, d)).cuda()
    poolA = K.StatePool(start.clone())
    poolB = K.StatePool(start.clone())
    ring = K.ReplayRing(P, H, d, T, _tt(dtype))
    snaps = K.snapshot_buffer(B, T, poolB)
    for step in range(2):
        tok = ki.round_to(ki.gen_tokens(rng, [T] * B, H, d), dtype)
        a = rng.permutation(np.arange(B, dtype=np.int32))   # 0..T, shuffled
        tA, tB = device_batch(tok, dtype), device_batch(tok, dtype)
        K.kda_verify(tA, T, poolA, slots, ring)
        K.kda_commit(i32(a), slots, poolA, ring)
        K.kda_materialize(slots, poolA, ring)
        K.kda_verify_snapshot(tB, T, poolB, slots, snaps)
        K.kda_commit_snapshot(i32(a), slots, poolB, snaps)
        torch.cuda.synchronize()
        assert torch.equal(poolA.data, poolB.data)
        assert_outputs(tA.o.cpu().numpy(), tB.o.cpu().numpy())
    assert K.kda_get_device_error() == 0


def test_snapshot_commit_zero_keeps_state_bytes():
    rng = np.random.default_rng(52)
    B, H, d, P, T = 4, 4, 128, 7, 8
    slots = i32(ki.slot_table(rng, B, P))
    pool = K.StatePool(to_gpu_states(_random_states(rng, P, H, d)).cuda())
    before = pool.data.clone()
    snaps = K.snapshot_buffer(B, T, pool)
    for _ in range(2):
        tok = ki.round_to(ki.gen_tokens(rng, [T] * B, H, d), "bf16")
        K.kda_verify_snapshot(device_batch(tok, "bf16"), T, pool, slots, snaps)
        K.kda_commit_snapshot(i32([0] * B), slots, pool, snaps)
    torch.cuda.synchronize()
    assert pool.data.view(torch.int32).equal(before.view(torch.int32))
    assert K.kda_get_device_error() == 0


def test_snapshot_device_errors_skip_rows():
    """Data-dependent errors: an accepted count above max_T, a slot outside
    the pool, a segment longer than max_T.  The affected rows are skipped
    (state untouched), the others run, and the error bits are set."""
    rng = np.random.default_rng(53)
    B, H, d, P, T = 3, 2, 64, 5, 4
    slots_np = np.array([0, 3, 1], dtype=np.int32)
    pool = K.StatePool(to_gpu_states(_random_states(rng, P, H, d)).cuda())
    start = pool.data.clone()
    snaps = K.snapshot_buffer(B, T, pool)
    tok = ki.round_to(ki.gen_tokens(rng, [T] * B, H, d), "bf16")
    K.kda_verify_snapshot(device_batch(tok, "bf16"), T, pool, i32(slots_np), snaps)
    assert K.kda_get_device_error() == 0
    K.kda_commit_snapshot(i32([T + 1, 2, 1]), i32(slots_np), pool, snaps)
    assert K.kda_get_device_error() == K.KDA_DERR_ACCEPT
    assert torch.equal(pool.data[0], start[0])        # a > max_T: skipped
    assert torch.equal(pool.data[3], snaps[1, 1])     # the others committed
    assert torch.equal(pool.data[1], snaps[2, 0])
    K.kda_commit_snapshot(i32([1, 1, 1]), i32([0, P, 1]), pool, snaps)
    assert K.kda_get_device_error() == K.KDA_DERR_SLOT
    long_tok = ki.round_to(ki.gen_tokens(rng, [T + 1, 1, 1], H, d), "bf16")
    K.kda_verify_snapshot(device_batch(long_tok, "bf16"), T, pool, i32(slots_np), snaps)
    assert K.kda_get_device_error() == K.KDA_DERR_DEPTH
