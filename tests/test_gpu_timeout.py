"""Bounded device waits that run out, made to run out on purpose.

kda_set_wait_limit(0) makes every kernel's first bounded wait (a pipeline
stage of the verify kernel, a tensor-core completion or a staging copy of the
tensor-core prefill) give up at once.  Nothing faults or hangs: the kernel
sets KDA_DERR_TIMEOUT, stops taking work, waits (with its own fixed limit)
for the copies and MMAs it already started, releases its tensor memory and
exits.  The tests check what is left written -- nothing: outputs keep their
NaN poison, the pool and the ring keep their bytes -- and that the context
stays usable: with the default limit restored the same call gives the
oracle's results.
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
def _limit_restored():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    K.kda_set_wait_limit(-1)
    K.kda_get_device_error()
    yield
    K.kda_set_wait_limit(-1)
    K.kda_get_device_error()


def test_verify_wait_runs_out_writes_nothing():
    """The pipelined verify (d = 128, bf16, depth 8) with a zero wait limit,
    on a ring with pending accepted entries: TIMEOUT is set and outputs,
    states, ring payload and control words are untouched; then the default
    limit gives the oracle's outputs and states from the same inputs."""
    rng = np.random.default_rng(6100)
    B, H, P, T = 20, 16, 32, 8
    slots_np = ki.slot_table(rng, B, P)
    slots = i32(slots_np)
    init = (rng.standard_normal((P, H, 128, 128)) * 0.3).astype(np.float32)
    pool = K.StatePool(to_gpu_states(init).cuda())
    ring = K.ReplayRing(P, H, 128, T, torch.bfloat16)
    sess = oracle.OracleSession(P, H, 128, 128,
                                init=init.astype(np.float64))
    # one ordinary step so that the next verify has entries to replay
    tok0 = ki.round_to(ki.gen_tokens(rng, [T] * B, H, 128), "bf16")
    a0 = ki.accepted_uniform(rng, B, T)
    tb0 = device_batch(tok0, "bf16")
    K.kda_verify(tb0, T, pool, slots, ring)
    K.kda_commit(i32(a0), slots, pool, ring)
    sess.verify(tok0, slots_np)
    sess.commit(a0, slots_np)
    torch.cuda.synchronize()
    assert K.kda_get_device_error() == 0

    tok = ki.round_to(ki.gen_tokens(rng, [T] * B, H, 128), "bf16")
    tb = device_batch(tok, "bf16")
    snap = {n: getattr(ring, n).clone() for n in ("k", "v", "alpha", "beta", "ctrl")}
    pool_before = pool.data.clone()
    tb.o.fill_(float("nan"))
    K.kda_set_wait_limit(0)
    K.kda_verify(tb, T, pool, slots, ring)
    bits = K.kda_get_device_error()
    K.kda_set_wait_limit(-1)
    assert bits & K.KDA_DERR_TIMEOUT
    assert not bits & K.KDA_DERR_UNSAFE
    assert torch.isnan(tb.o).all()
    assert torch.equal(pool.data, pool_before)
    for n, t in snap.items():
        assert torch.equal(getattr(ring, n), t), n

    K.kda_verify(tb, T, pool, slots, ring)
    o_ref = sess.verify(tok, slots_np)
    assert_outputs(tb.o.cpu().numpy(), o_ref)
    K.kda_materialize(slots, pool, ring)
    for s in slots_np:
        assert_states(from_gpu_states(pool.data[s]), sess.pool[s])
    assert K.kda_get_device_error() == 0


@pytest.mark.parametrize("single_pass", [False, True], ids=["two_pass", "single_pass"])
def test_prefill_wait_runs_out_writes_nothing(single_pass):
    """The tensor-core prefill (both paths) with a zero wait limit: TIMEOUT
    is set; outputs, the state slot and the checkpoint slots are untouched;
    then the default limit gives the oracle's results."""
    rng = np.random.default_rng(6200 + int(single_pass))
    H, L, P = 8, 700, 6
    tok = ki.round_to(ki.gen_tokens(rng, [L], H, 128), "bf16")
    init = (rng.standard_normal((P, H, 128, 128)) * 0.02).astype(np.float32)
    pool = K.StatePool(to_gpu_states(init).cuda())
    slots, ck = i32([2]), i32([[4, 5]])
    tb = device_batch(tok, "bf16")
    tb.o.fill_(float("nan"))
    before = pool.data.clone()
    K.kda_set_wait_limit(0)
    K.kda_prefill_chunked(tb, pool, slots, chunk=64, ckpt_every=256, ckpt_slots=ck,
                          single_pass=single_pass)
    bits = K.kda_get_device_error()
    K.kda_set_wait_limit(-1)
    assert bits & K.KDA_DERR_TIMEOUT
    assert not bits & K.KDA_DERR_UNSAFE
    assert torch.isnan(tb.o).all()
    assert torch.equal(pool.data, before)

    K.kda_prefill_chunked(tb, pool, slots, chunk=64, ckpt_every=256, ckpt_slots=ck,
                          single_pass=single_pass)
    sess = oracle.OracleSession(P, H, 128, 128,
                                init=init.astype(np.float64))
    o_ref, _ = sess.prefill(tok, [2], ckpt_every=256, ckpt_slots=np.array([[4, 5]]))
    assert_outputs(tb.o.cpu().numpy(), o_ref)
    for s in (2, 4, 5):
        assert_states(from_gpu_states(pool.data[s]), sess.pool[s])
    assert K.kda_get_device_error() == 0


def test_verify_raw_wait_runs_out_writes_nothing():
    """The projection-space verify (two prep groups on alternate units) with
    a zero wait limit, on a ring with pending accepted entries: TIMEOUT is
    set and outputs, states, ring payload and control words are untouched;
    with the default limit the same call gives the oracle's outputs and
    states from the inputs the oracle prepared."""
    from test_gpu_verify_raw import raw_tokens_clear_of_ties
    rng = np.random.default_rng(6300)
    B, H, P, T = 12, 16, 24, 8
    slots_np = ki.slot_table(rng, B, P)
    slots = i32(slots_np)
    init = (rng.standard_normal((P, H, 128, 128)) * 0.05).astype(np.float32)
    pool = K.StatePool(to_gpu_states(init).cuda())
    ring = K.ReplayRing(P, H, 128, T, torch.bfloat16)
    sess = oracle.OracleSession(P, H, 128, 128, init=init.astype(np.float64))
    raw0, prep0 = raw_tokens_clear_of_ties(rng, [T] * B, H)
    a0 = ki.accepted_uniform(rng, B, T)
    K.kda_verify(device_batch(raw0, "bf16"), T, pool, slots, ring, raw=True)
    K.kda_commit(i32(a0), slots, pool, ring)
    sess.verify(prep0, slots_np)
    sess.commit(a0, slots_np)
    torch.cuda.synchronize()
    assert K.kda_get_device_error() == 0

    raw, prep = raw_tokens_clear_of_ties(rng, [T] * B, H)
    tb = device_batch(raw, "bf16")
    snap = {n: getattr(ring, n).clone() for n in ("k", "v", "alpha", "beta", "ctrl")}
    pool_before = pool.data.clone()
    tb.o.fill_(float("nan"))
    K.kda_set_wait_limit(0)
    K.kda_verify(tb, T, pool, slots, ring, raw=True)
    bits = K.kda_get_device_error()
    K.kda_set_wait_limit(-1)
    assert bits & K.KDA_DERR_TIMEOUT
    assert not bits & K.KDA_DERR_UNSAFE
    assert torch.isnan(tb.o).all()
    assert torch.equal(pool.data, pool_before)
    for n, t in snap.items():
        assert torch.equal(getattr(ring, n), t), n

    K.kda_verify(tb, T, pool, slots, ring, raw=True)
    o_ref = sess.verify(prep, slots_np)
    assert_outputs(tb.o.cpu().numpy(), o_ref)
    K.kda_materialize(slots, pool, ring)
    for s in slots_np:
        assert_states(from_gpu_states(pool.data[s]), sess.pool[s])
    assert K.kda_get_device_error() == 0
