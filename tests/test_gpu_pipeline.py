"""The pipelined verify kernel (d = 128, bf16, ring depth <= 8, <= 8 tokens
per row) against the oracle and against the per-unit verify kernel.

A ring of depth 9 sends the same calls to the per-unit kernel, so the two
kernels can be run on identical inputs: the states they commit come from the
same single-token step and must agree bit for bit; the drafted outputs take
different contraction paths and must each meet the output tolerance against
the oracle.  Unit counts below and above the SM count exercise one unit per
CTA and several units per CTA (both pipeline stages, both prep buffers).
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
    K.kda_set_wait_limit(-1)
    K.kda_get_device_error()
    yield


def _flow(seed, B, H, P, steps, max_T=8, spec_frac=0.75, init_std=0.3):
    """A seeded schedule: per step the drafted lengths (0..max_T for
    speculative rows, 1 for ordinary rows), the row kinds and the accepted
    lengths."""
    rng = np.random.default_rng(seed)
    slots_np = ki.slot_table(rng, B, P)
    init = (rng.standard_normal((P, H, 128, 128)) * init_std).astype(np.float32)
    sched = []
    for _ in range(steps):
        spec = rng.random(B) < spec_frac
        lens = [int(rng.integers(0, max_T + 1)) if s else 1 for s in spec]
        tok = ki.round_to(ki.gen_tokens(rng, lens, H, 128), "bf16")
        acc = np.array([rng.integers(0, n + 1) if s else 0
                        for n, s in zip(lens, spec)], dtype=np.int32)
        sched.append((tok, spec.astype(np.int32), acc))
    return slots_np, init, sched


def _run(slots_np, init, sched, depth, H, P, check_oracle=True):
    pool = K.StatePool(to_gpu_states(init).cuda())
    ring = K.ReplayRing(P, H, 128, depth, torch.bfloat16)
    slots = i32(slots_np)
    sess = oracle.OracleSession(P, H, 128, 128,
                                init=init.astype(np.float64)) \
        if check_oracle else None
    outs = []
    for tok, spec, acc in sched:
        tb = device_batch(tok, "bf16")
        K.kda_verify(tb, 8, pool, slots, ring, is_spec=i32(spec))
        K.kda_commit(i32(acc), slots, pool, ring)
        outs.append(tb.o.cpu().numpy())
        if sess is not None:
            o_ref = sess.verify(tok, slots_np, spec.astype(bool))
            sess.commit(acc, slots_np)
            assert_outputs(outs[-1], o_ref)
    K.kda_materialize(slots, pool, ring)
    assert K.kda_get_device_error() == 0
    if sess is not None:
        for s in slots_np:
            assert_states(from_gpu_states(pool.data[s]), sess.pool[s])
    return pool.data.cpu(), outs


@pytest.mark.parametrize("B,H,P", [(6, 8, 13), (24, 32, 40)],
                         ids=["48_units", "768_units"])
def test_pipeline_vs_oracle_and_per_unit_kernel(B, H, P):
    """Ragged drafted counts 0..8, ordinary rows among speculative ones,
    accepted lengths 0..T, random initial states: the pipelined kernel
    (depth 8) against the oracle, and its committed states bit for bit
    against the per-unit kernel (depth 9) on the same inputs."""
    slots_np, init, sched = _flow(5100 + B, B, H, P, steps=4)
    small = B * H <= 64
    s8, o8 = _run(slots_np, init, sched, 8, H, P, check_oracle=small)
    s9, o9 = _run(slots_np, init, sched, 9, H, P, check_oracle=False)
    assert torch.equal(s8, s9), "committed states differ between the kernels"
    for a, b in zip(o8, o9):
        assert_outputs(a, b)


def test_pipeline_sampled_heads_many_units_vs_oracle():
    """768 units (about five per CTA) followed on the oracle for heads 0, 17
    and 31 over several steps."""
    B, H, P = 24, 32, 40
    hs = [0, 17, 31]
    slots_np, init, sched = _flow(5200, B, H, P, steps=5)
    pool = K.StatePool(to_gpu_states(init).cuda())
    ring = K.ReplayRing(P, H, 128, 8, torch.bfloat16)
    slots = i32(slots_np)
    sess = oracle.OracleSession(
        P, len(hs), 128, 128,
        init=init[:, hs].astype(np.float64))
    for tok, spec, acc in sched:
        tb = device_batch(tok, "bf16")
        K.kda_verify(tb, 8, pool, slots, ring, is_spec=i32(spec))
        K.kda_commit(i32(acc), slots, pool, ring)
        sub = {n: np.ascontiguousarray(tok[n][:, hs]) for n in
               ("q", "k", "v", "alpha", "beta")}
        sub["cu_seqlens"] = tok["cu_seqlens"]
        o_ref = sess.verify(sub, slots_np, spec.astype(bool))
        sess.commit(acc, slots_np)
        assert_outputs(tb.o[:, hs].cpu().numpy(), o_ref)
    K.kda_materialize(slots, pool, ring)
    for s in slots_np:
        assert_states(from_gpu_states(pool.data[s][hs]), sess.pool[s])
    assert K.kda_get_device_error() == 0


def test_pipeline_ring_contents_match_per_unit_kernel():
    """After a verify, the ring entries and control words the pipelined
    kernel writes equal the per-unit kernel's (entries 0..T-1 hold the
    drafted inputs as given; ctrl {T, 0} for speculative rows, {0, 0} for
    ordinary ones)."""
    B, H, P = 10, 16, 23
    slots_np, init, sched = _flow(5300, B, H, P, steps=1)
    tok, spec, _ = sched[0]
    rings = []
    for depth in (8, 9):
        pool = K.StatePool(to_gpu_states(init).cuda())
        ring = K.ReplayRing(P, H, 128, depth, torch.bfloat16)
        tb = device_batch(tok, "bf16")
        K.kda_verify(tb, 8, pool, i32(slots_np), ring, is_spec=i32(spec))
        torch.cuda.synchronize()
        rings.append(ring)
    r8, r9 = rings
    assert torch.equal(r8.ctrl, r9.ctrl)
    lens = np.diff(tok["cu_seqlens"])
    for i, s in enumerate(slots_np):
        if spec[i] and lens[i] > 0:
            n = int(lens[i])
            for name in ("k", "v", "alpha", "beta"):
                assert torch.equal(getattr(r8, name)[s][:, :n],
                                   getattr(r9, name)[s][:, :n]), name
    assert K.kda_get_device_error() == 0


def test_pipeline_device_errors_skip_units():
    """A slot out of range and a speculative segment longer than the ring
    skip their units (outputs, state, ring untouched) and set their bits;
    the other rows are served normally."""
    B, H, P = 4, 8, 8
    rng = np.random.default_rng(5400)
    init = (rng.standard_normal((P, H, 128, 128)) * 0.3).astype(np.float32)
    pool = K.StatePool(to_gpu_states(init).cuda())
    ring = K.ReplayRing(P, H, 128, 4, torch.bfloat16)
    lens = [3, 6, 2, 1]
    tok = ki.round_to(ki.gen_tokens(rng, lens, H, 128), "bf16")
    slots_np = np.array([1, 5, 99, 6], np.int32)  # row 2: bad slot
    tb = device_batch(tok, "bf16")
    tb.o.fill_(float("nan"))
    before = pool.data.clone()
    K.kda_verify(tb, 8, pool, i32(slots_np), ring, is_spec=i32([1, 1, 1, 0]))
    bits = K.kda_get_device_error()
    assert bits & K.KDA_DERR_SLOT and bits & K.KDA_DERR_DEPTH
    cu = tok["cu_seqlens"]
    o = tb.o.cpu().numpy()
    for i in (1, 2):  # row 1: 6 drafts > depth 4; row 2: bad slot
        assert np.isnan(o[cu[i]:cu[i + 1]]).all()
    assert torch.equal(pool.data[5], before[5])
    sess = oracle.OracleSession(P, H, 128, 128,
                                init=init.astype(np.float64))
    ok = [0, 3]
    sub = {n: np.concatenate([tok[n][cu[i]:cu[i + 1]] for i in ok]) for n in
           ("q", "k", "v", "alpha", "beta")}
    sub["cu_seqlens"] = np.array([0, lens[0], lens[0] + lens[3]], np.int32)
    o_ref = sess.verify(sub, slots_np[ok], [True, False])
    got = np.concatenate([o[cu[i]:cu[i + 1]] for i in ok])
    assert_outputs(got, o_ref)
    assert_states(from_gpu_states(pool.data[6]), sess.pool[6])


@pytest.mark.parametrize("lens,spec", [([3], [1]), ([2, 1], [1, 0]), ([1], [0])],
                         ids=["one_row_3", "spec2_plus_decode1", "one_decode"])
def test_pipeline_batch_shorter_than_a_token_box(lens, spec):
    """Batches of fewer than 8 tokens (the token boxes shrink to the batch):
    two verify + commit steps against the oracle and the per-unit kernel,
    with pending ring entries replayed in the second step."""
    H, P = 8, 5
    rng = np.random.default_rng(5500 + sum(lens))
    B = len(lens)
    slots_np = ki.slot_table(rng, B, P)
    init = (rng.standard_normal((P, H, 128, 128)) * 0.3).astype(np.float32)
    sched = []
    for _ in range(2):
        tok = ki.round_to(ki.gen_tokens(rng, lens, H, 128), "bf16")
        acc = np.array([rng.integers(0, n + 1) if s else 0 for n, s in zip(lens, spec)],
                       dtype=np.int32)
        sched.append((tok, np.array(spec, np.int32), acc))
    s8, o8 = _run(slots_np, init, sched, 8, H, P)
    s9, o9 = _run(slots_np, init, sched, 9, H, P, check_oracle=False)
    assert torch.equal(s8, s9)
    for a, b in zip(o8, o9):
        assert_outputs(a, b)
