"""kda_verify_raw: the verify with the input prep fused (keys L2-normalised,
alpha = exp(-softplus(z)), beta = sigmoid(b)), against the same verify on
inputs the oracle prepared, and against the oracle.

The reading under test: each prepared k, alpha, beta is computed once in
fp32 and rounded to bf16, and everything downstream uses those bits.  The
oracle prepares in fp64 (`oracle.prep_inputs`) and rounds to bf16 the same
way.  The two roundings agree wherever the fp64 value is not within the fp32
prep's error of a bf16 rounding midpoint, so the raw inputs are drawn clear
of such near-ties: an element whose prepared value lies within 2^-19
(relative) of a midpoint has its raw bf16 input moved by one step and the
check repeats (the kernel's prep error is below 2^-21).  On those inputs
the raw verify must equal the prepared verify bit for bit -- outputs,
committed states and ring entries -- and both must meet the output and
state tolerances against the oracle.
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


def _near_midpoint(x, rel=2.0 ** -19):
    """Where fp64 values lie within `rel` (relative) of a bf16 rounding
    midpoint (8 significant bits)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    m, e = np.frexp(a)                     # a = m 2^e, m in [0.5, 1)
    ulp = np.ldexp(1.0, e - 8)             # bf16 spacing in [2^(e-1), 2^e)
    frac = a / ulp - np.floor(a / ulp)
    return (a > 0) & (np.abs(frac - 0.5) * ulp < rel * a)


def _bump_bf16(x, mask):
    """Move the bf16 values x[mask] (held exactly in fp32) by one step."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    bits = f.view(np.uint32) >> 16
    bits = np.where(mask, bits + 1, bits).astype(np.uint32)
    return (bits << 16).view(np.float32)


def raw_tokens_clear_of_ties(rng, lens, H, D=128):
    """Raw bf16 tokens (q, k, v, z_alpha, z_beta) whose fp64 prep lands
    clear of bf16 rounding midpoints, and the oracle's prepared tokens
    rounded to bf16."""
    raw = ki.round_to(ki.gen_raw_tokens(rng, lens, H, D), "bf16")
    for _ in range(40):
        q, k, a, b = oracle.prep_inputs(raw["q"], raw["k"], raw["alpha"], raw["beta"])
        nk, na, nb = _near_midpoint(k), _near_midpoint(a), _near_midpoint(b)
        if not (nk.any() or na.any() or nb.any()):
            break
        raw["k"] = _bump_bf16(raw["k"], nk)
        raw["alpha"] = _bump_bf16(raw["alpha"], na)
        raw["beta"] = _bump_bf16(raw["beta"], nb)
    else:
        raise AssertionError("raw inputs did not clear the rounding midpoints")
    prepared = dict(q=q, k=k, v=raw["v"], alpha=a, beta=b,
                    cu_seqlens=raw["cu_seqlens"])
    return raw, ki.round_to(prepared, "bf16")


def _schedule(seed, B, H, P, steps, max_T=8, spec_frac=0.75, init_std=0.05):
    rng = np.random.default_rng(seed)
    slots_np = ki.slot_table(rng, B, P)
    init = (rng.standard_normal((P, H, 128, 128)) * init_std).astype(np.float32)
    sched = []
    for _ in range(steps):
        spec = rng.random(B) < spec_frac
        lens = [int(rng.integers(0, max_T + 1)) if s else 1 for s in spec]
        raw, prep = raw_tokens_clear_of_ties(rng, lens, H)
        acc = np.array([rng.integers(0, n + 1) if s else 0
                        for n, s in zip(lens, spec)], dtype=np.int32)
        sched.append((raw, prep, spec.astype(np.int32), acc))
    return slots_np, init, sched


@pytest.mark.parametrize("B,H,P", [(6, 8, 13), (24, 32, 40)],
                         ids=["48_units", "768_units"])
def test_verify_raw_equals_prepared_verify_and_oracle(B, H, P):
    """Ragged drafted counts 0..8 beside ordinary rows, several steps of
    verify + commit: the raw call and the prepared call agree bit for bit
    (outputs every step; states, ring entries and control words at the end),
    and the raw call meets the tolerances against the oracle (all units at
    48, heads 0, 13, 31 at 768)."""
    slots_np, init, sched = _schedule(7100 + B, B, H, P, steps=4)
    slots = i32(slots_np)
    hs = list(range(H)) if H <= 8 else [0, 13, 31]
    pools = [K.StatePool(to_gpu_states(init).cuda()) for _ in range(2)]
    rings = [K.ReplayRing(P, H, 128, 8, torch.bfloat16) for _ in range(2)]
    sess = oracle.OracleSession(P, len(hs), 128, 128,
                                init=init[:, hs].astype(np.float64))
    for raw, prep, spec, acc in sched:
        tr, tp = device_batch(raw, "bf16"), device_batch(prep, "bf16")
        K.kda_verify(tr, 8, pools[0], slots, rings[0], is_spec=i32(spec), raw=True)
        K.kda_verify(tp, 8, pools[1], slots, rings[1], is_spec=i32(spec))
        for pool, ring in zip(pools, rings):
            K.kda_commit(i32(acc), slots, pool, ring)
        assert torch.equal(tr.o, tp.o), "raw and prepared outputs differ"
        sub = {n: np.ascontiguousarray(prep[n][:, hs]) for n in
               ("q", "k", "v", "alpha", "beta")}
        sub["cu_seqlens"] = prep["cu_seqlens"]
        o_ref = sess.verify(sub, slots_np, spec.astype(bool))
        sess.commit(acc, slots_np)
        assert_outputs(tr.o[:, hs].cpu().numpy(), o_ref)
    for n in ("k", "v", "alpha", "beta", "ctrl"):
        assert torch.equal(getattr(rings[0], n), getattr(rings[1], n)), n
    for pool, ring in zip(pools, rings):
        K.kda_materialize(slots, pool, ring)
    assert torch.equal(pools[0].data, pools[1].data), "committed states differ"
    for s in slots_np:
        assert_states(from_gpu_states(pools[0].data[s][hs]), sess.pool[s])
    assert K.kda_get_device_error() == 0


def test_verify_raw_replay_equals_decode():
    """The same raw tokens applied as ordinary rows (decoded and committed at
    once) and as drafts accepted in full (recorded by kda_commit, replayed by
    kda_materialize from the ring): the states are equal bit for bit, since
    both read the prepared bits the kernel wrote once."""
    B, H, P, T = 12, 16, 20, 8
    rng = np.random.default_rng(7300)
    slots_np = ki.slot_table(rng, B, P)
    slots = i32(slots_np)
    init = (rng.standard_normal((P, H, 128, 128)) * 0.2).astype(np.float32)
    raw = ki.round_to(ki.gen_raw_tokens(rng, [T] * B, H, 128), "bf16")
    pools = [K.StatePool(to_gpu_states(init).cuda()) for _ in range(2)]
    rings = [K.ReplayRing(P, H, 128, 8, torch.bfloat16) for _ in range(2)]
    K.kda_verify(device_batch(raw, "bf16"), T, pools[0], slots, rings[0],
                 is_spec=i32([0] * B), raw=True)
    K.kda_verify(device_batch(raw, "bf16"), T, pools[1], slots, rings[1],
                 is_spec=i32([1] * B), raw=True)
    K.kda_commit(i32([T] * B), slots, pools[1], rings[1])
    K.kda_materialize(slots, pools[1], rings[1])
    assert torch.equal(pools[0].data, pools[1].data)
    assert K.kda_get_device_error() == 0
