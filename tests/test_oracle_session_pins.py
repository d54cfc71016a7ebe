"""Pins of the oracle's serving protocol (``OracleSession``) against the step.

``OracleSession`` carries the protocol every GPU parity test is checked
against: a speculative verify leaves the committed state alone and holds its
drafted tokens as pending, ``commit(a)`` folds the first ``a`` of them in and
drops the rest (vLLM Kimi K3 page, "ReplaySSM shrinks rollback state": a
rejection only moves a pointer), a second verify with no commit between
replaces the pending drafts, and ordinary rows of a mixed batch are applied
and committed at once ("Small tensor copies leave the hot path": each request
of a mixed batch is served as if alone).

Every pin below compares the session with the bare recurrence taken token by
token through ``oracle.step`` -- the single-token routine that
``test_oracle_pins`` fixes by exact rationals and closed forms -- never with
another session.  The second half plants one plausible mistake in a copy of
the session's source per branch and checks that some pin fails.
"""
import inspect

import numpy as np
import pytest

import kda_inputs as ki
import oracle
from oracle import kda_oracle

H, DK, DV, SLOTS = 2, 8, 6, 6
FIELDS = ("q", "k", "v", "alpha", "beta")


def _rng(s):
    return np.random.default_rng(777 + s)


def _batch(rng, lengths):
    return ki.gen_tokens(rng, lengths, H, DK, DV)


def _one(tok, i):
    """Segment i of a packed batch as a batch of its own."""
    lo, hi = int(tok["cu_seqlens"][i]), int(tok["cu_seqlens"][i + 1])
    one = {x: np.asarray(tok[x][lo:hi]) for x in FIELDS}
    one["cu_seqlens"] = np.array([0, hi - lo], np.int32)
    return one


def _steps(S, seg, n):
    """State [H][d_k][d_v] after the first n tokens of seg, and their outputs,
    one oracle.step per (token, head)."""
    S = np.array(S, dtype=np.float64, copy=True)
    outs = np.zeros((n, H, DV))
    for t in range(n):
        for h in range(H):
            S[h], outs[t, h] = oracle.step(S[h], seg["q"][t, h], seg["k"][t, h],
                                           seg["v"][t, h], seg["alpha"][t, h],
                                           seg["beta"][t, h])
    return S, outs


def _init(rng):
    return rng.standard_normal((SLOTS, H, DK, DV)) * 0.5


# --------------------------------------------------------------- the pins
# Each takes the session class so the mutants below can run the same checks.

def pin_ordinary_rows_commit_at_once(Session):
    """An ordinary (non-speculative) row is applied and committed in the
    verify itself: its outputs are the step's and pool[slot] is the state
    after all of its tokens; a run of one-token ordinary verifies equals the
    token-by-token recurrence over the whole run."""
    rng = _rng(1)
    init = _init(rng)
    tok = _batch(rng, [3])
    sess = Session(SLOTS, H, DK, DV, init=init)
    o = sess.verify(tok, [4], [False])
    S_ref, o_ref = _steps(init[4], _one(tok, 0), 3)
    assert np.array_equal(o, o_ref)
    assert np.array_equal(sess.pool[4], S_ref)
    run = _batch(rng, [5])
    sess = Session(SLOTS, H, DK, DV, init=init)
    for t in range(5):
        one = {x: run[x][t:t + 1] for x in FIELDS}
        one["cu_seqlens"] = np.array([0, 1], np.int32)
        sess.verify(one, [1], [False])
        sess.commit([1], [1])  # nothing pending: no effect
    S_ref, _ = _steps(init[1], run, 5)
    assert np.array_equal(sess.pool[1], S_ref)


def pin_spec_verify_leaves_state(Session):
    """A speculative verify writes the drafted tokens' outputs (the step's,
    from the committed state) and leaves every slot's bytes unchanged."""
    rng = _rng(2)
    init = _init(rng)
    tok = _batch(rng, [4, 2])
    sess = Session(SLOTS, H, DK, DV, init=init)
    o = sess.verify(tok, [0, 3], [True, True])
    for i, s in enumerate((0, 3)):
        lo, hi = tok["cu_seqlens"][i], tok["cu_seqlens"][i + 1]
        _, o_ref = _steps(init[s], _one(tok, i), hi - lo)
        assert np.array_equal(o[lo:hi], o_ref)
    assert sess.pool.tobytes() == init.tobytes()


def pin_commit_every_count(Session):
    """commit(a) after a speculative verify of T tokens is the state after
    the first a drafted tokens, for every a in 0..T; a = 0 keeps the bytes."""
    rng = _rng(3)
    init = _init(rng)
    T = 4
    tok = _batch(rng, [T])
    for a in range(T + 1):
        sess = Session(SLOTS, H, DK, DV, init=init)
        sess.verify(tok, [2], [True])
        sess.commit([a], [2])
        S_ref, _ = _steps(init[2], _one(tok, 0), a)
        assert np.array_equal(sess.pool[2], S_ref)
        if a == 0:
            assert sess.pool[2].tobytes() == init[2].tobytes()


def pin_second_verify_replaces_pending(Session):
    """verify, verify, commit(a): only the second verify's drafts are folded
    in (the first ones count as all rejected)."""
    rng = _rng(4)
    init = _init(rng)
    first, second = _batch(rng, [3]), _batch(rng, [4])
    for a in (1, 3, 4):
        sess = Session(SLOTS, H, DK, DV, init=init)
        sess.verify(first, [5], [True])
        o2 = sess.verify(second, [5], [True])
        sess.commit([a], [5])
        S_ref, o_ref = _steps(init[5], _one(second, 0), a)
        assert np.array_equal(sess.pool[5], S_ref)
        _, o_all = _steps(init[5], _one(second, 0), 4)
        assert np.array_equal(o2, o_all)


def pin_commit_consumes_pending(Session):
    """A commit folds the pending drafts once: a second commit with no verify
    between, or a commit with no verify at all, changes nothing."""
    rng = _rng(5)
    init = _init(rng)
    tok = _batch(rng, [4])
    sess = Session(SLOTS, H, DK, DV, init=init)
    sess.commit([3], [0])  # nothing pending
    assert sess.pool.tobytes() == init.tobytes()
    sess.verify(tok, [0], [True])
    sess.commit([2], [0])
    after = sess.pool.copy()
    sess.commit([3], [0])
    assert sess.pool.tobytes() == after.tobytes()
    S_ref, _ = _steps(init[0], _one(tok, 0), 2)
    assert np.array_equal(sess.pool[0], S_ref)


def pin_ordinary_row_drops_pending(Session):
    """An ordinary row on a slot with pending drafts applies its own tokens to
    the committed state; the drafts count as rejected, so a later commit of
    that slot changes nothing."""
    rng = _rng(6)
    init = _init(rng)
    drafts, plain = _batch(rng, [4]), _batch(rng, [1])
    sess = Session(SLOTS, H, DK, DV, init=init)
    sess.verify(drafts, [3], [True])
    sess.verify(plain, [3], [False])
    sess.commit([4], [3])
    S_ref, _ = _steps(init[3], _one(plain, 0), 1)
    assert np.array_equal(sess.pool[3], S_ref)


def pin_mixed_batch_rows(Session):
    """Speculative and ordinary rows of one packed batch, then one commit:
    each row's outputs and state are the step's, as if served alone."""
    rng = _rng(7)
    init = _init(rng)
    lengths = [3, 1, 2, 1]
    spec = [True, False, True, False]
    slots = [1, 4, 0, 5]
    acc = [2, 0, 0, 0]
    tok = _batch(rng, lengths)
    sess = Session(SLOTS, H, DK, DV, init=init)
    o = sess.verify(tok, slots, spec)
    sess.commit(acc, slots)
    for i, s in enumerate(slots):
        lo, hi = tok["cu_seqlens"][i], tok["cu_seqlens"][i + 1]
        seg = _one(tok, i)
        _, o_ref = _steps(init[s], seg, hi - lo)
        assert np.array_equal(o[lo:hi], o_ref)
        S_ref, _ = _steps(init[s], seg, acc[i] if spec[i] else hi - lo)
        assert np.array_equal(sess.pool[s], S_ref)
    for s in (2, 3):
        assert sess.pool[s].tobytes() == init[s].tobytes()


def pin_prefill_then_drafts(Session):
    """Prefill moves pool[slot] by every token (the step's outputs) and
    clears that slot's pending drafts; checkpoint slots receive the state at
    the block boundary."""
    rng = _rng(8)
    init = _init(rng)
    drafts, prompt = _batch(rng, [2]), _batch(rng, [8])
    sess = Session(SLOTS, H, DK, DV, init=init)
    sess.verify(drafts, [2], [True])
    o, n = sess.prefill(prompt, [2], ckpt_every=4, ckpt_slots=[[0, 5]])
    sess.commit([2], [2])
    S_ref, o_ref = _steps(init[2], _one(prompt, 0), 8)
    assert np.array_equal(o, o_ref)
    assert np.array_equal(sess.pool[2], S_ref)
    assert int(n[0]) == 2
    S4, _ = _steps(init[2], _one(prompt, 0), 4)
    assert np.array_equal(sess.pool[0], S4)
    assert np.array_equal(sess.pool[5], S_ref)


PINS = [pin_ordinary_rows_commit_at_once, pin_spec_verify_leaves_state,
        pin_commit_every_count, pin_second_verify_replaces_pending,
        pin_commit_consumes_pending, pin_ordinary_row_drops_pending,
        pin_mixed_batch_rows, pin_prefill_then_drafts]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_session_pin(pin):
    pin(oracle.OracleSession)


# ------------------------------------------------------------ the mutants
# One plausible mistake per branch of the session, planted in a copy of its
# source.  Anchors must match exactly, so a change to the session that moves
# them fails loudly here instead of silently testing nothing.
SESSION_MUTANTS = {
    # ordinary rows held as drafts instead of committed
    "ordinary_row_not_committed": [("if spec[i]:", "if True:")],
    # ordinary rows fold one token too few
    "ordinary_row_short_by_one": [("np.array([n], dtype=np.int32)",
                                   "np.array([n - 1], dtype=np.int32)")],
    # a second verify keeps the first verify's drafts pending
    "second_verify_keeps_first": [("self.pending[s] = seg",
                                   "self.pending.setdefault(s, seg)")],
    # a commit leaves its drafts pending, so a later commit folds them again
    "pending_not_cleared": [("seg = self.pending.pop(s, None)",
                             "seg = self.pending.get(s)")],
    # commit folds every drafted token whatever a is
    "commit_folds_all_drafts": [("np.array([int(a)], dtype=np.int32)",
                                 "np.array([n], dtype=np.int32)")],
    # an ordinary row leaves the slot's older drafts pending
    "ordinary_row_keeps_drafts": [("                self.pending.pop(s, None)\n",
                                   "                pass\n")],
    # prefill keeps the slot's older drafts pending
    "prefill_keeps_drafts": [("self.pending.pop(int(s), None)", "pass")],
}


def _mutant_session(name):
    src = inspect.getsource(kda_oracle.OracleSession)
    for a, b in SESSION_MUTANTS[name]:
        assert src.count(a) == 1, f"mutation anchor not unique: {a!r}"
        src = src.replace(a, b)
    ns = dict(vars(kda_oracle))
    exec(compile(src, f"<OracleSession:{name}>", "exec"), ns)
    return ns["OracleSession"]


def _failing_pins(Session):
    failed = []
    for pin in PINS:
        try:
            pin(Session)
        except AssertionError:
            failed.append(pin.__name__)
    return failed


def test_unmutated_copy_passes_every_pin():
    src = inspect.getsource(kda_oracle.OracleSession)
    ns = dict(vars(kda_oracle))
    exec(compile(src, "<OracleSession:copy>", "exec"), ns)
    assert _failing_pins(ns["OracleSession"]) == []


@pytest.mark.parametrize("name", sorted(SESSION_MUTANTS))
def test_session_mutant_is_caught(name):
    assert _failing_pins(_mutant_session(name)), f"mutant {name} passed every pin"
