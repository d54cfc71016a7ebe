"""Pins of the fp64 oracle against facts that do not come from the oracle.

The recurrence under test (gated delta rule, the reading of KDA used here):
    S_t = (I - b_t k_t k_t^T) Diag(a_t) S_{t-1} + b_t k_t v_t^T,   o_t = S_t^T q_t
Each pin is a closed form, an invariant derived by hand from that formula, a
special case with a textbook answer, or exact rational arithmetic, chosen so
that a dropped term, a wrong sign, a transposed operand, decay applied after
instead of before the correction, or an output read from the pre-update state
fails at least one of them.
"""
from fractions import Fraction

import numpy as np
import pytest

import kda_inputs as ki
import oracle


def _rng(s=0):
    return np.random.default_rng(12345 + s)


# ---------------------------------------------------------------- scalar case
def test_scalar_case_exact_rational():
    """d_k = d_v = 1: s_t = a (1 - b k^2) s + b k v and o_t = s_t q exactly.

    The scalar form is derived by hand from the matrix formula; the reference
    values are computed in exact rational arithmetic.
    """
    rng = _rng(1)
    s_exact = Fraction(0)
    S = np.zeros((1, 1))
    for _ in range(40):
        a, b = rng.uniform(0.2, 1.0), rng.uniform(0.0, 1.0)
        k, v, q = rng.standard_normal(3)
        s_exact = (Fraction(a) * (1 - Fraction(b) * Fraction(k) ** 2) * s_exact
                   + Fraction(b) * Fraction(k) * Fraction(v))
        S, o = oracle.step(S, [q], [k], [v], [a], b)
        assert abs(S[0, 0] - float(s_exact)) <= 1e-13 * max(1, abs(s_exact))
        assert abs(o[0] - float(s_exact * Fraction(q))) <= 1e-13 * max(
            1, abs(s_exact * Fraction(q)))


def test_scalar_case_hand_values():
    """Three steps computed by hand: a=1/2, b=1/2, k=1; v = 2, 4, -2; q = 1.

    s1 = 1/2*(1-1/2)*0 + 1/2*2 = 1
    s2 = 1/2*(1/2)*1 + 1/2*4   = 9/4
    s3 = 1/2*(1/2)*9/4 - 1     = -7/16
    """
    S = np.zeros((1, 1))
    want = [1.0, 2.25, -0.4375]
    for v, w in zip([2.0, 4.0, -2.0], want):
        S, o = oracle.step(S, [1.0], [1.0], [v], [0.5], 0.5)
        assert S[0, 0] == w and o[0] == w


# ------------------------------------------------------------ closed forms
def test_beta_zero_is_pure_row_decay():
    """b = 0: S_t = Diag(prod a) S_0 (decay acts on key rows), o_t = S_t^T q_t."""
    rng = _rng(2)
    dk, dv = 5, 3  # unequal, so a transposed operand cannot pass
    S0 = rng.standard_normal((dk, dv))
    S = S0.copy()
    prod = np.ones(dk)
    for _ in range(7):
        a = rng.uniform(0.1, 1.0, dk)
        q = rng.standard_normal(dk)
        S, o = oracle.step(S, q, rng.standard_normal(dk),
                           rng.standard_normal(dv), a, 0.0)
        prod *= a
        np.testing.assert_allclose(S, prod[:, None] * S0, rtol=1e-14, atol=0)
        np.testing.assert_allclose(o, (prod[:, None] * S0).T @ q, rtol=1e-13,
                                   atol=1e-15)


def test_alpha_one_beta_zero_state_constant():
    """a = 1, b = 0: the state never moves (the literal reading of the formula)."""
    rng = _rng(3)
    S0 = rng.standard_normal((4, 4))
    S = S0.copy()
    for _ in range(5):
        S, _ = oracle.step(S, rng.standard_normal(4), rng.standard_normal(4),
                           rng.standard_normal(4), np.ones(4), 0.0)
    assert np.array_equal(S, S0)


def test_orthonormal_keys_running_sum():
    """a = 1, mutually orthogonal unit keys, S_0 = 0: S_t = sum_s b_s k_s v_s^T."""
    rng = _rng(4)
    dk, dv = 6, 4
    order = rng.permutation(dk)
    S = np.zeros((dk, dv))
    acc = np.zeros((dk, dv))
    for t in range(dk):
        k = np.zeros(dk)
        k[order[t]] = 1.0
        v = rng.standard_normal(dv)
        b = rng.uniform()
        q = rng.standard_normal(dk)
        S, o = oracle.step(S, q, k, v, np.ones(dk), b)
        acc += b * np.outer(k, v)
        np.testing.assert_allclose(S, acc, rtol=0, atol=1e-15)
        np.testing.assert_allclose(o, acc.T @ q, rtol=1e-14, atol=1e-15)


def test_unit_key_overwrite():
    """a = 1, b = 1, one unit key k reused: k^T S_t = v_t^T after every step."""
    rng = _rng(5)
    dk, dv = 7, 5
    k = rng.standard_normal(dk)
    k /= np.linalg.norm(k)
    S = rng.standard_normal((dk, dv))
    for _ in range(4):
        v = rng.standard_normal(dv)
        S, _ = oracle.step(S, rng.standard_normal(dk), k, v, np.ones(dk), 1.0)
        np.testing.assert_allclose(k @ S, v, rtol=0, atol=1e-13)


def test_key_readback_identity():
    """k^T S_t = (1 - b|k|^2) k^T Diag(a) S_{t-1} + b |k|^2 v_t^T (hand-derived)."""
    rng = _rng(6)
    dk, dv = 6, 3
    S = rng.standard_normal((dk, dv))
    for _ in range(6):
        a = rng.uniform(0.05, 1.0, dk)
        k = rng.standard_normal(dk) * 0.7
        v = rng.standard_normal(dv)
        b = rng.uniform()
        prev = S.copy()
        S, _ = oracle.step(S, rng.standard_normal(dk), k, v, a, b)
        n2 = k @ k
        want = (1 - b * n2) * (k @ (a[:, None] * prev)) + b * n2 * v
        np.testing.assert_allclose(k @ S, want, rtol=1e-12, atol=1e-12)


def test_orthogonal_complement_only_decays():
    """x orthogonal to k: x^T S_t = x^T Diag(a) S_{t-1} (the correction is along k)."""
    rng = _rng(7)
    dk, dv = 5, 4
    S = rng.standard_normal((dk, dv))
    for _ in range(5):
        a = rng.uniform(0.1, 1.0, dk)
        k = rng.standard_normal(dk)
        x = rng.standard_normal(dk)
        x -= (x @ k) / (k @ k) * k
        prev = S.copy()
        S, _ = oracle.step(S, rng.standard_normal(dk), k,
                           rng.standard_normal(dv), a, rng.uniform())
        np.testing.assert_allclose(x @ S, x @ (a[:, None] * prev), rtol=1e-12,
                                   atol=1e-12)


def test_constant_inputs_geometric_series():
    """Uniform decay a, fixed unit k, fixed v, S_0 = 0:
    k^T S_t = b v (1 - r^t) / (1 - r) with r = a (1 - b); o_t uses S_t (post-update).
    """
    rng = _rng(8)
    dk, dv = 4, 3
    a, b = 0.9, 0.3
    k = rng.standard_normal(dk)
    k /= np.linalg.norm(k)
    v = rng.standard_normal(dv)
    S = np.zeros((dk, dv))
    r = a * (1 - b)
    for t in range(1, 12):
        S, o = oracle.step(S, k, k, v, np.full(dk, a), b)
        want = b * v * (1 - r ** t) / (1 - r)
        np.testing.assert_allclose(k @ S, want, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(o, want, rtol=1e-13, atol=1e-15)
        # nothing outside span{k}
        np.testing.assert_allclose(S, np.outer(k, k @ S), atol=1e-14)


def test_explicit_matrix_product_tiny():
    """Literal (I - b k k^T) Diag(a) S + b k v^T with dense matrices, tiny sizes."""
    rng = _rng(9)
    dk, dv = 3, 2
    S = rng.standard_normal((dk, dv))
    for _ in range(5):
        a = rng.uniform(0.1, 1, dk)
        k, q = rng.standard_normal(dk), rng.standard_normal(dk)
        v, b = rng.standard_normal(dv), rng.uniform()
        want = (np.eye(dk) - b * np.outer(k, k)) @ np.diag(a) @ S + b * np.outer(k, v)
        S, o = oracle.step(S, q, k, v, a, b)
        np.testing.assert_allclose(S, want, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(o, want.T @ q, rtol=1e-13, atol=1e-14)


# ------------------------------------------------- protocol-level pins
def _tok(rng, lengths, H=2, dk=8, dv=6):
    return ki.gen_tokens(rng, lengths, H, dk, dv)


def test_prefill_checkpoints_equal_truncated_runs():
    """Checkpoint m is the state after (m+1)*ckpt_every tokens (absolute)."""
    rng = _rng(10)
    for start in (0, 8, 13):
        tok = _tok(rng, [50])
        S0 = rng.standard_normal((1, 2, 8, 6)) * 0.1
        o, S, ck, n = oracle.prefill(tok["cu_seqlens"], tok["q"], tok["k"],
                                     tok["v"], tok["alpha"], tok["beta"], S0,
                                     start_pos=[start], ckpt_every=16,
                                     max_ckpt=4)
        bounds = [p for p in range(start + 1, start + 51) if p % 16 == 0]
        assert n[0] == len(bounds)
        for m, p in enumerate(bounds):
            L = p - start
            sub = {x: tok[x][:L] for x in ("q", "k", "v", "alpha", "beta")}
            _, Sp, _, _ = oracle.prefill(np.array([0, L], np.int32), sub["q"],
                                         sub["k"], sub["v"], sub["alpha"],
                                         sub["beta"], S0)
            assert np.array_equal(ck[0, m], Sp[0])


def test_verify_then_commit_equals_sequential_steps():
    """verify outputs = first T sequential outputs; commit(a) = a sequential steps;
    commit(0) leaves the state bytes unchanged."""
    rng = _rng(11)
    T = 5
    tok = _tok(rng, [T, T, T])
    S0 = rng.standard_normal((3, 2, 8, 6))
    o_v = oracle.verify(tok["cu_seqlens"], tok["q"], tok["k"], tok["v"],
                        tok["alpha"], tok["beta"], S0)
    o_p, S_full, _, _ = oracle.prefill(tok["cu_seqlens"], tok["q"], tok["k"],
                                       tok["v"], tok["alpha"], tok["beta"], S0)
    assert np.array_equal(o_v, o_p)
    for a in range(T + 1):
        acc = np.array([a, 0, T], np.int32)
        S1 = oracle.commit(tok["cu_seqlens"], tok["q"], tok["k"], tok["v"],
                           tok["alpha"], tok["beta"], acc, S0)
        assert S1[1].tobytes() == S0[1].tobytes()
        assert np.array_equal(S1[2], S_full[2])
        S_ref = S0[0].copy()
        for t in range(a):
            S_ref = np.stack([oracle.step(S_ref[h], tok["q"][t, h], tok["k"][t, h],
                                          tok["v"][t, h], tok["alpha"][t, h],
                                          tok["beta"][t, h])[0] for h in range(2)])
        assert np.array_equal(S1[0], S_ref)


def test_session_mixed_equals_separate():
    """A packed batch of spec and decode requests equals per-request calls."""
    rng = _rng(12)
    lengths = [4, 1, 1, 4, 1]
    spec = [True, False, False, True, False]
    tok = _tok(rng, lengths)
    init = rng.standard_normal((8, 2, 8, 6))
    slots = [5, 0, 7, 2, 3]
    sess = oracle.OracleSession(8, 2, 8, 6, init=init)
    o_all = sess.verify(tok, slots, spec)
    sess.commit([3, 0, 0, 0, 0], slots)
    for i in range(5):
        lo, hi = tok["cu_seqlens"][i], tok["cu_seqlens"][i + 1]
        one = {x: tok[x][lo:hi] for x in ("q", "k", "v", "alpha", "beta")}
        one["cu_seqlens"] = np.array([0, hi - lo], np.int32)
        s2 = oracle.OracleSession(8, 2, 8, 6, init=init)
        o1 = s2.verify(one, [slots[i]], [spec[i]])
        s2.commit([[3, 0, 0, 0, 0][i]], [slots[i]])
        assert np.array_equal(o1, o_all[lo:hi])
        assert np.array_equal(s2.pool[slots[i]], sess.pool[slots[i]])


def test_thread_count_does_not_change_bits():
    rng = _rng(13)
    tok = _tok(rng, [9, 17, 4, 30], H=3)
    S0 = rng.standard_normal((4, 3, 8, 6))
    n0 = oracle.num_threads()
    oracle.set_num_threads(1)
    a = oracle.prefill(tok["cu_seqlens"], tok["q"], tok["k"], tok["v"],
                       tok["alpha"], tok["beta"], S0)
    oracle.set_num_threads(max(n0, 2))
    b = oracle.prefill(tok["cu_seqlens"], tok["q"], tok["k"], tok["v"],
                       tok["alpha"], tok["beta"], S0)
    oracle.set_num_threads(n0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_capped_geometric_reading():
    """rho = 0.8802, cap 8: mean sum_{j=1..8} rho^j = 4.70, P(0) = 0.12, P(8) = 0.36."""
    rho = 0.8802
    assert abs(sum(rho ** j for j in range(1, 9)) - 4.70) < 5e-3
    a = ki.accepted_capped_geometric(np.random.default_rng(0), 200000, rho, 8)
    assert abs(a.mean() - 4.70) < 0.03
    assert abs((a == 0).mean() - (1 - rho)) < 0.01
    assert abs((a == 8).mean() - rho ** 8) < 0.01


# ------------------------------------------------------------ input prep
def test_prep_inputs_closed_forms():
    """The input prep (the generator's formulas) against values fixed by the
    mathematics: softplus(0) = ln 2, so z = 0 gives alpha = 1/2 exactly;
    sigmoid(0) = 1/2; alpha -> e^{-z} for large z and -> 1 for very negative
    z; sigmoid is odd about 1/2; a 3-4-5 key normalises to (0.6, 0.8); a zero
    key stays zero; q passes through."""
    q = np.array([[[1.5, -2.0]]])
    k = np.array([[[3.0, 4.0]]])
    z = np.array([[[0.0, 40.0]]])
    b = np.array([[0.0]])
    q2, k2, a2, b2 = oracle.prep_inputs(q, k, z, b)
    assert np.array_equal(q2, q)
    assert np.allclose(k2, [[[0.6, 0.8]]], rtol=0, atol=1e-15)
    assert a2[0, 0, 0] == 0.5
    assert abs(a2[0, 0, 1] / np.exp(-40.0) - 1.0) < 1e-12
    assert b2[0, 0] == 0.5
    _, _, a3, b3 = oracle.prep_inputs(q, k, np.array([[[-40.0, 3.0]]]),
                                      np.array([[2.5]]))
    assert abs(a3[0, 0, 0] - 1.0) < 1e-15
    assert abs(a3[0, 0, 1] - 1.0 / (1.0 + np.exp(3.0))) < 1e-15  # exp(-softplus(z)) = sigmoid(-z)
    _, _, _, b4 = oracle.prep_inputs(q, k, z, np.array([[-2.5]]))
    assert abs(b3[0, 0] + b4[0, 0] - 1.0) < 1e-15
    _, k5, _, _ = oracle.prep_inputs(q, np.zeros((1, 1, 2)), z, b)
    assert np.array_equal(k5, np.zeros((1, 1, 2)))


def test_prep_inputs_matches_generator():
    """Random projections: unit-norm keys parallel to the raw keys, and
    alpha, beta as the generator draws them from the same normal values."""
    rng = np.random.default_rng(8)
    kr = rng.standard_normal((5, 3, 16)) * 3.0
    z = rng.standard_normal((5, 3, 16))
    b = rng.standard_normal((5, 3))
    _, k, a, bb = oracle.prep_inputs(np.zeros_like(kr), kr, z, b)
    assert np.allclose(np.linalg.norm(k, axis=-1), 1.0, atol=1e-14)
    assert np.allclose(k * np.linalg.norm(kr, axis=-1, keepdims=True), kr, atol=1e-12)
    assert np.allclose(a, 1.0 / (1.0 + np.exp(z)), atol=1e-15)
    assert np.allclose(bb, 1.0 / (1.0 + np.exp(-b)), atol=1e-15)
