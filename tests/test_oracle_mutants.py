"""Planted mistakes in a copy of the oracle must each fail a pin.

Each mutant is the oracle's C source with one plausible error, compiled to a
temporary library on the CPU.  Errors in the step are a dropped term, a
flipped sign, decay on the wrong index, the output read before the update,
and the correction computed from the undecayed state.  Errors in the
protocol are a checkpoint one token early, a checkpoint that ignores the
start offset, and a commit that folds in one token too many.  The pin
battery below is the closed-form subset of test_oracle_pins plus brute force
over the protocol: checkpoints and commits against the library's own step
taken token by token.  Every mutant must fail at least one pin, and the
unmodified source must pass all of them.
"""
import ctypes
import os
import subprocess
from fractions import Fraction

import numpy as np
import pytest

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "oracle", "kda_oracle.c")

MUTANTS = {
    "none": [],
    "drop_beta_on_v": [("+ beta * k[c] * v[j]", "+ k[c] * v[j]")],
    "sign_of_correction": [("- beta * k[c] * kM[j]", "+ beta * k[c] * kM[j]")],
    "decay_on_value_index": [("alpha[c] * S[c * dv + j]",
                              "alpha[j % dk] * S[c * dv + j]")],
    "output_before_update": [("acc += S[c * dv + j] * q[c]",
                              "acc += M[c * dv + j] * q[c]")],
    "correction_from_undecayed": [("acc += k[c] * M[c * dv + j]",
                                   "acc += k[c] * S[c * dv + j]")],
    "checkpoint_one_token_early": [("const int p = p0 + (t - cu_seqlens[i]) + 1;",
                                    "const int p = p0 + (t - cu_seqlens[i]);")],
    "checkpoint_ignores_start": [("const int p0 = start_pos ? start_pos[i] : 0;",
                                  "const int p0 = 0;")],
    "commit_one_token_too_many": [
        ("for (int t = cu_seqlens[i]; t < cu_seqlens[i] + a; ++t) {",
         "for (int t = cu_seqlens[i]; t < cu_seqlens[i] + a + (a < len); ++t) {")],
}


def _compile(name, tmp_path):
    src = open(SRC).read()
    for a, b in MUTANTS[name]:
        assert a in src, f"mutation anchor missing: {a}"
        src = src.replace(a, b)
    c = tmp_path / f"{name}.c"
    c.write_text(src)
    so = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O1", "-ffp-contract=off", "-shared", "-fPIC",
                    str(c), "-o", str(so)], check=True, capture_output=True)
    return ctypes.CDLL(str(so))


def _stepper(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    lib.kdao_step.argtypes = [ctypes.c_int, ctypes.c_int, dp, dp, dp, dp, dp,
                              ctypes.c_double, dp]

    def step(S, q, k, v, a, b):
        S = np.array(S, dtype=np.float64, order="C", copy=True)
        arr = [np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v, a)]
        o = np.zeros(S.shape[1])
        P = lambda x: x.ctypes.data_as(dp)  # noqa: E731
        lib.kdao_step(S.shape[0], S.shape[1], P(S), *map(P, arr), float(b), P(o))
        return S, o
    return step


def _pins(step):
    """Return the names of the closed-form pins that fail for ``step``."""
    fails = []
    rng = np.random.default_rng(5)
    # scalar exact
    s, S = Fraction(0), np.zeros((1, 1))
    ok = True
    for _ in range(10):
        a, b = rng.uniform(0.2, 1), rng.uniform()
        k, v, q = rng.standard_normal(3)
        s = Fraction(a) * (1 - Fraction(b) * Fraction(k) ** 2) * s + \
            Fraction(b) * Fraction(k) * Fraction(v)
        S, o = step(S, [q], [k], [v], [a], b)
        ok &= abs(S[0, 0] - float(s)) < 1e-12 and abs(o[0] - float(s) * q) < 1e-12
    if not ok:
        fails.append("scalar")
    # beta = 0 row decay, unequal dims
    S0 = rng.standard_normal((5, 3))
    a = rng.uniform(0.1, 1, 5)
    S, _ = step(S0, rng.standard_normal(5), rng.standard_normal(5),
                rng.standard_normal(3), a, 0.0)
    if not np.allclose(S, a[:, None] * S0, rtol=1e-13, atol=0):
        fails.append("beta0")
    # key readback identity, with decay
    S = rng.standard_normal((6, 4))
    k, v, q = rng.standard_normal(6), rng.standard_normal(4), rng.standard_normal(6)
    a, b = rng.uniform(0.1, 1, 6), 0.4
    S1, o = step(S, q, k, v, a, b)
    want = (1 - b * (k @ k)) * (k @ (a[:, None] * S)) + b * (k @ k) * v
    if not np.allclose(k @ S1, want, rtol=1e-11, atol=1e-11):
        fails.append("readback")
    if not np.allclose(o, S1.T @ q, rtol=1e-12, atol=1e-12):
        fails.append("post_update_output")
    return fails


def _protocol_pins(lib):
    """Checkpoints (with and without a start offset) and commits of every
    count against the library's own step, taken token by token."""
    step = _stepper(lib)
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int32)
    P = lambda x: x.ctypes.data_as(dp)  # noqa: E731
    Pi = lambda x: x.ctypes.data_as(ip)  # noqa: E731
    fails = []
    rng = np.random.default_rng(11)
    H, dk, dv, L, E, M = 1, 3, 2, 10, 4, 4
    q, k = rng.standard_normal((L, H, dk)), rng.standard_normal((L, H, dk))
    v = rng.standard_normal((L, H, dv))
    al = rng.uniform(0.3, 1.0, (L, H, dk))
    be = rng.uniform(0.0, 1.0, (L, H))
    S0 = rng.standard_normal((1, H, dk, dv))
    cu = np.array([0, L], dtype=np.int32)
    for p0 in (0, 3):
        want, S = [], S0[0, 0]
        for t in range(L):
            S, _ = step(S, q[t, 0], k[t, 0], v[t, 0], al[t, 0], be[t, 0])
            if (p0 + t + 1) % E == 0:
                want.append(S)
        S_out = np.zeros_like(S0)
        o = np.zeros((L, H, dv))
        ck = np.zeros((1, M, H, dk, dv))
        nck = np.zeros(1, dtype=np.int32)
        sp = np.array([p0], dtype=np.int32)
        lib.kdao_prefill(1, H, dk, dv, Pi(cu), P(q), P(k), P(v), P(al), P(be),
                         P(S0), P(S_out), P(o), Pi(sp), E, M, P(ck), Pi(nck))
        ok = nck[0] == len(want) and all(
            np.allclose(ck[0, m, 0], w, rtol=1e-13, atol=1e-13)
            for m, w in enumerate(want))
        if not ok:
            fails.append("checkpoints_p0_%d" % p0)
    for a in range(L + 1):
        S = S0[0, 0]
        for t in range(a):
            S, _ = step(S, q[t, 0], k[t, 0], v[t, 0], al[t, 0], be[t, 0])
        Sc = S0.copy()
        acc = np.array([a], dtype=np.int32)
        lib.kdao_commit(1, H, dk, dv, Pi(cu), P(q), P(k), P(v), P(al), P(be),
                        Pi(acc), P(Sc))
        if not np.allclose(Sc[0, 0], S, rtol=1e-13, atol=1e-13):
            fails.append("commit")
            break
    return fails


@pytest.mark.parametrize("name", list(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    lib = _compile(name, tmp_path)
    fails = _pins(_stepper(lib)) + _protocol_pins(lib)
    if name == "none":
        assert fails == []
    else:
        assert fails, f"mutant {name} passed every pin"
