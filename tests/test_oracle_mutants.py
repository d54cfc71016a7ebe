"""Planted mistakes in a copy of the oracle must each fail a pin.

Each mutant is the oracle's C source with one plausible error (a dropped term,
a flipped sign, decay on the wrong index, the output read before the update,
the correction computed from the undecayed state), compiled to a temporary
library on the CPU.  The pin battery below is the closed-form subset of
test_oracle_pins; every mutant must fail at least one of them, and the
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
    lib = ctypes.CDLL(str(so))
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


@pytest.mark.parametrize("name", list(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    fails = _pins(_compile(name, tmp_path))
    if name == "none":
        assert fails == []
    else:
        assert fails, f"mutant {name} passed every pin"
