"""The oracle still reproduces its committed tiny-workload fixture."""
import os

import numpy as np

from golden.make_golden import lines

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _parse(ls):
    d = {}
    for ln in ls:
        if ln.startswith("#"):
            continue
        key, *vals = ln.split()
        d[key] = vals
    return d


def test_tiny_fixture_reproduces():
    want = _parse(open(os.path.join(HERE, "tiny_oracle.txt")).read().splitlines())
    got = _parse(lines())
    assert want.keys() == got.keys()
    for key in want:
        if key in ("n_ckpt", "accepted"):
            assert want[key] == got[key]
        else:
            np.testing.assert_allclose(np.array(got[key], float),
                                       np.array(want[key], float),
                                       rtol=1e-12, atol=1e-13)
