"""The chunk-wise (WY/UT) algebra equals the token-by-token oracle in fp64.

This pins the oracle against an independent derivation of the same recurrence
(the chunk form is obtained by unrolling the recurrence over C tokens and
solving the resulting unit-lower-triangular system), and it pins the chunk
algebra the CUDA prefill implements before any kernel runs.
"""
import numpy as np
import pytest

import kda_inputs as ki
import oracle
from chunkform_ref import chunk_prefill_one


@pytest.mark.parametrize("C,L,start,dk,dv", [
    (16, 64, 0, 16, 16),     # the tiny workload's shape
    (16, 53, 0, 12, 9),      # ragged tail, unequal dims
    (32, 100, 7, 8, 8),      # unaligned start: first chunk is partial
    (64, 130, 0, 16, 12),
])
def test_chunk_form_matches_sequential(C, L, start, dk, dv):
    rng = np.random.default_rng(100 + C + L)
    tok = ki.gen_tokens(rng, [L], 2, dk, dv)
    S0 = rng.standard_normal((1, 2, dk, dv)) * 0.5
    o, S, ck, n = oracle.prefill(tok["cu_seqlens"], tok["q"], tok["k"],
                                 tok["v"], tok["alpha"], tok["beta"], S0,
                                 start_pos=[start], ckpt_every=2 * C,
                                 max_ckpt=8)
    for h in range(2):
        oc, Sc, ckc = chunk_prefill_one(tok["q"][:, h], tok["k"][:, h],
                                        tok["v"][:, h], tok["alpha"][:, h],
                                        tok["beta"][:, h], S0[0, h], C,
                                        start_pos=start, ckpt_every=2 * C)
        np.testing.assert_allclose(oc, o[:, h], rtol=0, atol=1e-11)
        np.testing.assert_allclose(Sc, S[0, h], rtol=0, atol=1e-11)
        assert len(ckc) == n[0]
        for m, c in enumerate(ckc):
            np.testing.assert_allclose(c, ck[0, m, h], rtol=0, atol=1e-11)


def test_chunk_size_does_not_change_result():
    rng = np.random.default_rng(7)
    tok = ki.gen_tokens(rng, [96], 1, 8, 8)
    S0 = rng.standard_normal((8, 8))
    outs = [chunk_prefill_one(tok["q"][:, 0], tok["k"][:, 0], tok["v"][:, 0],
                              tok["alpha"][:, 0], tok["beta"][:, 0], S0, C)
            for C in (16, 32, 64)]
    for o, S, _ in outs[1:]:
        np.testing.assert_allclose(o, outs[0][0], atol=1e-11)
        np.testing.assert_allclose(S, outs[0][1], atol=1e-11)
