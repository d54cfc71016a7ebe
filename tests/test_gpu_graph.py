"""Verify, commit and materialize captured in CUDA graphs against the same
calls issued eagerly, and against the oracle.

Inside a graph consecutive verify / materialize launches are programmatic
dependents of one another: a launch may start while the previous one (which
may write the very states it reads, e.g. materialize then verify on the same
slots) is finishing, and must still read only completed data.  Eager and
graph runs use the same kernels, so outputs and states must agree bit for
bit; both are checked against the fp64 oracle too.
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


def test_graph_replay_matches_eager_and_oracle():
    rng = np.random.default_rng(91)
    B, H, d, P, T, NL, steps = 5, 4, 128, 12, 8, 3, 4
    slots_np = ki.slot_table(rng, B, P)
    slots = i32(slots_np)
    S0 = rng.standard_normal((P, H, d, d)) * 0.3
    start = to_gpu_states(S0).cuda()
    toks = [[ki.round_to(ki.gen_tokens(rng, [T, 3, T, 1, 5], H, d), "bf16")
             for _ in range(NL)] for _ in range(steps)]
    acc_np = [np.array([rng.integers(0, n + 1) for n in (T, 3, T, 1, 5)],
                       dtype=np.int32) for _ in range(steps)]
    accs = [i32(a) for a in acc_np]
    batches = [[device_batch(t, "bf16") for t in row] for row in toks]

    def fresh():
        pools = [K.StatePool(start.clone()) for _ in range(NL)]
        rings = [K.ReplayRing(P, H, d, T, torch.bfloat16) for _ in range(NL)]
        return pools, rings

    def step(s, pools, rings, stream):
        for l in range(NL):
            K.kda_verify(batches[s][l], T, pools[l], slots, rings[l], stream=stream)
        K.kda_commit_layers(accs[s], slots, pools[0], rings, stream=stream)
        if s % 2 == 1:   # materialize, then the next step's verify on the same slots
            for l in range(NL):
                K.kda_materialize(slots, pools[l], rings[l], stream=stream)

    # eager
    pools_e, rings_e = fresh()
    outs_e = []
    for s in range(steps):
        step(s, pools_e, rings_e, None)
        torch.cuda.synchronize()
        outs_e.append([b.o.clone() for b in batches[s]])
    for l in range(NL):
        K.kda_materialize(slots, pools_e[l], rings_e[l])
    torch.cuda.synchronize()
    assert K.kda_get_device_error() == 0

    # graphs, one per step, replayed in order
    pools_g, rings_g = fresh()
    side = torch.cuda.Stream()
    graphs = []
    with torch.cuda.stream(side):
        for s in range(steps):
            g = torch.cuda.CUDAGraph()
            g.capture_begin()
            step(s, pools_g, rings_g, side)
            g.capture_end()
            graphs.append(g)
    torch.cuda.synchronize()
    for row in batches:
        for b in row:
            b.o.fill_(float("nan"))
    with torch.cuda.stream(side):
        for g in graphs:
            g.replay()
        for l in range(NL):
            K.kda_materialize(slots, pools_g[l], rings_g[l], stream=side)
    torch.cuda.synchronize()
    assert K.kda_get_device_error() == 0
    for s in range(steps):
        for l in range(NL):
            assert torch.equal(batches[s][l].o, outs_e[s][l])
    for l in range(NL):
        assert torch.equal(pools_g[l].data, pools_e[l].data)

    # the oracle, layer by layer
    for l in range(NL):
        sess = oracle.OracleSession(P, H, d, d, init=S0)
        for s in range(steps):
            assert_outputs(outs_e[s][l].cpu().numpy(), sess.verify(toks[s][l], slots_np))
            sess.commit(acc_np[s], slots_np)
        for sl in slots_np:
            assert_states(from_gpu_states(pools_e[l].data[sl]), sess.pool[sl])
