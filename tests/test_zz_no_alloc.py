"""The prefill entry point for callers that cannot allocate device memory.

kda_prefill_chunked_noalloc takes no workspace: hosts that own all device
memory through their own allocator (or that have no allocator handle to hand
over) can still run the chunked prefill, and the library keeps a fixed scratch
array for it instead.  This file checks, through the C ABI, that it produces
what the workspace entry point produces, on two calls in a row (the second
call reuses the scratch the first left behind), and that sizes beyond the
scratch are refused before anything runs.  It is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import kda_inputs as ki
from kda_gpu import assert_outputs, assert_states, device_batch, i32, to_gpu_states
from recurrent_kda_state_gb300 import kda as K
from recurrent_kda_state_gb300._build import build_library

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_library()
    K.kda_get_device_error()
    yield


def _prefill_pair(seed, lengths, starts, H, d, C, ckpt_every, max_ckpt):
    """Run the same prefill through both entry points; return both results."""
    rng = np.random.default_rng(seed)
    B = len(lengths)
    tok = ki.round_to(ki.gen_tokens(rng, lengths, H, d), "bf16")
    P = B * (1 + max_ckpt)
    init = to_gpu_states(ki.initial_states(rng, P, H, d, d, 0.05)).cuda()
    slots = i32(np.arange(B))
    ck = i32((B + np.arange(B * max_ckpt)).reshape(B, max_ckpt))
    sp = i32(starts)
    out = []
    for noalloc in (False, True):
        pool = K.StatePool(init.clone())
        tb = device_batch(tok, "bf16")
        if noalloc:
            K.kda_prefill_chunked_noalloc(tb, pool, slots, C, ckpt_every, ck, sp)
        else:
            K.kda_prefill_chunked(tb, pool, slots, C, ckpt_every, ck, sp)
        torch.cuda.synchronize()
        out.append((tb.o.cpu().numpy(), pool.data.cpu().numpy()))
    assert K.kda_get_device_error() == 0
    return out


def test_noalloc_matches_workspace_entry_two_calls_in_a_row():
    cases = [
        (501, [200, 77], [0, 5], 8, 128, 64, 128, 2),
        (502, [130, 1, 64], [64, 3, 0], 2, 64, 32, 64, 3),
        (503, [200, 77], [0, 5], 4, 128, 64, 128, 2),  # d=128, 4 heads: scratch
        # tensor-core shape whose two-pass workspace exceeds the scratch: the
        # single pass, against the two-pass path of the workspace entry
        (504, [3300], [0], 8, 128, 64, 1024, 3),
    ]
    for seed, lengths, starts, H, d, C, E, mc in cases:
        (o_ref, s_ref), (o_na, s_na) = _prefill_pair(seed, lengths, starts, H, d,
                                                    C, E, mc)
        assert_outputs(o_na, o_ref)
        for s in range(s_ref.shape[0]):
            assert_states(s_na[s], s_ref[s])


def test_noalloc_refuses_sizes_beyond_its_scratch():
    H, d, C = 32, 64, 64  # d=64: the CUDA-core kernels, which need a workspace
    N = 8192  # needs ~340 MB of workspace, far above the fixed scratch
    need = K.kda_prefill_workspace_size(N, 1, H, d, d, C, K.KDA_BF16)
    assert need > K.KDA_NOALLOC_SCRATCH_BYTES
    z = torch.zeros(N, H, d, dtype=torch.bfloat16, device="cuda")
    tb = K.TokenBatch(z, z, z, z, torch.zeros(N, H, dtype=torch.bfloat16,
                                              device="cuda"),
                      i32([0, N]))
    pool = K.StatePool.zeros(1, H, d)
    before = pool.data.clone()
    with pytest.raises(K.KdaError) as e:
        K.kda_prefill_chunked_noalloc(tb, pool, i32([0]), C)
    assert e.value.status == K.KDA_ENOSPC
    torch.cuda.synchronize()
    assert torch.equal(pool.data, before)
