"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Tolerances (fixed for the path): outputs max-abs <= 2e-3, states relative
Frobenius <= 1e-3, bf16 or fp32 inputs, fp32 state.  Replay-committed state
must be bit-identical to step-by-step decode; slot and ring bookkeeping must
be bit-exact.  Workload shapes follow the five named workloads; the largest
runs sample heads on the oracle side (heads are independent units).
"""
import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle
from kda_gpu import (assert_outputs, assert_states, device_batch,
                     from_gpu_states, heads, i32, to_gpu_states)
from recurrent_kda_state_gb300 import kda as K

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_error_word():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    K.kda_get_device_error()
    yield


def _spec_tokens(rng, B, H, d, T, dtype):
    return ki.round_to(ki.gen_tokens(rng, [T] * B, H, d), dtype)


# ------------------------------------------------------------ tiny workload
def test_tiny_workload_end_to_end():
    """64-token fp32 prefill (chunk 16, checkpoint every 32), then 8 verify
    steps of T = 4 with accepted_len ~ U{0..4}, lazily committed."""
    w = ki.TINY
    rng = np.random.default_rng(w.seed)
    H, d = w.num_heads, w.d
    pre = ki.gen_tokens(rng, [64], H, d)
    P = 3
    pool = K.StatePool.zeros(P, H, d)
    ring = K.ReplayRing(P, H, d, 4, torch.float32)
    sess = oracle.OracleSession(P, H, d, d)
    slots = i32([0])
    tb = device_batch(pre, "f32")
    K.kda_prefill_chunked(tb, pool, slots, chunk=16, ckpt_every=32,
                          ckpt_slots=i32([[1, 2]]))
    o_ref, nck = sess.prefill(pre, [0], ckpt_every=32,
                              ckpt_slots=np.array([[1, 2]]))
    assert nck[0] == 2
    assert_outputs(tb.o.cpu().numpy(), o_ref)
    for s in range(3):
        assert_states(from_gpu_states(pool.data[s]), sess.pool[s])
    for _ in range(w.extra["steps"]):
        tok = ki.gen_tokens(rng, [4], H, d)
        tb = device_batch(tok, "f32")
        K.kda_verify(tb, 4, pool, slots, ring)
        assert_outputs(tb.o.cpu().numpy(), sess.verify(tok, [0]))
        a = ki.accepted_uniform(rng, 1, 4)
        K.kda_commit(i32(a), slots, pool, ring)
        sess.commit(a, [0])
    K.kda_materialize(slots, pool, ring)
    assert_states(from_gpu_states(pool.data[0]), sess.pool[0])
    assert K.kda_get_device_error() == 0


# ------------------------------------------------- spec verify + commit
def _run_spec(steps, hs, seed=ki.SEED_SPEC, B=16, H=32, d=128, P=64, T=8,
              dtype="bf16"):
    rng = np.random.default_rng(seed)
    slots_np = ki.slot_table(rng, B, P)
    slots = i32(slots_np)
    pool = K.StatePool.zeros(P, H, d)
    ring = K.ReplayRing(P, H, d, T, ki_torch(dtype))
    sess = oracle.OracleSession(P, len(hs), d, d)
    for _ in range(steps):
        tok = _spec_tokens(rng, B, H, d, T, dtype)
        a = ki.accepted_uniform(rng, B, T)
        tb = device_batch(tok, dtype)
        K.kda_verify(tb, T, pool, slots, ring)
        K.kda_commit(i32(a), slots, pool, ring)
        o_ref = sess.verify(heads(tok, hs), slots_np)
        sess.commit(a, slots_np)
        assert_outputs(tb.o[:, hs].cpu().numpy(), o_ref)
    K.kda_materialize(slots, pool, ring)
    for s in slots_np:
        assert_states(from_gpu_states(pool.data[s][hs]), sess.pool[s])
    assert K.kda_get_device_error() == 0
    return pool


def ki_torch(dtype):
    return torch.bfloat16 if dtype == "bf16" else torch.float32


def test_spec_verify_all_heads_few_steps():
    _run_spec(steps=5, hs=list(range(32)))


def test_spec_verify_full_256_steps_sampled_heads():
    """The full spec-verify workload (16 seqs, 32 heads, d=128, 256 steps) on
    the GPU; the oracle follows heads 0 and 29 through every step."""
    _run_spec(steps=256, hs=[0, 29])


def test_spec_verify_fp32_small_dims():
    for d in (16, 32, 64):
        _run_spec(steps=4, hs=[0, 1, 2], B=5, H=3, d=d, P=9, T=4, dtype="f32",
                  seed=77 + d)


def test_spec_verify_ragged_drafts_depth16():
    """Ring depth 16 and up to 16 drafted tokens (the 16-row draft tiles), with
    ragged draft counts per sequence (including 0 and 1); accepted lengths
    up to each sequence's own count; d=128, bf16, all heads followed."""
    rng = np.random.default_rng(916)
    B, H, d, P, D16 = 6, 8, 128, 12, 16
    slots_np = ki.slot_table(rng, B, P)
    slots = i32(slots_np)
    pool = K.StatePool.zeros(P, H, d)
    ring = K.ReplayRing(P, H, d, D16, torch.bfloat16)
    sess = oracle.OracleSession(P, H, d, d)
    hs = list(range(H))
    for step in range(5):
        lens = [16, 0, 5, 9, 1, 12] if step % 2 == 0 else [3, 16, 0, 8, 11, 2]
        tok = ki.round_to(ki.gen_tokens(rng, lens, H, d), "bf16")
        a = np.array([rng.integers(0, n + 1) for n in lens], dtype=np.int32)
        tb = device_batch(tok, "bf16")
        K.kda_verify(tb, D16, pool, slots, ring)
        K.kda_commit(i32(a), slots, pool, ring)
        o_ref = sess.verify(tok, slots_np)
        sess.commit(a, slots_np)
        assert_outputs(tb.o.cpu().numpy(), o_ref)
    K.kda_materialize(slots, pool, ring)
    for s_ in slots_np:
        assert_states(from_gpu_states(pool.data[s_]), sess.pool[s_])
    assert K.kda_get_device_error() == 0


# ------------------------------------------------------ bit-exact replay
def _random_pool(rng, P, H, d, std=0.3):
    return K.StatePool(to_gpu_states(
        rng.standard_normal((P, H, d, d)).astype(np.float32) * std).cuda())


@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (16, "f32"), (64, "bf16")])
def test_replay_commit_is_bit_identical_to_step_by_step(d, dtype):
    rng = np.random.default_rng(5 + d)
    B, H, P, T = 6, 4, 10, 8
    slots_np = ki.slot_table(rng, B, P)
    slots = i32(slots_np)
    poolA = _random_pool(rng, P, H, d)
    poolB = K.StatePool(poolA.data.clone())
    ringA = K.ReplayRing(P, H, d, T, ki_torch(dtype))
    ringB = K.ReplayRing(P, H, d, T, ki_torch(dtype))
    tok = _spec_tokens(rng, B, H, d, T, dtype)
    a = np.array([0, 1, 3, 8, 5, 2], dtype=np.int32)
    # A: verify T drafts, commit(a), materialize (replay)
    K.kda_verify(device_batch(tok, dtype), T, poolA, slots, ringA)
    K.kda_commit(i32(a), slots, poolA, ringA)
    K.kda_materialize(slots, poolA, ringA)
    # B: ordinary one-token decode launches, token t for every seq with t < a_i
    for t in range(int(a.max())):
        lens = [1 if t < a[i] else 0 for i in range(B)]
        rows = [i * T + t for i in range(B) if t < a[i]]
        one = {n: tok[n][rows] for n in ("q", "k", "v", "alpha", "beta")}
        one["cu_seqlens"] = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        K.kda_verify(device_batch(one, dtype), 1, poolB, slots, ringB,
                     is_spec=i32([0] * B))
    torch.cuda.synchronize()
    assert torch.equal(poolA.data, poolB.data)
    assert K.kda_get_device_error() == 0


def test_verify1_commit1_equals_decode_state():
    rng = np.random.default_rng(21)
    B, H, d, P = 4, 2, 128, 6
    slots = i32(ki.slot_table(rng, B, P))
    poolA = _random_pool(rng, P, H, d)
    poolB = K.StatePool(poolA.data.clone())
    ringA = K.ReplayRing(P, H, d, 8, torch.bfloat16)
    ringB = K.ReplayRing(P, H, d, 8, torch.bfloat16)
    tok = _spec_tokens(rng, B, H, d, 1, "bf16")
    K.kda_verify(device_batch(tok, "bf16"), 1, poolA, slots, ringA)
    K.kda_commit(i32([1] * B), slots, poolA, ringA)
    K.kda_materialize(slots, poolA, ringA)
    K.kda_verify(device_batch(tok, "bf16"), 1, poolB, slots, ringB,
                 is_spec=i32([0] * B))
    torch.cuda.synchronize()
    assert torch.equal(poolA.data, poolB.data)


def test_commit_layers_equals_per_layer_commit():
    """One kda_commit_layers launch == kda_commit on each layer, bit for bit."""
    rng = np.random.default_rng(23)
    B, H, d, P, T, NL = 5, 4, 128, 9, 8, 3
    slots = i32(ki.slot_table(rng, B, P))
    pools = [_random_pool(rng, P, H, d) for _ in range(NL)]
    pools2 = [K.StatePool(p.data.clone()) for p in pools]
    rings = [K.ReplayRing(P, H, d, T, torch.bfloat16) for _ in range(NL)]
    rings2 = [K.ReplayRing(P, H, d, T, torch.bfloat16) for _ in range(NL)]
    for step in range(3):
        toks = [device_batch(_spec_tokens(rng, B, H, d, T, "bf16"), "bf16")
                for _ in range(NL)]
        a = i32(ki.accepted_uniform(rng, B, T))
        for l in range(NL):
            K.kda_verify(toks[l], T, pools[l], slots, rings[l])
        K.kda_commit_layers(a, slots, pools[0], rings)
        for l in range(NL):
            t2 = K.TokenBatch(toks[l].q, toks[l].k, toks[l].v, toks[l].alpha,
                              toks[l].beta, toks[l].cu_seqlens)
            K.kda_verify(t2, T, pools2[l], slots, rings2[l])
            K.kda_commit(a, slots, pools2[l], rings2[l])
            assert torch.equal(t2.o, toks[l].o)
    for l in range(NL):
        assert torch.equal(rings[l].ctrl, rings2[l].ctrl)
        K.kda_materialize(slots, pools[l], rings[l])
        K.kda_materialize(slots, pools2[l], rings2[l])
        torch.cuda.synchronize()
        assert torch.equal(pools[l].data, pools2[l].data)
    assert K.kda_get_device_error() == 0


def test_commit_zero_leaves_state_bytes():
    rng = np.random.default_rng(22)
    B, H, d, P, T = 3, 4, 128, 5, 8
    slots = i32(ki.slot_table(rng, B, P))
    pool = _random_pool(rng, P, H, d)
    before = pool.data.clone()
    ring = K.ReplayRing(P, H, d, T, torch.bfloat16)
    for _ in range(3):
        K.kda_verify(device_batch(_spec_tokens(rng, B, H, d, T, "bf16"), "bf16"),
                     T, pool, slots, ring)
        K.kda_commit(i32([0] * B), slots, pool, ring)
    K.kda_materialize(slots, pool, ring)
    torch.cuda.synchronize()
    assert pool.data.view(torch.int32).equal(before.view(torch.int32))


# ------------------------------------------------------------ mixed batch
def _mixed_step_tokens(rng, spec_mask, H, d, T):
    lens = [T if s else 1 for s in spec_mask]
    return ki.round_to(ki.gen_tokens(rng, lens, H, d), "bf16")


def test_mixed_batch_vs_oracle_and_separate_calls():
    """64 sequences in 256 shuffled slots, 8 speculative (T=8) at seeded random
    positions among 56 ordinary decodes, one packed launch per step."""
    w = ki.MIXED
    rng = np.random.default_rng(w.seed)
    B, H, d, P, T = 64, 32, 128, 256, 8
    slots_np = ki.slot_table(rng, B, P)
    spec_mask = np.zeros(B, dtype=bool)
    spec_mask[rng.choice(B, 8, replace=False)] = True
    slots, is_spec = i32(slots_np), i32(spec_mask.astype(np.int32))
    pool = K.StatePool.zeros(P, H, d)
    ring = K.ReplayRing(P, H, d, T, torch.bfloat16)
    hs = [0, 7, 31]
    sess = oracle.OracleSession(P, len(hs), d, d)
    for step in range(4):
        tok = _mixed_step_tokens(rng, spec_mask, H, d, T)
        a = np.where(spec_mask, ki.accepted_uniform(rng, B, T), 0).astype(np.int32)
        if step == 3:  # separate per-request launches on a clone, bit for bit
            pool2 = K.StatePool(pool.data.clone())
            ring2 = K.ReplayRing(P, H, d, T, torch.bfloat16)
            for n in ("k", "v", "alpha", "beta", "ctrl"):
                getattr(ring2, n).copy_(getattr(ring, n))
        tb = device_batch(tok, "bf16")
        K.kda_verify(tb, T, pool, slots, ring, is_spec=is_spec)
        K.kda_commit(i32(a), slots, pool, ring)
        o_ref = sess.verify(heads(tok, hs), slots_np, spec_mask)
        sess.commit(a, slots_np)
        assert_outputs(tb.o[:, hs].cpu().numpy(), o_ref)
    cu = tok["cu_seqlens"]
    for i in range(B):
        one = {n: tok[n][cu[i]:cu[i + 1]] for n in ("q", "k", "v", "alpha", "beta")}
        one["cu_seqlens"] = np.array([0, cu[i + 1] - cu[i]], np.int32)
        t1 = device_batch(one, "bf16")
        K.kda_verify(t1, T, pool2, slots[i:i + 1], ring2, is_spec=is_spec[i:i + 1])
        K.kda_commit(i32(a[i:i + 1]), slots[i:i + 1], pool2, ring2)
        assert torch.equal(t1.o, tb.o[cu[i]:cu[i + 1]])
    K.kda_materialize(slots, pool, ring)
    K.kda_materialize(slots, pool2, ring2)
    torch.cuda.synchronize()
    assert torch.equal(pool.data, pool2.data)
    assert torch.equal(ring.ctrl, ring2.ctrl)
    for s in slots_np:
        assert_states(from_gpu_states(pool.data[s][hs]), sess.pool[s])
    assert K.kda_get_device_error() == 0


def test_slot_permutation_invariance():
    rng = np.random.default_rng(31)
    B, H, d, P, T = 8, 4, 128, 20, 8
    tok = _spec_tokens(rng, B, H, d, T, "bf16")
    a = ki.accepted_uniform(rng, B, T)
    init = rng.standard_normal((B, H, d, d)).astype(np.float32) * 0.2
    results = []
    for perm_seed in (0, 1):
        prng = np.random.default_rng(100 + perm_seed)
        slots_np = ki.slot_table(prng, B, P)
        order = prng.permutation(B)      # launch order of the sequences
        pool = K.StatePool.zeros(P, H, d)
        pool.data[torch.as_tensor(slots_np[order], dtype=torch.long)] = \
            to_gpu_states(init[order]).cuda()
        ring = K.ReplayRing(P, H, d, T, torch.bfloat16)
        rows = np.concatenate([np.arange(i * T, (i + 1) * T) for i in order])
        t = {n: tok[n][rows] for n in ("q", "k", "v", "alpha", "beta")}
        t["cu_seqlens"] = np.arange(0, (B + 1) * T, T, dtype=np.int32)
        tb = device_batch(t, "bf16")
        sl = i32(slots_np[order])
        K.kda_verify(tb, T, pool, sl, ring)
        K.kda_commit(i32(a[order]), sl, pool, ring)
        K.kda_materialize(sl, pool, ring)
        o = torch.empty_like(tb.o)
        o[torch.as_tensor(rows, dtype=torch.long, device="cuda")] = tb.o
        st = torch.empty(B, H, d, d, device="cuda")
        st[torch.as_tensor(order, dtype=torch.long, device="cuda")] = \
            pool.data[torch.as_tensor(slots_np[order], dtype=torch.long)]
        results.append((o, st))
    assert torch.equal(results[0][0], results[1][0])
    assert torch.equal(results[0][1], results[1][1])


# ------------------------------------------------------------ prefill
def _run_prefill(lengths, starts, H, d, C, ckpt_every, dtype, max_ckpt, hs,
                 seed, s0_std=0.0, skip_ckpt=(), alpha=None, single_pass=False):
    rng = np.random.default_rng(seed)
    B = len(lengths)
    tok = ki.gen_tokens(rng, lengths, H, d)
    if alpha is not None:  # another decay distribution, same shape
        tok["alpha"] = alpha(rng, tok["alpha"].shape).astype(np.float32)
    tok = ki.round_to(tok, dtype)
    P = B * (1 + max_ckpt) + 1
    init = ki.initial_states(rng, P, H, d, d, s0_std)
    pool = K.StatePool(to_gpu_states(init).cuda())
    slots_np = np.arange(B, dtype=np.int32)
    ck = (B + np.arange(B * max_ckpt, dtype=np.int32)).reshape(B, max_ckpt)
    for (i, m) in skip_ckpt:
        ck[i, m] = -1
    tb = device_batch(tok, dtype)
    K.kda_prefill_chunked(tb, pool, i32(slots_np), chunk=C, ckpt_every=ckpt_every,
                          ckpt_slots=i32(ck) if max_ckpt else None,
                          start_pos=i32(starts), single_pass=single_pass)
    sess = oracle.OracleSession(P, len(hs), d, d, init=init[:, hs])
    o_ref, nck = sess.prefill(heads(tok, hs), slots_np, ckpt_every=ckpt_every,
                              ckpt_slots=ck if max_ckpt else None,
                              start_pos=np.asarray(starts, np.int32))
    assert_outputs(tb.o[:, hs].cpu().numpy(), o_ref)
    got = from_gpu_states(pool.data[:, hs])
    for s in range(P):
        assert_states(got[s], sess.pool[s])
    assert K.kda_get_device_error() == 0
    return tb, pool, nck


@pytest.mark.parametrize("single_pass", [False, True], ids=["two_pass", "single_pass"])
def test_prefill_full_workload_sampled_heads(single_pass):
    """1 x 8192 tokens, 32 heads, d=128, bf16, chunk 64, checkpoints every
    1024 tokens, S0 ~ N(0, 0.02^2); the oracle follows heads 0, 13 and 31.
    Both tensor-core paths: two passes through a workspace, and one pass."""
    w = ki.PREFILL
    _, _, nck = _run_prefill([8192], [0], 32, 128, 64, 1024, "bf16", 8,
                             [0, 13, 31], w.seed, s0_std=0.02, single_pass=single_pass)
    assert nck[0] == 8


@pytest.mark.parametrize("C,d,single_pass", [(16, 64, False), (32, 64, False),
                                             (64, 64, False), (64, 128, False),
                                             (64, 128, True)])
def test_prefill_ragged_and_offsets(C, d, single_pass):
    lengths = [0, 1, C - 1, C, C + 1, 3 * C + 5, 100]
    starts = [0, 5, 0, 2 * C, C - 3, 7, 0]
    H = 8 if d == 128 else 4  # d=128, chunk 64, 8 heads: the tensor-core kernels
    _run_prefill(lengths, starts, H, d, C, 2 * C, "bf16", 3, [0, 1, H // 2 + 1, H - 1],
                 seed=900 + C + d, s0_std=0.1, skip_ckpt=[(5, 1)],
                 single_pass=single_pass)


@pytest.mark.parametrize("single_pass", [False, True], ids=["two_pass", "single_pass"])
def test_prefill_slow_decay_carries_state(single_pass):
    """alpha in [0.97, 1): the state carried across chunks dominates the
    outputs (with the default alpha ~ 0.5 it fades within a chunk), so the
    inter-chunk pass and the checkpoints are tested at full weight."""
    _run_prefill([1000, 333, 64], [0, 17, 64], 8, 128, 64, 128, "bf16", 8,
                 [0, 3, 7], seed=912, s0_std=0.5,
                 alpha=lambda rng, shp: 1.0 - 0.03 * rng.random(shp),
                 single_pass=single_pass)


def test_prefill_d128_chunk64_fallback_heads():
    """d=128, chunk 64 with a head count that is not a multiple of 8 takes
    the CUDA-core kernels (the tensor-core kernel's beta map needs 16-byte
    rows); same bar against the oracle."""
    _run_prefill([200, 64, 1], [0, 64, 3], 4, 128, 64, 64, "bf16", 3,
                 [0, 1, 2, 3], seed=913, s0_std=0.1)


def test_prefill_tiny_dims_fp32():
    _run_prefill([64, 37, 5], [0, 16, 3], 2, 16, 16, 32, "f32", 2, [0, 1],
                 seed=5, s0_std=0.05)


def test_prefill_chunk_size_independent():
    rng_lengths = [300, 129]
    outs = []
    for C in (16, 32, 64):
        tb, pool, _ = _run_prefill(rng_lengths, [0, 0], 8, 128, C, 64, "bf16",
                                   1, [0, 7], seed=44, s0_std=0.02)
        outs.append((tb.o.cpu().numpy(), pool.data[:2].cpu().numpy()))
    for o, s in outs[1:]:
        assert np.max(np.abs(o - outs[0][0])) <= 2e-3
        assert np.linalg.norm(s - outs[0][1]) <= 1e-3 * np.linalg.norm(s)


def test_prefill_then_verify_from_checkpoint():
    """Partial prefix hit: fork a checkpoint into a fresh slot, prefill the
    rest of the prompt from its absolute position, then verify drafts."""
    rng = np.random.default_rng(61)
    H, d, C = 8, 128, 64
    prompt = ki.round_to(ki.gen_tokens(rng, [256], H, d), "bf16")
    pool = K.StatePool.zeros(8, H, d)
    ring = K.ReplayRing(8, H, d, 8, torch.bfloat16)
    tb = device_batch(prompt, "bf16")
    K.kda_prefill_chunked(tb, pool, i32([0]), chunk=C, ckpt_every=128,
                          ckpt_slots=i32([[1, 2]]))
    # new request shares the first 128 tokens: fork checkpoint slot 1 -> 3
    K.kda_copy_slots(pool, i32([1]), i32([3]))
    K.kda_ring_reset(i32([3]), pool, ring)
    rest = {n: prompt[n][128:] for n in ("q", "k", "v", "alpha", "beta")}
    rest["cu_seqlens"] = np.array([0, 128], np.int32)
    tr = device_batch(rest, "bf16")
    K.kda_prefill_chunked(tr, pool, i32([3]), chunk=C, start_pos=i32([128]))
    torch.cuda.synchronize()
    np.testing.assert_allclose(tr.o.cpu().numpy(), tb.o[128:].cpu().numpy(),
                               atol=2e-3, rtol=0)
    drafts = _spec_tokens(rng, 1, H, d, 8, "bf16")
    t0, t3 = device_batch(drafts, "bf16"), device_batch(drafts, "bf16")
    K.kda_verify(t0, 8, pool, i32([0]), ring)
    K.kda_verify(t3, 8, pool, i32([3]), ring)
    sess = oracle.OracleSession(1, H, d, d)
    sess.prefill(prompt, [0])
    o_ref = sess.verify(drafts, [0])
    assert_outputs(t0.o.cpu().numpy(), o_ref)
    assert_outputs(t3.o.cpu().numpy(), o_ref)
    assert K.kda_get_device_error() == 0


# ------------------------------------------------------- serving-shaped
def test_serving_shaped_reduced():
    """Serving-shaped load at reduced scale: 3 seqs x 512-token prefill (chunk
    64, checkpoint every 128), then T=8 verify + commit with accepted_len from
    the capped geometric (rho = 0.8802) until 64 tokens are committed."""
    w = ki.SERVING
    rng = np.random.default_rng(w.seed)
    B, H, d, T, P = 3, 8, 128, 8, 3 + 12
    prompt = ki.round_to(ki.gen_tokens(rng, [512] * B, H, d), "bf16")
    pool = K.StatePool.zeros(P, H, d)
    ring = K.ReplayRing(P, H, d, T, torch.bfloat16)
    sess = oracle.OracleSession(P, H, d, d)
    slots_np = np.arange(B, dtype=np.int32)
    ck = (B + np.arange(B * 4, dtype=np.int32)).reshape(B, 4)
    tb = device_batch(prompt, "bf16")
    K.kda_prefill_chunked(tb, pool, i32(slots_np), chunk=64, ckpt_every=128,
                          ckpt_slots=i32(ck))
    o_ref, _ = sess.prefill(prompt, slots_np, ckpt_every=128, ckpt_slots=ck)
    assert_outputs(tb.o.cpu().numpy(), o_ref)
    committed = np.zeros(B, dtype=np.int64)
    while committed.min() < 64:
        live = np.nonzero(committed < 64)[0]
        tok = _spec_tokens(rng, len(live), H, d, T, "bf16")
        a = ki.accepted_capped_geometric(rng, len(live), w.extra["rho"], T)
        a = np.minimum(a, 64 - committed[live]).astype(np.int32)
        tl = device_batch(tok, "bf16")
        K.kda_verify(tl, T, pool, i32(slots_np[live]), ring)
        K.kda_commit(i32(a), i32(slots_np[live]), pool, ring)
        assert_outputs(tl.o.cpu().numpy(), sess.verify(tok, slots_np[live]))
        sess.commit(a, slots_np[live])
        committed[live] += a
    K.kda_materialize(i32(slots_np), pool, ring)
    for s in range(P):
        assert_states(from_gpu_states(pool.data[s]), sess.pool[s])


# ---------------------------------------------------- bookkeeping / errors
def test_gather_and_copy_slots_bit_exact():
    rng = np.random.default_rng(71)
    P, H, d = 9, 3, 64
    pool = _random_pool(rng, P, H, d)
    idx = [4, 0, 8]
    out = K.kda_gather_states(pool, i32(idx))
    torch.cuda.synchronize()
    assert torch.equal(out, pool.data[idx])
    before = pool.data.clone()
    K.kda_copy_slots(pool, i32([1, 2]), i32([5, 7]))
    torch.cuda.synchronize()
    assert torch.equal(pool.data[[5, 7]], before[[1, 2]])
    keep = [0, 1, 2, 3, 4, 6, 8]
    assert torch.equal(pool.data[keep], before[keep])


def test_canaries_untouched():
    """Slots, ring entries and ctrl words outside the launch stay byte-equal;
    every output row of the batch is written."""
    rng = np.random.default_rng(72)
    B, H, d, P, T = 4, 2, 128, 12, 8
    pool = _random_pool(rng, P, H, d)
    ring = K.ReplayRing(P, H, d, T, torch.bfloat16)
    for n in ("k", "v", "alpha", "beta"):
        getattr(ring, n).copy_(torch.randn_like(getattr(ring, n).float()))
    slots_np = np.array([3, 9, 0, 6], np.int32)
    slots = i32(slots_np)
    others = [s for s in range(P) if s not in slots_np]
    snap = {n: getattr(ring, n)[others].clone() for n in ("k", "v", "alpha", "beta", "ctrl")}
    pool_snap = pool.data[others].clone()
    tb = device_batch(_spec_tokens(rng, B, H, d, T, "bf16"), "bf16")
    tb.o.fill_(float("nan"))
    K.kda_verify(tb, T, pool, slots, ring)
    K.kda_commit(i32([2, 0, 8, 5]), slots, pool, ring)
    K.kda_materialize(slots, pool, ring)
    torch.cuda.synchronize()
    assert not torch.isnan(tb.o).any()
    assert torch.equal(pool.data[others], pool_snap)
    for n, v in snap.items():
        assert torch.equal(getattr(ring, n)[others], v), n


def test_device_errors_skip_units_and_set_bits():
    rng = np.random.default_rng(73)
    B, H, d, P, T = 2, 2, 64, 4, 4
    pool = _random_pool(rng, P, H, d)
    ring = K.ReplayRing(P, H, d, T, torch.bfloat16)
    before = pool.data.clone()
    tok = _spec_tokens(rng, B, H, d, T, "bf16")
    # slot id outside the pool
    K.kda_verify(device_batch(tok, "bf16"), T, pool, i32([1, P]), ring)
    assert K.kda_get_device_error() & K.KDA_DERR_SLOT
    # accepted above pending
    K.kda_commit(i32([T + 1, 0]), i32([1, 2]), pool, ring)
    assert K.kda_get_device_error() & K.KDA_DERR_ACCEPT
    # speculative segment longer than the ring (ordinary row may be longer)
    long = ki.round_to(ki.gen_tokens(rng, [T + 2, T + 2], H, d), "bf16")
    K.kda_verify(device_batch(long, "bf16"), T + 2, pool, i32([2, 3]), ring,
                 is_spec=i32([1, 0]))
    assert K.kda_get_device_error() & K.KDA_DERR_DEPTH
    K.kda_materialize(i32([0, 1, 2]), pool, ring)
    torch.cuda.synchronize()
    # slot 1's first verify was fine (drafts pending, commit rejected): unchanged
    assert torch.equal(pool.data[[0, 1, 2]], before[[0, 1, 2]])
    assert not torch.equal(pool.data[3], before[3])  # the ordinary row applied
    assert K.kda_get_device_error() == 0


def test_prefill_decay_range_flag():
    rng = np.random.default_rng(74)
    tok = ki.round_to(ki.gen_tokens(rng, [64], 1, 16), "f32")
    tok["alpha"][:] = 1e-3   # log-decay ~ -6.9 per token: -220 per half chunk
    pool = K.StatePool.zeros(1, 1, 16)
    K.kda_prefill_chunked(device_batch(tok, "f32"), pool, i32([0]), chunk=64)
    assert K.kda_get_device_error() & K.KDA_DERR_RANGE


def test_prefill_decay_range_flag_tensor_core_shape():
    rng = np.random.default_rng(75)
    tok = ki.round_to(ki.gen_tokens(rng, [64], 8, 128), "bf16")
    tok["alpha"][:] = 1e-3
    pool = K.StatePool.zeros(1, 8, 128)
    K.kda_prefill_chunked(device_batch(tok, "bf16"), pool, i32([0]), chunk=64)
    assert K.kda_get_device_error() & K.KDA_DERR_RANGE


def test_determinism():
    p1 = _run_spec(steps=3, hs=[0])
    p2 = _run_spec(steps=3, hs=[0])
    assert torch.equal(p1.data, p2.data)


# ------------------------------------------- prefill beside verify, one call
@pytest.mark.parametrize("use_side", [False, True], ids=["one_stream", "side_stream"])
def test_forward_mixed_prefill_and_verify_segments(use_side):
    """One packed batch: two prefill segments (checkpoints, a start offset)
    followed by speculative and ordinary rows, run by kda_forward_mixed as
    zero-copy views; equals the two separate calls on separate tensors bit for
    bit (outputs, states, ring), and the oracle, also after the commit."""
    rng = np.random.default_rng(71)
    H, d, C, T, P = 8, 128, 64, 8, 24
    spec_mask = [1, 0, 1, 0, 0, 1]
    lens = [200, 77] + [T if m else 1 for m in spec_mask]
    npf, starts = 2, [0, 64]
    tok = ki.round_to(ki.gen_tokens(rng, lens, H, d), "bf16")
    ptok = int(tok["cu_seqlens"][npf])
    slots_np = np.array([0, 1, 5, 6, 7, 8, 9, 10], np.int32)
    ck = np.array([[2, 3], [4, -1]], np.int32)
    init = ki.initial_states(rng, P, H, d, d, 0.1)
    is_spec = np.array([0] * npf + spec_mask, np.int32)

    poolA = K.StatePool(to_gpu_states(init).cuda())
    ringA = K.ReplayRing(P, H, d, T, torch.bfloat16)
    tbA = device_batch(tok, "bf16")
    side = torch.cuda.Stream() if use_side else None
    K.kda_forward_mixed(tbA, npf, ptok, poolA, i32(slots_np), C, T, ringA,
                        ckpt_every=128, ckpt_slots=i32(ck), start_pos=i32(starts),
                        is_spec=i32(is_spec), side_stream=side)

    names = ("q", "k", "v", "alpha", "beta")
    pre = {n: tok[n][:ptok] for n in names}
    pre["cu_seqlens"] = tok["cu_seqlens"][:npf + 1]
    rest = {n: tok[n][ptok:] for n in names}
    rest["cu_seqlens"] = (tok["cu_seqlens"][npf:] - ptok).astype(np.int32)
    poolB = K.StatePool(to_gpu_states(init).cuda())
    ringB = K.ReplayRing(P, H, d, T, torch.bfloat16)
    tbP, tbR = device_batch(pre, "bf16"), device_batch(rest, "bf16")
    K.kda_prefill_chunked(tbP, poolB, i32(slots_np[:npf]), chunk=C, ckpt_every=128,
                          ckpt_slots=i32(ck), start_pos=i32(starts))
    K.kda_verify(tbR, T, poolB, i32(slots_np[npf:]), ringB, is_spec=i32(spec_mask))
    torch.cuda.synchronize()
    assert torch.equal(tbA.o[:ptok], tbP.o) and torch.equal(tbA.o[ptok:], tbR.o)
    assert torch.equal(poolA.data, poolB.data)
    for n in ("k", "v", "alpha", "beta", "ctrl"):
        assert torch.equal(getattr(ringA, n), getattr(ringB, n))

    sess = oracle.OracleSession(P, H, d, d, init=init)
    o_pre, nck = sess.prefill(pre, slots_np[:npf], ckpt_every=128, ckpt_slots=ck,
                              start_pos=np.asarray(starts, np.int32))
    o_rest = sess.verify(rest, slots_np[npf:], is_spec=spec_mask)
    assert list(nck) == [1, 1]
    assert_outputs(tbA.o[:ptok].cpu().numpy(), o_pre)
    assert_outputs(tbA.o[ptok:].cpu().numpy(), o_rest)
    a = np.array([rng.integers(0, T + 1) if m else 0 for m in spec_mask], np.int32)
    K.kda_commit(i32(a), i32(slots_np[npf:]), poolA, ringA)
    sess.commit(a, slots_np[npf:])
    K.kda_materialize(i32(slots_np[npf:]), poolA, ringA)
    got = from_gpu_states(poolA.data)
    for s in range(P):
        assert_states(got[s], sess.pool[s])
    assert K.kda_get_device_error() == 0


# ------------------------------------------------ fused input preparation
@pytest.mark.parametrize("single_pass", [False, True], ids=["two_pass", "single_pass"])
@pytest.mark.parametrize("case", ["ragged", "full"])
def test_prefill_raw_inputs_fused_prep(single_pass, case):
    """kda_prefill_chunked_raw: projection-space inputs (raw keys, decay and
    beta logits) with the prep fused into the tensor-core kernels, against
    the oracle's fp64 prep followed by its prefill; ragged lengths and start
    offsets at 8 heads, and the full 8192-token workload (heads sampled)."""
    if case == "full":
        lengths, starts, H, E, mc, hs, seed = [8192], [0], 32, 1024, 8, [0, 17, 31], 931
    else:
        lengths, starts = [0, 1, 63, 64, 65, 197, 100], [0, 5, 0, 128, 61, 7, 0]
        H, E, mc, hs, seed = 8, 128, 3, [0, 3, 4, 7], 932
    d, C = 128, 64
    rng = np.random.default_rng(seed)
    raw = ki.round_to(ki.gen_raw_tokens(rng, lengths, H, d), "bf16")
    B = len(lengths)
    P = B * (1 + mc) + 1
    init = ki.initial_states(rng, P, H, d, d, 0.05)
    pool = K.StatePool(to_gpu_states(init).cuda())
    slots_np = np.arange(B, dtype=np.int32)
    ck = (B + np.arange(B * mc, dtype=np.int32)).reshape(B, mc)
    tb = device_batch(raw, "bf16")
    K.kda_prefill_chunked(tb, pool, i32(slots_np), chunk=C, ckpt_every=E, ckpt_slots=i32(ck),
                          start_pos=i32(starts), single_pass=single_pass, raw=True)
    q, k, a, b = oracle.prep_inputs(raw["q"], raw["k"], raw["alpha"], raw["beta"])
    prep = dict(q=q, k=k, v=raw["v"].astype(np.float64), alpha=a, beta=b,
                cu_seqlens=raw["cu_seqlens"])
    sess = oracle.OracleSession(P, len(hs), d, d, init=init[:, hs])
    o_ref, _ = sess.prefill(heads(prep, hs), slots_np, ckpt_every=E, ckpt_slots=ck,
                            start_pos=np.asarray(starts, np.int32))
    assert_outputs(tb.o[:, hs].cpu().numpy(), o_ref)
    got = from_gpu_states(pool.data[:, hs])
    for s in range(P):
        assert_states(got[s], sess.pool[s])
    assert K.kda_get_device_error() == 0


def test_verify_launch_configurations_interleave():
    """Launches of the verify kernel with different shared-memory sizes
    (ring depth 16 with 16-token drafts, depth 8, materialize with no tokens)
    interleave in any order: the launch set-up is cached per configuration and
    one configuration must not invalidate another."""
    rng = np.random.default_rng(95)
    B, H, d, P = 3, 8, 128, 8
    slots_np = ki.slot_table(rng, B, P)
    slots = i32(slots_np)
    pool8, pool16 = K.StatePool.zeros(P, H, d), K.StatePool.zeros(P, H, d)
    ring8 = K.ReplayRing(P, H, d, 8, torch.bfloat16)
    ring16 = K.ReplayRing(P, H, d, 16, torch.bfloat16)
    sess8, sess16 = oracle.OracleSession(P, H, d, d), oracle.OracleSession(P, H, d, d)
    for step in range(3):
        for T, pool, ring, sess in ((16, pool16, ring16, sess16), (8, pool8, ring8, sess8)):
            tok = _spec_tokens(rng, B, H, d, T, "bf16")
            tb = device_batch(tok, "bf16")
            K.kda_verify(tb, T, pool, slots, ring)
            a = ki.accepted_uniform(rng, B, T)
            K.kda_commit(i32(a), slots, pool, ring)
            assert_outputs(tb.o.cpu().numpy(), sess.verify(tok, slots_np))
            sess.commit(a, slots_np)
            K.kda_materialize(slots, pool, ring)
    for pool, sess in ((pool8, sess8), (pool16, sess16)):
        got = from_gpu_states(pool.data)
        for s_ in slots_np:
            assert_states(got[s_], sess.pool[s_])
    assert K.kda_get_device_error() == 0
