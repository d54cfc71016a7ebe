"""Seeded synthetic inputs for the KDA recurrent-state path.

Shared by the tests, the benchmark and the smoke check; holds none of the
method's arithmetic.  Distributions (per token, per head):

* q, v ~ N(0, 1)
* k ~ N(0, 1), then L2-normalised over d_k (in fp32, before any cast)
* alpha = exp(-softplus(z)), z ~ N(0, 1), per key channel
* beta = sigmoid(z), z ~ N(0, 1)

Values are generated in fp64 with numpy's PCG64, rounded to fp32, and then
(for bf16 workloads) rounded to bf16 by torch; both the CUDA path and the
oracle consume exactly those rounded values.  Workload shapes follow the five
named workloads of the path (tiny, spec-verify, prefill, mixed, serving).
"""
from dataclasses import dataclass, field

import numpy as np

# Seeds: workload index i uses 1000 + i.
SEED_TINY, SEED_SPEC, SEED_PREFILL, SEED_MIXED, SEED_SERVING = (
    1001, 1002, 1003, 1004, 1005)


@dataclass
class Workload:
    name: str
    num_seqs: int
    num_heads: int
    d: int
    dtype: str  # "f32" or "bf16"
    seed: int
    extra: dict = field(default_factory=dict)


TINY = Workload("tiny: 1 seq, 2 heads, d=16, fp32; 64-token prefill chunk 16 "
                "ckpt 32; 8 verify steps T=4, a~U{0..4}", 1, 2, 16, "f32",
                SEED_TINY, dict(prefill_len=64, chunk=16, ckpt_every=32,
                                steps=8, T=4))
SPEC = Workload("spec verify+commit: 16 seqs, 32 heads, d=128, bf16, "
                "64 shuffled slots, T=8, a~U{0..8}, ring depth 8, 256 steps",
                16, 32, 128, "bf16", SEED_SPEC,
                dict(num_slots=64, T=8, depth=8, steps=256))
PREFILL = Workload("chunked prefill: 1 seq x 8192 tokens, 32 heads, d=128, "
                   "bf16, chunk 64, ckpt every 1024, S0~N(0,0.02^2)", 1, 32,
                   128, "bf16", SEED_PREFILL,
                   dict(prefill_len=8192, chunk=64, ckpt_every=1024,
                        s0_std=0.02))
MIXED = Workload("mixed batch: 64 seqs in 256 shuffled slots, 8 spec (T=8, "
                 "a~U{0..8}) + 56 decode, 32 heads, d=128, bf16, 128 steps",
                 64, 32, 128, "bf16", SEED_MIXED,
                 dict(num_slots=256, num_spec=8, T=8, depth=8, steps=128))
SERVING = Workload("serving-shaped: 16 seqs x (8192-token prefill, ckpt 1024) "
                   "then T=8 verify until 1024 committed, a ~ capped geometric "
                   "mean 4.7", 16, 32, 128, "bf16", SEED_SERVING,
                   dict(prefill_len=8192, chunk=64, ckpt_every=1024, T=8,
                        depth=8, decode_tokens=1024, rho=0.8802))


def _softplus(z):
    return np.logaddexp(0.0, z)


def gen_tokens(rng, lengths, H, dk, dv=None):
    """Packed token tensors for sequences of the given lengths (fp32 numpy)."""
    dv = dk if dv is None else dv
    lengths = np.asarray(lengths, dtype=np.int64)
    N = int(lengths.sum())
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    q = rng.standard_normal((N, H, dk))
    k = rng.standard_normal((N, H, dk))
    nrm = np.sqrt((k.astype(np.float32) ** 2).sum(-1, keepdims=True))
    k = k.astype(np.float32) / np.maximum(nrm, np.float32(1e-12))
    v = rng.standard_normal((N, H, dv))
    alpha = np.exp(-_softplus(rng.standard_normal((N, H, dk))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((N, H))))
    f = np.float32
    return dict(q=q.astype(f), k=k.astype(f), v=v.astype(f),
                alpha=alpha.astype(f), beta=beta.astype(f), cu_seqlens=cu)


def gen_raw_tokens(rng, lengths, H, dk, dv=None):
    """Projection-space tokens for the fused-prep prefill (fp32 numpy): the
    draws gen_tokens prepares -- raw keys k ~ N(0, 1) (not normalised), decay
    logits alpha ~ N(0, 1), logits beta ~ N(0, 1), q, v ~ N(0, 1).  The
    preparation itself belongs to the path under test and to the oracle."""
    dv = dk if dv is None else dv
    lengths = np.asarray(lengths, dtype=np.int64)
    N = int(lengths.sum())
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    f = np.float32
    return dict(q=rng.standard_normal((N, H, dk)).astype(f),
                k=rng.standard_normal((N, H, dk)).astype(f),
                v=rng.standard_normal((N, H, dv)).astype(f),
                alpha=rng.standard_normal((N, H, dk)).astype(f),
                beta=rng.standard_normal((N, H)).astype(f), cu_seqlens=cu)


def round_to(tok, dtype):
    """Round the float tensors of ``tok`` to ``dtype`` ("f32" or "bf16").

    Returns fp32 numpy arrays holding exactly the rounded values.
    """
    if dtype == "f32":
        return dict(tok)
    import torch
    out = dict(tok)
    for n in ("q", "k", "v", "alpha", "beta"):
        out[n] = (torch.from_numpy(np.ascontiguousarray(tok[n]))
                  .to(torch.bfloat16).float().numpy())
    return out


def slot_table(rng, num_seqs, num_slots):
    """A shuffled sample of distinct pool slots, one per sequence."""
    return rng.permutation(num_slots)[:num_seqs].astype(np.int32)


def accepted_uniform(rng, n, T):
    """accepted_len ~ U{0..T}."""
    return rng.integers(0, T + 1, size=n).astype(np.int32)


def accepted_capped_geometric(rng, n, rho, cap):
    """Consecutive accepts, each with probability rho, capped at ``cap``.

    P(a = j) = rho^j (1 - rho) for j < cap and P(cap) = rho^cap, so the mean
    is sum_{j=1..cap} rho^j (4.7 for rho = 0.8802, cap = 8).
    """
    u = rng.random((n, cap))
    a = np.zeros(n, dtype=np.int32)
    alive = np.ones(n, dtype=bool)
    for j in range(cap):
        alive &= u[:, j] < rho
        a += alive
    return a


def initial_states(rng, num_slots, H, dk, dv, std):
    """Pool-initial states in the oracle's orientation [slot][H][d_k][d_v]."""
    if std == 0:
        return np.zeros((num_slots, H, dk, dv), dtype=np.float32)
    return (rng.standard_normal((num_slots, H, dk, dv)) * std).astype(
        np.float32)
