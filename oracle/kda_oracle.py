"""Python face of the fp64 oracle -- TEST INFRASTRUCTURE ONLY.

The arithmetic lives in ``kda_oracle.c`` (plain fp64 loops over the gated
delta rule ``S_t = (I - b_t k_t k_t^T) Diag(a_t) S_{t-1} + b_t k_t v_t^T``,
``o_t = S_t^T q_t``).  This module marshals numpy arrays into it and states
the serving protocol around the recurrence in the plainest way:

* prefill: every token in order; after absolute position p with
  ``p % ckpt_every == 0`` the state is copied out ("KDA checkpoints stay inside
  the prefill" on the vLLM Kimi K3 page).
* verify: a speculative sequence runs its drafted tokens on a copy of the
  committed state; the committed state does not move.
* commit(a): the committed state becomes the state after the first ``a``
  drafted tokens; ``a = 0`` leaves it untouched ("ReplaySSM shrinks rollback
  state": rejection only moves a pointer).
* ordinary decode inside a mixed batch: the token is applied and committed at
  once ("Small tensor copies leave the hot path": each request of a mixed batch
  is served independently).

Oracle layout: a state is ``[d_k][d_v]`` (row = key channel), fp64.
"""
import ctypes
import os

import numpy as np

from .build import build_oracle

_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build_oracle())
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int32)
        i = ctypes.c_int
        lib.kdao_step.argtypes = [i, i, dp, dp, dp, dp, dp, ctypes.c_double, dp]
        lib.kdao_prefill.argtypes = [i, i, i, i, ip, dp, dp, dp, dp, dp, dp,
                                     dp, dp, ip, i, i, dp, ip]
        lib.kdao_verify.argtypes = [i, i, i, i, ip, dp, dp, dp, dp, dp, dp, dp]
        lib.kdao_commit.argtypes = [i, i, i, i, ip, dp, dp, dp, dp, dp, ip, dp]
        lib.kdao_num_threads.restype = ctypes.c_int
        lib.kdao_set_num_threads.argtypes = [i]
        _lib = lib
    return _lib


def _d(a):
    """C-contiguous fp64 view (copy if needed) and its pointer."""
    a = np.ascontiguousarray(a, dtype=np.float64)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _i(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


_NULL_D = ctypes.POINTER(ctypes.c_double)()
_NULL_I = ctypes.POINTER(ctypes.c_int32)()


def num_threads() -> int:
    return _load().kdao_num_threads()


def set_num_threads(n: int) -> None:
    _load().kdao_set_num_threads(int(n))


def step(S, q, k, v, alpha, beta):
    """One token on one state.  Returns (S_t, o_t); S is not modified."""
    S = np.array(S, dtype=np.float64, order="C", copy=True)
    dk, dv = S.shape
    q, qp = _d(q)
    k, kp = _d(k)
    v, vp = _d(v)
    alpha, ap = _d(alpha)
    o = np.zeros(dv, dtype=np.float64)
    _load().kdao_step(dk, dv, S.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                      qp, kp, vp, ap, float(beta),
                      o.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return S, o


def prefill(cu_seqlens, q, k, v, alpha, beta, S_in, start_pos=None,
            ckpt_every=0, max_ckpt=0):
    """Run every token of every sequence.

    Shapes: q, k, alpha [N][H][d_k]; v [N][H][d_v]; beta [N][H];
    S_in [B][H][d_k][d_v].  Returns (o [N][H][d_v], S_out [B][H][d_k][d_v],
    ckpt [B][max_ckpt][H][d_k][d_v], n_ckpt [B]).
    """
    cu, cup = _i(cu_seqlens)
    B = cu.shape[0] - 1
    N, H, dk = np.shape(k)
    dv = np.shape(v)[2]
    q, qp = _d(q)
    k, kp = _d(k)
    v, vp = _d(v)
    alpha, ap = _d(alpha)
    beta, bp = _d(beta)
    S_in, sip = _d(S_in)
    S_out = np.zeros((B, H, dk, dv))
    o = np.zeros((N, H, dv))
    ck = np.zeros((B, max(max_ckpt, 0), H, dk, dv))
    nck = np.zeros(B, dtype=np.int32)
    if start_pos is None:
        spp = _NULL_I
    else:
        sp, spp = _i(start_pos)
    _load().kdao_prefill(
        B, H, dk, dv, cup, qp, kp, vp, ap, bp, sip,
        S_out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
        o.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), spp,
        int(ckpt_every), int(max_ckpt),
        ck.ctypes.data_as(ctypes.POINTER(ctypes.c_double)) if max_ckpt > 0
        else _NULL_D,
        nck.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))
    return o, S_out, ck, nck


def verify(cu_seqlens, q, k, v, alpha, beta, S):
    """Outputs of every segment run on a copy of S [B][H][d_k][d_v]."""
    cu, cup = _i(cu_seqlens)
    B = cu.shape[0] - 1
    N, H, dk = np.shape(k)
    dv = np.shape(v)[2]
    q, qp = _d(q)
    k, kp = _d(k)
    v, vp = _d(v)
    alpha, ap = _d(alpha)
    beta, bp = _d(beta)
    S, sp = _d(S)
    o = np.zeros((N, H, dv))
    _load().kdao_verify(B, H, dk, dv, cup, qp, kp, vp, ap, bp, sp,
                        o.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return o


def commit(cu_seqlens, q, k, v, alpha, beta, accepted_len, S):
    """State after the first accepted_len[i] tokens of each segment (new array)."""
    cu, cup = _i(cu_seqlens)
    B = cu.shape[0] - 1
    N, H, dk = np.shape(k)
    dv = np.shape(v)[2]
    q, qp = _d(q)
    k, kp = _d(k)
    v, vp = _d(v)
    alpha, ap = _d(alpha)
    beta, bp = _d(beta)
    acc, accp = _i(accepted_len)
    S = np.array(S, dtype=np.float64, order="C", copy=True)
    _load().kdao_commit(B, H, dk, dv, cup, qp, kp, vp, ap, bp, accp,
                        S.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return S


def prep_inputs(q, k_raw, z_alpha, z_beta):
    """The input-side preparation in front of the path, in fp64: the pages do
    not define it, so it follows the input generator's formulas for the
    synthetic workloads -- each key L2-normalised over d_k per (token, head),
    alpha = exp(-softplus(z_alpha)) per key channel, beta = sigmoid(z_beta)
    per (token, head); q is used as given.  Returns (q, k, alpha, beta)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k_raw, dtype=np.float64)
    nrm = np.sqrt((k * k).sum(-1, keepdims=True))
    k = k / np.maximum(nrm, 1e-12)
    alpha = np.exp(-np.logaddexp(0.0, np.asarray(z_alpha, dtype=np.float64)))
    beta = 1.0 / (1.0 + np.exp(-np.asarray(z_beta, dtype=np.float64)))
    return q, k, alpha, beta


class OracleSession:
    """Paged state pool plus the speculative protocol, evaluated eagerly.

    ``pool[slot]`` is the committed state ``[H][d_k][d_v]`` of whatever
    sequence owns the slot.  ``pending[slot]`` holds the drafted tokens of the
    last verify of that slot until the matching commit.
    """

    def __init__(self, num_slots, H, dk, dv, init=None):
        self.H, self.dk, self.dv = H, dk, dv
        self.pool = (np.zeros((num_slots, H, dk, dv)) if init is None
                     else np.array(init, dtype=np.float64, copy=True))
        self.pending = {}

    @staticmethod
    def _segment(tok, i):
        lo, hi = int(tok["cu_seqlens"][i]), int(tok["cu_seqlens"][i + 1])
        return {n: np.asarray(tok[n][lo:hi], dtype=np.float64)
                for n in ("q", "k", "v", "alpha", "beta")}

    def prefill(self, tok, slots, ckpt_every=0, ckpt_slots=None,
                start_pos=None):
        """Prefill every sequence from pool[slot]; checkpoints into ckpt slots.

        ckpt_slots [B][max_ckpt] (entries < 0 are skipped).  Returns outputs
        [N][H][d_v] and the number of checkpoints each sequence crossed.
        """
        slots = np.asarray(slots)
        max_ckpt = 0 if ckpt_slots is None else np.shape(ckpt_slots)[1]
        o, S_out, ck, nck = prefill(
            tok["cu_seqlens"], tok["q"], tok["k"], tok["v"], tok["alpha"],
            tok["beta"], self.pool[slots], start_pos=start_pos,
            ckpt_every=ckpt_every, max_ckpt=max_ckpt)
        for i, s in enumerate(slots):
            self.pool[s] = S_out[i]
            self.pending.pop(int(s), None)
            for m in range(min(int(nck[i]), max_ckpt)):
                cs = int(ckpt_slots[i][m])
                if cs >= 0:
                    self.pool[cs] = ck[i, m]
        return o, nck

    def verify(self, tok, slots, is_spec=None):
        """Outputs of one verify launch; ordinary (non-spec) rows commit now."""
        slots = np.asarray(slots)
        B = len(slots)
        spec = np.ones(B, dtype=bool) if is_spec is None else np.asarray(
            is_spec, dtype=bool)
        o = verify(tok["cu_seqlens"], tok["q"], tok["k"], tok["v"],
                   tok["alpha"], tok["beta"], self.pool[slots])
        for i in range(B):
            s = int(slots[i])
            seg = self._segment(tok, i)
            n = seg["k"].shape[0]
            if spec[i]:
                self.pending[s] = seg
            else:
                cu = np.array([0, n], dtype=np.int32)
                self.pool[s] = commit(cu, seg["q"], seg["k"], seg["v"],
                                      seg["alpha"], seg["beta"],
                                      np.array([n], dtype=np.int32),
                                      self.pool[s][None])[0]
                self.pending.pop(s, None)
        return o

    def commit(self, accepted_len, slots):
        """Fold the first accepted_len[i] drafted tokens into pool[slot]."""
        for a, s in zip(np.asarray(accepted_len), np.asarray(slots)):
            s = int(s)
            seg = self.pending.pop(s, None)
            if seg is None or int(a) == 0:
                continue
            n = seg["k"].shape[0]
            cu = np.array([0, n], dtype=np.int32)
            self.pool[s] = commit(cu, seg["q"], seg["k"], seg["v"],
                                  seg["alpha"], seg["beta"],
                                  np.array([int(a)], dtype=np.int32),
                                  self.pool[s][None])[0]

    def copy_slots(self, src, dst):
        for a, b in zip(np.asarray(src), np.asarray(dst)):
            self.pool[int(b)] = self.pool[int(a)]
