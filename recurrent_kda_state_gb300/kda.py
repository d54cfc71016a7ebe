"""ctypes binding of libkda.so (argument marshalling only).

Every function here has the name of the C entry point it calls and does
nothing but turn torch tensors into pointers and sizes; all arithmetic of the
path runs in the library's CUDA kernels.  The library must have been built
(``recurrent_kda_state_gb300._build.build_library``); if it is missing the
first call raises, there is no fallback.
"""
import ctypes
import os

import torch

from ._build import LIB

KDA_OK, KDA_EINVAL, KDA_EDTYPE, KDA_ESHAPE, KDA_EALIGN = 0, -1, -2, -3, -4
KDA_EPROTO, KDA_ECUDA, KDA_EDEVICE, KDA_ENOSPC = -5, -6, -7, -8
KDA_DERR_SLOT, KDA_DERR_ACCEPT, KDA_DERR_DEPTH = 1, 2, 4
KDA_DERR_SEGMENT, KDA_DERR_RING, KDA_DERR_RANGE = 8, 16, 32
KDA_DERR_TIMEOUT, KDA_DERR_UNSAFE = 64, 128
KDA_F32, KDA_BF16 = 0, 1

_P = ctypes.c_void_p
_I32 = ctypes.c_int32


class kda_tokens(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("q", _P), ("k", _P), ("v", _P),
                ("alpha", _P), ("beta", _P), ("o", _P), ("cu_seqlens", _P),
                ("num_seqs", _I32), ("num_tokens", _I32), ("num_heads", _I32),
                ("d_k", _I32), ("d_v", _I32)]


class kda_state_pool(ctypes.Structure):
    _fields_ = [("base", _P), ("num_slots", _I32), ("num_heads", _I32),
                ("d_k", _I32), ("d_v", _I32)]


class kda_replay_ring(ctypes.Structure):
    _fields_ = [("k", _P), ("v", _P), ("alpha", _P), ("beta", _P),
                ("ctrl", _P), ("depth", _I32), ("dtype", ctypes.c_int)]


EXPORTS = ("kda_prefill_chunked", "kda_prefill_chunked_raw", "kda_prefill_chunked_noalloc",
           "kda_prefill_workspace_size", "kda_verify", "kda_verify_raw",
           "kda_commit", "kda_commit_layers", "kda_materialize", "kda_ring_reset",
           "kda_gather_states", "kda_copy_slots", "kda_verify_snapshot",
           "kda_commit_snapshot", "kda_forward_mixed", "kda_get_device_error",
           "kda_set_wait_limit", "kda_status_string", "kda_version")

_lib = None


def lib():
    """The loaded libkda.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(
                "libkda.so is not built (%s); run __graft_entry__.build()" % LIB)
        L = ctypes.CDLL(LIB)
        tp, pp, rp = (ctypes.POINTER(kda_tokens), ctypes.POINTER(kda_state_pool),
                      ctypes.POINTER(kda_replay_ring))
        L.kda_prefill_chunked.argtypes = [tp, pp, _P, _P, _I32, _I32, _I32, _P,
                                          _P, ctypes.c_size_t, _P]
        L.kda_prefill_chunked_raw.argtypes = [tp, pp, _P, _P, _I32, _I32, _I32, _P,
                                              _P, ctypes.c_size_t, _P]
        L.kda_prefill_chunked_noalloc.argtypes = [tp, pp, _P, _P, _I32, _I32,
                                                  _I32, _P, _P]
        L.kda_prefill_workspace_size.argtypes = [_I32] * 6 + [ctypes.c_int]
        L.kda_prefill_workspace_size.restype = ctypes.c_size_t
        L.kda_verify.argtypes = [tp, _I32, pp, _P, rp, _P, _P]
        L.kda_verify_raw.argtypes = [tp, _I32, pp, _P, rp, _P, _P]
        L.kda_commit.argtypes = [_P, _P, _I32, pp, rp, _P]
        L.kda_commit_layers.argtypes = [_P, _P, _I32, pp, rp, _I32, _P]
        L.kda_materialize.argtypes = [_P, _I32, pp, rp, _P]
        L.kda_ring_reset.argtypes = [_P, _I32, pp, rp, _P]
        L.kda_gather_states.argtypes = [pp, _P, _I32, _P, _P]
        L.kda_copy_slots.argtypes = [pp, _P, _P, _I32, _P]
        L.kda_verify_snapshot.argtypes = [tp, _I32, pp, _P, _P, _P]
        L.kda_forward_mixed.argtypes = [tp, _I32, _I32, pp, _P, _P, _I32, _I32, _I32,
                                        _P, _P, ctypes.c_size_t, _I32, rp, _P, _P, _P]
        L.kda_commit_snapshot.argtypes = [_P, _P, _I32, pp, _P, _I32, _P]
        L.kda_get_device_error.argtypes = [ctypes.POINTER(_I32), _P]
        L.kda_set_wait_limit.argtypes = [_I32]
        L.kda_status_string.argtypes = [ctypes.c_int]
        L.kda_status_string.restype = ctypes.c_char_p
        L.kda_version.restype = ctypes.c_int
        for name in EXPORTS:
            getattr(L, name).restype = getattr(L, name).restype or ctypes.c_int
        _lib = L
    return _lib


class KdaError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = lib().kda_status_string(status).decode()
        super().__init__("%s: %s" % (where, msg))


def _check(status, where):
    if status != KDA_OK:
        raise KdaError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(dt):
    if dt == torch.float32:
        return KDA_F32
    if dt == torch.bfloat16:
        return KDA_BF16
    raise ValueError("unsupported input dtype %s" % dt)


class StatePool:
    """fp32 states [num_slots][H][d_v][d_k] (each column of S contiguous)."""

    def __init__(self, data):
        assert data.dtype == torch.float32 and data.dim() == 4
        assert data.is_contiguous()
        self.data = data
        P, H, dv, dk = data.shape
        self.c = kda_state_pool(data.data_ptr(), P, H, dk, dv)

    @classmethod
    def zeros(cls, num_slots, H, d, device="cuda"):
        return cls(torch.zeros(num_slots, H, d, d, dtype=torch.float32,
                               device=device))


class ReplayRing:
    """ReplaySSM ring for one pool: payload [P][H][depth][d] + ctrl [P][H][2]."""

    def __init__(self, num_slots, H, d, depth, dtype, device="cuda"):
        self.k = torch.zeros(num_slots, H, depth, d, dtype=dtype, device=device)
        self.v = torch.zeros_like(self.k)
        self.alpha = torch.zeros_like(self.k)
        self.beta = torch.zeros(num_slots, H, depth, dtype=dtype, device=device)
        self.ctrl = torch.zeros(num_slots, H, 2, dtype=torch.int32, device=device)
        self.depth = depth
        self.c = kda_replay_ring(self.k.data_ptr(), self.v.data_ptr(),
                                 self.alpha.data_ptr(), self.beta.data_ptr(),
                                 self.ctrl.data_ptr(), depth, _dtype_code(dtype))


class TokenBatch:
    """Packed tokens q, k, alpha [N][H][d_k], v [N][H][d_v], beta [N][H],
    fp32 outputs o [N][H][d_v] and cu_seqlens [B + 1] (int32, device)."""

    def __init__(self, q, k, v, alpha, beta, cu_seqlens, o=None):
        self.q, self.k, self.v, self.alpha, self.beta = q, k, v, alpha, beta
        self.cu_seqlens = cu_seqlens
        N, H, dk = k.shape
        dv = v.shape[2]
        self.o = o if o is not None else torch.empty(
            N, H, dv, dtype=torch.float32, device=k.device)
        for t in (q, k, v, alpha, beta, self.o, cu_seqlens):
            assert t.is_contiguous()
        self.c = kda_tokens(_dtype_code(k.dtype), q.data_ptr(), k.data_ptr(),
                            v.data_ptr(), alpha.data_ptr(), beta.data_ptr(),
                            self.o.data_ptr(), cu_seqlens.data_ptr(),
                            cu_seqlens.numel() - 1, N, H, dk, dv)


def kda_prefill_workspace_size(num_tokens, num_seqs, H, d_k, d_v, chunk, dtype):
    """Workspace bytes for these sizes and input dtype (KDA_F32 / KDA_BF16);
    0 when the call needs none."""
    return int(lib().kda_prefill_workspace_size(num_tokens, num_seqs, H, d_k,
                                                d_v, chunk, dtype))


def kda_prefill_chunked(tok, pool, state_slots, chunk, ckpt_every=0,
                        ckpt_slots=None, start_pos=None, workspace=None,
                        stream=None, single_pass=False, raw=False):
    """Chunked prefill; ckpt_slots [B][max_ckpt] int32 (device) or None.
    workspace None: one of the required size is allocated here;
    single_pass: pass no workspace (the tensor-core shape's single pass);
    raw: projection-space inputs, prep fused (kda_prefill_chunked_raw)."""
    max_ckpt = 0 if ckpt_slots is None else int(ckpt_slots.shape[1])
    if single_pass:
        workspace = None
    elif workspace is None:
        nbytes = kda_prefill_workspace_size(tok.c.num_tokens, tok.c.num_seqs,
                                            tok.c.num_heads, tok.c.d_k,
                                            tok.c.d_v, chunk, tok.c.dtype)
        if nbytes > 0:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=tok.k.device)
    fn, name = ((lib().kda_prefill_chunked_raw, "kda_prefill_chunked_raw") if raw
                else (lib().kda_prefill_chunked, "kda_prefill_chunked"))
    _check(fn(
        ctypes.byref(tok.c), ctypes.byref(pool.c), _ptr(state_slots),
        _ptr(ckpt_slots), max_ckpt, ckpt_every, chunk, _ptr(start_pos),
        _ptr(workspace), 0 if workspace is None else workspace.numel(),
        _stream(stream)), name)
    return workspace


KDA_NOALLOC_SCRATCH_BYTES = 64 << 20


def kda_prefill_chunked_noalloc(tok, pool, state_slots, chunk, ckpt_every=0,
                                ckpt_slots=None, start_pos=None, stream=None):
    """kda_prefill_chunked with the library's own fixed scratch instead of a
    workspace argument, for callers that cannot allocate device memory."""
    max_ckpt = 0 if ckpt_slots is None else int(ckpt_slots.shape[1])
    _check(lib().kda_prefill_chunked_noalloc(
        ctypes.byref(tok.c), ctypes.byref(pool.c), _ptr(state_slots),
        _ptr(ckpt_slots), max_ckpt, ckpt_every, chunk, _ptr(start_pos),
        _stream(stream)), "kda_prefill_chunked_noalloc")


def kda_verify(tok, max_T, pool, state_slots, ring, is_spec=None, stream=None,
               raw=False):
    """raw: projection-space keys, decay and beta logits, prep fused
    (kda_verify_raw)."""
    fn, name = ((lib().kda_verify_raw, "kda_verify_raw") if raw
                else (lib().kda_verify, "kda_verify"))
    _check(fn(ctypes.byref(tok.c), max_T, ctypes.byref(pool.c), _ptr(state_slots),
              ctypes.byref(ring.c), _ptr(is_spec), _stream(stream)), name)


def kda_forward_mixed(tok, num_prefill, prefill_tokens, pool, state_slots, chunk,
                      max_T, ring, ckpt_every=0, ckpt_slots=None, start_pos=None,
                      is_spec=None, workspace=None, single_pass=False, stream=None,
                      side_stream=None):
    """Prefill segments (the first num_prefill sequences, token rows
    [0, prefill_tokens)) and verify/decode segments of one packed batch in one
    call; side_stream: run the prefill part there, forked and joined."""
    max_ckpt = 0 if ckpt_slots is None else int(ckpt_slots.shape[1])
    if single_pass or num_prefill == 0:
        workspace = None
    elif workspace is None:
        nbytes = kda_prefill_workspace_size(prefill_tokens, num_prefill,
                                            tok.c.num_heads, tok.c.d_k, tok.c.d_v,
                                            chunk, tok.c.dtype)
        if nbytes > 0:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=tok.k.device)
    side = None if side_stream is None else ctypes.c_void_p(side_stream.cuda_stream)
    _check(lib().kda_forward_mixed(
        ctypes.byref(tok.c), num_prefill, prefill_tokens, ctypes.byref(pool.c),
        _ptr(state_slots), _ptr(ckpt_slots), max_ckpt, ckpt_every, chunk,
        _ptr(start_pos), _ptr(workspace),
        0 if workspace is None else workspace.numel(), max_T,
        ctypes.byref(ring.c), _ptr(is_spec), _stream(stream), side),
        "kda_forward_mixed")
    return workspace


def kda_commit(accepted_len, state_slots, pool, ring, stream=None):
    _check(lib().kda_commit(_ptr(accepted_len), _ptr(state_slots),
                            state_slots.numel(), ctypes.byref(pool.c),
                            ctypes.byref(ring.c), _stream(stream)), "kda_commit")


def kda_commit_layers(accepted_len, state_slots, pool, rings, stream=None):
    """kda_commit on several layers' rings (same pool geometry), one launch."""
    arr = (kda_replay_ring * len(rings))(*[r.c for r in rings])
    _check(lib().kda_commit_layers(_ptr(accepted_len), _ptr(state_slots),
                                   state_slots.numel(), ctypes.byref(pool.c),
                                   arr, len(rings), _stream(stream)),
           "kda_commit_layers")


def kda_materialize(state_slots, pool, ring, stream=None):
    _check(lib().kda_materialize(_ptr(state_slots), state_slots.numel(),
                                 ctypes.byref(pool.c), ctypes.byref(ring.c),
                                 _stream(stream)), "kda_materialize")


def kda_ring_reset(slots, pool, ring, stream=None):
    _check(lib().kda_ring_reset(_ptr(slots), slots.numel(), ctypes.byref(pool.c),
                                ctypes.byref(ring.c), _stream(stream)),
           "kda_ring_reset")


def kda_gather_states(pool, slots, out=None, stream=None):
    if out is None:
        P, H, dv, dk = pool.data.shape
        out = torch.empty(slots.numel(), H, dv, dk, dtype=torch.float32,
                          device=pool.data.device)
    _check(lib().kda_gather_states(ctypes.byref(pool.c), _ptr(slots),
                                   slots.numel(), _ptr(out), _stream(stream)),
           "kda_gather_states")
    return out


def kda_copy_slots(pool, src, dst, stream=None):
    _check(lib().kda_copy_slots(ctypes.byref(pool.c), _ptr(src), _ptr(dst),
                                src.numel(), _stream(stream)), "kda_copy_slots")


def snapshot_buffer(num_seqs, max_T, pool):
    """Per-position snapshots [num_seqs][max_T][H][d_v][d_k] fp32 for
    kda_verify_snapshot (the direct design's extra state cache)."""
    P, H, dv, dk = pool.data.shape
    return torch.empty(num_seqs, max_T, H, dv, dk, dtype=torch.float32,
                       device=pool.data.device)


def kda_verify_snapshot(tok, max_T, pool, state_slots, snapshots, stream=None):
    _check(lib().kda_verify_snapshot(ctypes.byref(tok.c), max_T,
                                     ctypes.byref(pool.c), _ptr(state_slots),
                                     _ptr(snapshots), _stream(stream)),
           "kda_verify_snapshot")


def kda_commit_snapshot(accepted_len, state_slots, pool, snapshots, stream=None):
    _check(lib().kda_commit_snapshot(_ptr(accepted_len), _ptr(state_slots),
                                     state_slots.numel(), ctypes.byref(pool.c),
                                     _ptr(snapshots), int(snapshots.shape[1]),
                                     _stream(stream)), "kda_commit_snapshot")


def kda_get_device_error(stream=None):
    """Synchronize, read and clear the device error word; returns its bits."""
    bits = _I32(0)
    st = lib().kda_get_device_error(ctypes.byref(bits), _stream(stream))
    if st not in (KDA_OK, KDA_EDEVICE):
        raise KdaError(st, "kda_get_device_error")
    return int(bits.value)


def kda_set_wait_limit(polls):
    """Testing hook: bounded device waits give up after `polls` polls
    (KDA_DERR_TIMEOUT); a negative value restores the default."""
    _check(lib().kda_set_wait_limit(int(polls)), "kda_set_wait_limit")
