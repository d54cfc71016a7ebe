"""C ABI checks that need no GPU: the library builds and loads, exports every
function include/kda.h declares, and rejects bad arguments on the host before
any CUDA call."""
import ctypes
import os
import re

import pytest

from recurrent_kda_state_gb300 import kda
from recurrent_kda_state_gb300._build import build_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build_library()
    return kda.lib()


def _declared():
    txt = open(os.path.join(ROOT, "include", "kda.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_]+)\s*\(", txt)))


def test_header_declares_the_calls():
    names = _declared()
    for n in ("kda_prefill_chunked", "kda_verify", "kda_commit",
              "kda_gather_states", "kda_materialize", "kda_copy_slots"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for name in _declared():
        assert hasattr(L, name), name
    assert set(_declared()) == set(kda.EXPORTS)


def test_version_and_status_strings(L):
    assert L.kda_version() == 1
    for st in range(0, -9, -1):
        assert L.kda_status_string(st).startswith(b"KDA_")


def _pool(base=0x10000, P=4, H=2, d=16):
    return kda.kda_state_pool(base, P, H, d, d)


def _tokens(dtype=kda.KDA_F32, B=1, N=4, H=2, d=16, ptr=0x20000):
    return kda.kda_tokens(dtype, ptr, ptr, ptr, ptr, ptr, ptr, ptr, B, N, H, d, d)


def _ring(depth=4, dtype=kda.KDA_F32, ptr=0x30000):
    return kda.kda_replay_ring(ptr, ptr, ptr, ptr, ptr, depth, dtype)


def test_verify_validation(L):
    pool, tok, ring = _pool(), _tokens(), _ring()
    s = ctypes.c_void_p(0x40000)
    by = ctypes.byref
    assert L.kda_verify(None, 4, by(pool), s, by(ring), None, None) == kda.KDA_EINVAL
    bad = _pool(d=48)
    assert L.kda_verify(by(tok), 4, by(bad), s, by(ring), None, None) == kda.KDA_ESHAPE
    mis = _tokens(H=3)
    assert L.kda_verify(by(mis), 4, by(pool), s, by(ring), None, None) == kda.KDA_ESHAPE
    una = _tokens(ptr=0x20004)
    assert L.kda_verify(by(una), 4, by(pool), s, by(ring), None, None) == kda.KDA_EALIGN
    r16 = _ring(dtype=kda.KDA_BF16)
    assert L.kda_verify(by(tok), 4, by(pool), s, by(r16), None, None) == kda.KDA_EDTYPE
    # all-speculative launch with T above the ring depth
    assert L.kda_verify(by(tok), 5, by(pool), s, by(ring), None, None) == kda.KDA_EPROTO
    assert L.kda_verify(by(tok), -1, by(pool), s, by(ring), None, None) == kda.KDA_EINVAL
    dt = _tokens(dtype=7)
    assert L.kda_verify(by(dt), 4, by(pool), s, by(ring), None, None) == kda.KDA_EDTYPE


def test_prefill_validation(L):
    pool, tok = _pool(), _tokens()
    by = ctypes.byref
    s = ctypes.c_void_p(0x40000)
    ws = ctypes.c_void_p(0x100000)
    need = L.kda_prefill_workspace_size(4, 1, 2, 16, 16, 16, kda.KDA_F32)
    assert need > 0
    # chunk not supported
    assert L.kda_prefill_chunked(by(tok), by(pool), s, None, 0, 0, 24, None, ws,
                                 need, None) == kda.KDA_EINVAL
    # checkpoint spacing not a multiple of the chunk
    assert L.kda_prefill_chunked(by(tok), by(pool), s, s, 1, 24, 16, None, ws,
                                 need, None) == kda.KDA_EINVAL
    # workspace too small / misaligned
    assert L.kda_prefill_chunked(by(tok), by(pool), s, None, 0, 0, 16, None, ws,
                                 need - 1, None) == kda.KDA_ENOSPC
    assert L.kda_prefill_chunked(by(tok), by(pool), s, None, 0, 0, 16, None,
                                 ctypes.c_void_p(0x100010), need,
                                 None) == kda.KDA_EALIGN
    assert L.kda_prefill_workspace_size(4, 1, 2, 16, 16, 24, kda.KDA_F32) == 0
    # no workspace at all is refused where one is needed
    assert L.kda_prefill_chunked(by(tok), by(pool), s, None, 0, 0, 16, None, None,
                                 0, None) == kda.KDA_EINVAL


def test_workspace_size_formula(L):
    # table (B+1 int32, 256-byte padded) + (N/C + 2B) chunks x H x entry,
    # entry = 4*C*D + C*C + D floats rounded up to 64 floats
    N, B, H, D, C = 8192, 1, 32, 128, 64
    entry = (4 * C * D + C * C + D + 63) // 64 * 64
    want = 256 + (N // C + 2 * B) * H * entry * 4
    assert L.kda_prefill_workspace_size(N, B, H, D, D, C, kda.KDA_F32) == want
    # bf16 at d=128, chunk 64, heads a multiple of 8: the two-pass
    # tensor-core path, table padded to 1 KiB + (N/C + 2B) x H entries of
    # 165888 bytes (tile images, U', decay vectors); other bf16 shapes follow
    # the formula above
    assert L.kda_prefill_workspace_size(N, B, H, D, D, C, kda.KDA_BF16) == \
        1024 + (N // C + 2 * B) * H * 165888
    assert L.kda_prefill_workspace_size(N, B, 4, D, D, C, kda.KDA_BF16) == \
        256 + (N // C + 2 * B) * 4 * entry * 4
    assert L.kda_prefill_workspace_size(N, B, H, D, D, 32, kda.KDA_BF16) > 0
    assert L.kda_prefill_workspace_size(N, B, H, D, D, C, 7) == 0


def test_commit_and_slot_validation(L):
    pool, ring = _pool(), _ring()
    by = ctypes.byref
    s = ctypes.c_void_p(0x40000)
    assert L.kda_commit(None, s, 1, by(pool), by(ring), None) == kda.KDA_EINVAL
    assert L.kda_commit(s, s, -1, by(pool), by(ring), None) == kda.KDA_EINVAL
    assert L.kda_commit(s, s, 0, by(pool), by(ring), None) == kda.KDA_OK
    assert L.kda_materialize(s, -2, by(pool), by(ring), None) == kda.KDA_EINVAL
    assert L.kda_gather_states(by(pool), s, 1, ctypes.c_void_p(0x50008),
                               None) == kda.KDA_EALIGN
    assert L.kda_copy_slots(by(pool), None, s, 1, None) == kda.KDA_EINVAL
    assert L.kda_ring_reset(s, 1, by(pool), None, None) == kda.KDA_EINVAL
    rings = (kda.kda_replay_ring * 2)(_ring(), _ring())
    assert L.kda_commit_layers(s, s, 1, by(pool), rings, 65, None) == kda.KDA_EINVAL
    assert L.kda_commit_layers(s, s, 1, by(pool), None, 2, None) == kda.KDA_EINVAL
    assert L.kda_commit_layers(s, s, 0, by(pool), rings, 2, None) == kda.KDA_OK
    assert L.kda_get_device_error(None, None) == kda.KDA_EINVAL


def test_snapshot_validation(L):
    """The direct-snapshot ablation calls reject bad arguments on the host."""
    pool, tok = _pool(), _tokens()
    by = ctypes.byref
    s = ctypes.c_void_p(0x40000)
    snap = ctypes.c_void_p(0x60000)
    assert L.kda_verify_snapshot(None, 4, by(pool), s, snap, None) == kda.KDA_EINVAL
    assert L.kda_verify_snapshot(by(tok), 0, by(pool), s, snap, None) == kda.KDA_EINVAL
    assert L.kda_verify_snapshot(by(tok), 17, by(pool), s, snap, None) == kda.KDA_EINVAL
    assert L.kda_verify_snapshot(by(tok), 4, by(pool), s, None, None) == kda.KDA_EINVAL
    assert L.kda_verify_snapshot(by(tok), 4, by(pool), None, snap, None) == kda.KDA_EINVAL
    assert L.kda_verify_snapshot(by(tok), 4, by(pool), s, ctypes.c_void_p(0x60004),
                                 None) == kda.KDA_EALIGN
    bad = _pool(d=48)
    assert L.kda_verify_snapshot(by(tok), 4, by(bad), s, snap, None) == kda.KDA_ESHAPE
    none = _tokens(B=0, N=0)
    assert L.kda_verify_snapshot(by(none), 4, by(pool), None, None, None) == kda.KDA_OK
    assert L.kda_commit_snapshot(None, s, 1, by(pool), snap, 4, None) == kda.KDA_EINVAL
    assert L.kda_commit_snapshot(s, s, 1, by(pool), None, 4, None) == kda.KDA_EINVAL
    assert L.kda_commit_snapshot(s, s, -1, by(pool), snap, 4, None) == kda.KDA_EINVAL
    assert L.kda_commit_snapshot(s, s, 1, by(pool), snap, 0, None) == kda.KDA_EINVAL
    assert L.kda_commit_snapshot(s, s, 1, by(pool), ctypes.c_void_p(0x60008), 4,
                                 None) == kda.KDA_EALIGN
    assert L.kda_commit_snapshot(s, s, 0, by(pool), snap, 4, None) == kda.KDA_OK


def test_forward_mixed_validation(L):
    """The mixed prefill + verify call checks its split on the host."""
    pool, tok, ring = _pool(), _tokens(B=2, N=8), _ring()
    by = ctypes.byref
    s = ctypes.c_void_p(0x40000)

    def call(npf, ptok, slots=s, ring_=ring, max_T=4, chunk=16):
        return L.kda_forward_mixed(by(tok), npf, ptok, by(pool), slots, None, 0, 0,
                                   chunk, None, None, 0, max_T,
                                   by(ring_) if ring_ is not None else None,
                                   None, None, None)
    assert call(3, 0) == kda.KDA_EINVAL          # more prefill rows than sequences
    assert call(-1, 0) == kda.KDA_EINVAL
    assert call(1, 9) == kda.KDA_EINVAL          # beyond the batch's tokens
    assert call(0, 4) == kda.KDA_EINVAL          # prefill tokens without sequences
    assert call(1, 4, slots=None) == kda.KDA_EINVAL
    assert call(1, 4, ring_=None) == kda.KDA_EINVAL   # the verify part needs a ring
    assert call(1, 4, max_T=5) == kda.KDA_EPROTO      # drafts longer than the ring
    assert call(1, 4, chunk=24) == kda.KDA_EINVAL     # prefill chunk size
    none = _tokens(B=0, N=0)
    assert L.kda_forward_mixed(by(none), 0, 0, by(pool), None, None, 0, 0, 16, None,
                               None, 0, 4, by(ring), None, None, None) == kda.KDA_OK


def test_prefill_raw_needs_the_tensor_core_shape(L):
    """The fused-prep prefill exists only where the prep is fused."""
    pool, tok = _pool(), _tokens()
    s = ctypes.c_void_p(0x40000)
    ws = ctypes.c_void_p(0x80000)
    assert L.kda_prefill_chunked_raw(ctypes.byref(tok), ctypes.byref(pool), s, None, 0, 0,
                                     16, None, ws, 1 << 20, None) == kda.KDA_ESHAPE


def test_verify_raw_needs_the_pipelined_shape(L):
    """The fused-prep verify exists only where the prep is fused: bf16 tokens,
    d = 128, ring depth <= 8, at most 8 tokens per row; every other shape is
    refused on the host."""
    by = ctypes.byref
    s = ctypes.c_void_p(0x40000)
    pool16, tok16, ring16 = _pool(), _tokens(), _ring()
    assert L.kda_verify_raw(by(tok16), 4, by(pool16), s, by(ring16), None,
                            None) == kda.KDA_ESHAPE                     # d = 16, fp32
    pool = _pool(P=4, H=2, d=128)
    tok = _tokens(dtype=kda.KDA_BF16, d=128)
    deep = _ring(depth=9, dtype=kda.KDA_BF16)
    assert L.kda_verify_raw(by(tok), 4, by(pool), s, by(deep), None,
                            None) == kda.KDA_ESHAPE                     # ring depth 9
    ring = _ring(depth=8, dtype=kda.KDA_BF16)
    flag = ctypes.c_void_p(0x50000)
    assert L.kda_verify_raw(by(tok), 9, by(pool), s, by(ring), flag,
                            None) == kda.KDA_ESHAPE                     # 9 tokens per row
    f32 = _tokens(dtype=kda.KDA_F32, d=128)
    r32 = _ring(depth=8, dtype=kda.KDA_F32)
    assert L.kda_verify_raw(by(f32), 4, by(pool), s, by(r32), None,
                            None) == kda.KDA_ESHAPE                     # fp32 tokens
