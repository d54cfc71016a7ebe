"""Helpers for the GPU parity tests: move seeded inputs to the device, convert
between the oracle's state orientation [d_k][d_v] and the library's
[d_v][d_k], and measure errors with the tolerances of the path
(outputs max-abs <= 2e-3, states relative Frobenius <= 1e-3)."""
import numpy as np
import torch

from recurrent_kda_state_gb300 import kda as K

OUT_TOL = 2e-3
STATE_TOL = 1e-3
TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def device_batch(tok, dtype, device="cuda"):
    dt = TORCH_DT[dtype]

    def t(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device=device,
                                                             dtype=dt)
    cu = torch.from_numpy(np.asarray(tok["cu_seqlens"], dtype=np.int32)).to(device)
    return K.TokenBatch(t(tok["q"]), t(tok["k"]), t(tok["v"]), t(tok["alpha"]),
                        t(tok["beta"]), cu)


def i32(x, device="cuda"):
    return torch.as_tensor(np.asarray(x, dtype=np.int32), device=device)


def to_gpu_states(S):
    """oracle [..., d_k, d_v] -> library fp32 [..., d_v, d_k] (CPU tensor)."""
    return torch.from_numpy(np.ascontiguousarray(
        np.swapaxes(np.asarray(S), -1, -2)).astype(np.float32))


def from_gpu_states(t):
    """library [..., d_v, d_k] -> oracle orientation fp64 numpy."""
    return np.swapaxes(t.detach().cpu().numpy().astype(np.float64), -1, -2)


def heads(tok, hs):
    """The token tensors restricted to heads hs (oracle-side sampling)."""
    out = {n: np.ascontiguousarray(tok[n][:, hs])
           for n in ("q", "k", "v", "alpha", "beta")}
    out["cu_seqlens"] = tok["cu_seqlens"]
    return out


def max_abs(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b))) if a.size else 0.0


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def assert_outputs(got, want, tol=OUT_TOL):
    err = max_abs(got, want)
    assert err <= tol, "outputs max-abs error %.3e > %.1e" % (err, tol)


def assert_states(got, want, tol=STATE_TOL):
    err = rel_fro(got, want)
    assert err <= tol, "state relative Frobenius error %.3e > %.1e" % (err, tol)
