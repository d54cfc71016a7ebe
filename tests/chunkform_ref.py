"""fp64 numpy statement of the chunk-wise (WY/UT) form of the KDA recurrence.

Test-only.  It restates, per chunk of C tokens, the algebra the CUDA prefill
implements, so a test can check that algebra against the token-by-token
oracle before any kernel is trusted:

    g_t   = sum_{s<=t} log alpha_s                (per key channel, inclusive)
    A_ts  = beta_t sum_c k_tc k_sc exp(g_tc - g_sc)        for s < t
    T     = (I + A)^{-1} diag(beta)
    W     = T (exp(g) * K),   U' = T V,   U = U' - W S
    O     = (exp(g) * Q) S + M U,   M_ts = sum_c q_tc k_sc exp(g_tc - g_sc), s <= t
    S'    = Diag(exp(g_C)) S + (exp(g_C - g) * K)^T U

Chunks are aligned to absolute positions (start_pos + local index), so a
checkpoint boundary that is a multiple of C always ends a chunk.
"""
import numpy as np


def chunk_prefill_one(q, k, v, alpha, beta, S0, C, start_pos=0, ckpt_every=0):
    """One (sequence, head).  Returns (o [L][d_v], S_final, [checkpoints])."""
    q, k, v, alpha, beta = (np.asarray(x, dtype=np.float64)
                            for x in (q, k, v, alpha, beta))
    S = np.array(S0, dtype=np.float64, copy=True)
    L = k.shape[0]
    o = np.zeros((L, v.shape[1]))
    ckpts = []
    t0 = 0
    while t0 < L:
        p = start_pos + t0
        end = min(L, t0 + (C - p % C))
        n = end - t0
        kc, qc, vc = k[t0:end], q[t0:end], v[t0:end]
        bc = beta[t0:end]
        g = np.cumsum(np.log(alpha[t0:end]), axis=0)
        D = np.exp(g[:, None, :] - g[None, :, :])  # [t][s][c], used for s <= t
        A = np.zeros((n, n))
        M = np.zeros((n, n))
        for t in range(n):
            for s in range(t + 1):
                if s < t:
                    A[t, s] = bc[t] * np.sum(kc[t] * kc[s] * D[t, s])
                M[t, s] = np.sum(qc[t] * kc[s] * D[t, s])
        Tm = np.linalg.solve(np.eye(n) + A, np.diag(bc))
        W = Tm @ (np.exp(g) * kc)
        U = Tm @ vc - W @ S
        o[t0:end] = (np.exp(g) * qc) @ S + M @ U
        Kbar = np.exp(g[-1][None, :] - g) * kc
        S = np.exp(g[-1])[:, None] * S + Kbar.T @ U
        if ckpt_every > 0 and (start_pos + end) % ckpt_every == 0:
            ckpts.append(S.copy())
        t0 = end
    return o, S, ckpts
