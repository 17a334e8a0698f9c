"""Chunk-parallel form of the KDA recurrence in numpy (fp64), for CPU tests.

This is the WY/UT chunk formulation that the CUDA prefill kernels implement,
written out plainly so that its algebra can be checked against the
token-by-token oracle on the CPU (Lecture 04, section 1: one chunk reduces to
one affine update that does not depend on the incoming state; section 4: the
recurrent and chunked executions agree on outputs and on the state at every
chunk boundary).  It is test code only and shares nothing with the kernels.

For a chunk of tokens r = 0..L'-1 with incoming state S:
    b_r    = sum_{s<=r} g_s                     (per channel)
    A[r,s] = beta_r sum_c k_rc k_sc exp(b_rc - b_sc),  s < r
    P[r,s] = sum_c q_rc k_sc exp(b_rc - b_sc),         s <= r
    (I + A) [W | U~] = diag(beta) [K_G | V],   K_G[r] = exp(b_r) * k_r
    U      = U~ - W S
    O      = Q_G S + P U = (Q_G - P W) S + P U~,  Q_G[r] = exp(b_r) * q_r
    S_next = diag(exp(b_last)) S + K_end^T U,  K_end[s] = exp(b_last - b_s) * k_s
"""
import numpy as np


def chunk_prepare(q, k, v, g, beta):
    """Everything of one chunk that does not depend on the incoming state."""
    Lc = q.shape[0]
    b = np.cumsum(g, axis=0)
    diff = b[:, None, :] - b[None, :, :]  # [r, s, c] = b_r - b_s
    mask_strict = np.tril(np.ones((Lc, Lc)), -1)
    mask_incl = np.tril(np.ones((Lc, Lc)), 0)
    # exp only where s <= r: there b_r - b_s <= 0 for non-positive g
    E = np.where(mask_incl[:, :, None] > 0, np.exp(np.minimum(diff, 0.0) if np.all(g <= 0) else diff), 0.0)
    A = beta[:, None] * np.einsum("rc,sc,rsc->rs", k, k, E) * mask_strict
    P = np.einsum("rc,sc,rsc->rs", q, k, E) * mask_incl
    KG = np.exp(b) * k
    QG = np.exp(b) * q
    Kend = np.exp(b[-1][None, :] - b) * k
    M = np.eye(Lc) + A
    W = np.linalg.solve(M, beta[:, None] * KG)
    Ut = np.linalg.solve(M, beta[:, None] * v)
    return dict(W=W, Ut=Ut, Qp=QG - P @ W, Oloc=P @ Ut, Kend=Kend, gamma=np.exp(b[-1]))


def chunk_apply(prep, S):
    U = prep["Ut"] - prep["W"] @ S
    O = prep["Qp"] @ S + prep["Oloc"]
    S_next = prep["gamma"][:, None] * S + prep["Kend"].T @ U
    return O, S_next


def run_chunked(q, k, v, g, beta, cu_seqlens, chunk, S0=None):
    """Returns (o [T,H,dv], S_final [N,H,dk,dv], boundary states {(seq, t_local): S [H,dk,dv]})."""
    T, H, dk = q.shape
    dv = v.shape[2]
    N = len(cu_seqlens) - 1
    o = np.zeros((T, H, dv))
    S_fin = np.zeros((N, H, dk, dv))
    bounds = {}
    for n in range(N):
        a, e = int(cu_seqlens[n]), int(cu_seqlens[n + 1])
        for h in range(H):
            S = np.zeros((dk, dv)) if S0 is None else np.array(S0[n, h], dtype=np.float64)
            for c0 in range(a, e, chunk):
                c1 = min(c0 + chunk, e)
                prep = chunk_prepare(q[c0:c1, h], k[c0:c1, h], v[c0:c1, h], g[c0:c1, h], beta[c0:c1, h])
                O, S = chunk_apply(prep, S)
                o[c0:c1, h] = O
                bounds.setdefault((n, c1 - a), np.zeros((H, dk, dv)))[h] = S
            S_fin[n, h] = S
    return o, S_fin, bounds
