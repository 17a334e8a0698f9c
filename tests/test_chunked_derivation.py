"""The chunk (WY/UT) formulation used by the prefill kernels equals the token loop (CPU).

Lecture 04, section 4 test design: several chunk sizes, including sizes that
do not divide the sequence length; outputs, the final state and the state at
every chunk boundary are compared, at tolerance 1e-4 (here the gap is at the
fp64 rounding level).
"""
import numpy as np
import pytest

from oracle import oracle
from tests.chunked_numpy import run_chunked


def _inputs(seed, lens, H, d):
    rng = np.random.default_rng(seed)
    T = sum(lens)
    q = rng.standard_normal((T, H, d)); q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((T, H, d)); k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, d))
    g = -np.exp(rng.normal(-1.0, 0.5, (T, H, d)))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return q, k, v, g, beta, cu


@pytest.mark.parametrize("chunk", [4, 7, 16, 64])
def test_chunked_equals_recurrent_at_every_boundary(chunk, oracle_lib):
    q, k, v, g, beta, cu = _inputs(1, [50, 23, 1], 2, 8)
    rng = np.random.default_rng(2)
    S0 = rng.standard_normal((3, 2, 8, 8)) * 0.1
    o_c, S_c, bounds = run_chunked(q, k, v, g, beta, cu, chunk, S0=S0)
    snap = sorted({t for (_, t) in bounds})
    o_r, S_r, snaps = oracle.run(q, k, v, g, beta, cu, S0=S0, snap_t=snap, lib=oracle_lib)
    assert oracle.rel_err(o_c, o_r) < 1e-10
    assert oracle.rel_err(S_c, S_r) < 1e-10
    for (n, t), S in bounds.items():
        assert oracle.rel_err(S, snaps[snap.index(t), n]) < 1e-10


def test_chunk_pair_composition(oracle_lib):
    """The composition of two chunk steps, with odd-chunk outputs from the even chunk's incoming state.

    This is the chunk-pair form that the design notes propose for halving the tensor-core state chain; it is
    checked here in fp64 against the token loop. Per chunk, with G = diag(gamma), M = -Kend^T W and
    Bc = Kend^T Ut, the step is S' = (G + M) S + Bc. Two steps compose to
        S'' = G1 G0 S + N S + B2,  N = G1 M0 + M1 G0 + M1 M0,  B2 = (G1 + M1) Bc0 + Bc1,
    and the second chunk's output needs no second state:
        O1 = Q2 S + R,  Q2 = Qp1 (G0 + M0),  R = Qp1 Bc0 + P1 Ut1.
    """
    from tests.chunked_numpy import chunk_prepare
    L, d, chunks = 8, 6, 7
    q, k, v, g, beta, cu = _inputs(3, [L * chunks - 3], 1, d)  # three pairs and a ragged unpaired chunk
    T = int(cu[-1])
    rng = np.random.default_rng(4)
    S0 = rng.standard_normal((1, 1, d, d)) * 0.1
    snap = list(range(0, T, L))[1:] + [T]
    o_r, S_r, snaps = oracle.run(q, k, v, g, beta, cu, S0=S0, snap_t=snap, lib=oracle_lib)
    preps = [chunk_prepare(q[c0:c0 + L, 0], k[c0:c0 + L, 0], v[c0:c0 + L, 0], g[c0:c0 + L, 0], beta[c0:c0 + L, 0])
             for c0 in range(0, T, L)]
    step = [(np.diag(p["gamma"]), -p["Kend"].T @ p["W"], p["Kend"].T @ p["Ut"]) for p in preps]
    S = S0[0, 0].copy()
    o = np.zeros((T, d))
    for c in range(0, len(preps), 2):
        G0, M0, B0 = step[c]
        o[c * L:(c + 1) * L] = preps[c]["Qp"] @ S + preps[c]["Oloc"]
        if c + 1 == len(preps):  # an unpaired last chunk: one ordinary step
            S = (G0 + M0) @ S + B0
            break
        G1, M1, B1 = step[c + 1]
        Q2 = preps[c + 1]["Qp"] @ (G0 + M0)
        R = preps[c + 1]["Qp"] @ B0 + preps[c + 1]["Oloc"]
        o[(c + 1) * L:(c + 2) * L] = Q2 @ S + R
        N = G1 @ M0 + M1 @ G0 + M1 @ M0
        B2 = (G1 + M1) @ B0 + B1
        S = G1 @ G0 @ S + N @ S + B2
        assert oracle.rel_err(S, snaps[snap.index(min((c + 2) * L, T)), 0, 0]) < 1e-10
    assert oracle.rel_err(o, o_r[:, 0]) < 1e-10
    assert oracle.rel_err(S, S_r[0, 0]) < 1e-10
