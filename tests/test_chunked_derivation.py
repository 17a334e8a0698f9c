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
