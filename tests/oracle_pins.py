"""Checks that pin the fp64 oracle to facts fixed outside the oracle itself.

Each pin takes a loaded oracle library and raises AssertionError when the
oracle disagrees with: a step worked by hand from the closed form, the dense
affine-composition product (a different route to the same state), closed
forms of degenerate gates, the delta-rule write identity, and the
prefix/continuation and packing invariants.  The same pins are run against
deliberately broken copies of the oracle (tests/test_oracle_mutations.py) to
show that each plausible mistake is caught by at least one of them.
"""
from __future__ import annotations

import json
import os

import numpy as np

from oracle import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _random_chain(rng, T, dk, dv, unit_k=True, beta_range=(0.0, 1.0), g_scale=0.5):
    q = rng.standard_normal((T, 1, dk))
    k = rng.standard_normal((T, 1, dk))
    if unit_k:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, 1, dv))
    g = -g_scale * np.exp(rng.standard_normal((T, 1, dk)) * 0.5 - 1.0)
    beta = rng.uniform(beta_range[0], beta_range[1], (T, 1))
    return q, k, v, g, beta


def pin_hand_step(lib):
    """One step worked by hand (golden fixture); also separates the two operator orders."""
    with open(os.path.join(GOLDEN, "hand_step.json")) as f:
        gd = json.load(f)
    q = np.array(gd["q"])[None, None]
    k = np.array(gd["k"])[None, None]
    v = np.array(gd["v"])[None, None]
    g = np.log(np.array(gd["decay"]))[None, None]
    beta = np.array([[gd["beta"]]])
    S0 = np.array(gd["S0"])[None, None]
    o, S, _ = oracle.run(q, k, v, g, beta, [0, 1], S0=S0, lib=lib)
    assert np.allclose(S[0, 0], gd["S1"], atol=1e-14, rtol=0), S[0, 0]
    assert np.allclose(o[0, 0], gd["o1"], atol=1e-14, rtol=0), o[0, 0]
    assert np.max(np.abs(S[0, 0] - np.array(gd["S1_wrong_order"]))) > 0.1


def pin_dense_affine_composition(lib):
    """S_T = (A_T...A_1) S_0 + sum_t (A_T...A_{t+1}) B_t with dense A_t, B_t (tiny sizes only).

    Lecture 04, section 1: affine updates compose; A_t = (I - beta k k^T) D_t
    and B_t = beta k v^T are formed explicitly here, which a kernel must never do.
    """
    rng = _rng(11)
    for (T, dk, dv) in [(8, 4, 4), (16, 4, 3), (13, 3, 5)]:
        q, k, v, g, beta = _random_chain(rng, T, dk, dv, unit_k=False, beta_range=(0.0, 1.5))
        S0 = rng.standard_normal((1, 1, dk, dv))
        o, S_fin, snaps = oracle.run(q, k, v, g, beta, [0, T], S0=S0, snap_t=list(range(T + 1)), lib=lib)
        A = [np.eye(dk) - beta[t, 0] * np.outer(k[t, 0], k[t, 0]) for t in range(T)]
        A = [A[t] @ np.diag(np.exp(g[t, 0])) for t in range(T)]
        B = [beta[t, 0] * np.outer(k[t, 0], v[t, 0]) for t in range(T)]
        for t_end in range(1, T + 1):
            prod = np.eye(dk)
            acc = np.zeros((dk, dv))
            for t in range(t_end - 1, -1, -1):  # accumulate A_{t_end}...A_{t+2} B_{t+1}
                acc += prod @ B[t]
                prod = prod @ A[t]
            S_t = prod @ S0[0, 0] + acc
            assert np.allclose(snaps[t_end, 0, 0], S_t, atol=1e-12, rtol=1e-12)
            assert np.allclose(o[t_end - 1, 0], S_t.T @ q[t_end - 1, 0], atol=1e-12, rtol=1e-12)
        assert np.array_equal(S_fin[0, 0], snaps[T, 0, 0])


def pin_write_identity(lib):
    """S_t^T k_t = (1 - beta ||k||^2) (D_t S_{t-1})^T k_t + beta ||k||^2 v_t, from the closed form."""
    rng = _rng(12)
    T, dk, dv = 24, 6, 5
    q, k, v, g, beta = _random_chain(rng, T, dk, dv, unit_k=False, beta_range=(0.0, 1.0))
    S0 = rng.standard_normal((1, 1, dk, dv))
    _, _, snaps = oracle.run(q, k, v, g, beta, [0, T], S0=S0, snap_t=list(range(T + 1)), lib=lib)
    for t in range(T):
        kt, vt, bt = k[t, 0], v[t, 0], beta[t, 0]
        prev = np.exp(g[t, 0])[:, None] * snaps[t, 0, 0]
        nk = kt @ kt
        lhs = snaps[t + 1, 0, 0].T @ kt
        rhs = (1.0 - bt * nk) * (prev.T @ kt) + bt * nk * vt
        assert np.allclose(lhs, rhs, atol=1e-12, rtol=1e-12), (t, lhs, rhs)


def pin_unit_write_recalls_value(lib):
    """With beta = 1 and ||k|| = 1 the state maps k_t exactly to v_t after the write."""
    rng = _rng(13)
    T, dk, dv = 10, 8, 8
    q, k, v, g, beta = _random_chain(rng, T, dk, dv, unit_k=True)
    beta[:] = 1.0
    S0 = rng.standard_normal((1, 1, dk, dv))
    _, _, snaps = oracle.run(q, k, v, g, beta, [0, T], S0=S0, snap_t=list(range(1, T + 1)), lib=lib)
    for t in range(T):
        assert np.allclose(snaps[t, 0, 0].T @ k[t, 0], v[t, 0], atol=1e-12)


def pin_pure_decay(lib):
    """beta = 0: S_t = diag(exp(sum_{s<=t} g_s)) S_0 and o_t = S_t^T q_t."""
    rng = _rng(14)
    T, dk, dv = 12, 5, 7
    q, k, v, g, beta = _random_chain(rng, T, dk, dv)
    beta[:] = 0.0
    S0 = rng.standard_normal((1, 1, dk, dv))
    o, S, _ = oracle.run(q, k, v, g, beta, [0, T], S0=S0, lib=lib)
    cum = np.cumsum(g[:, 0], axis=0)
    for t in range(T):
        St = np.exp(cum[t])[:, None] * S0[0, 0]
        assert np.allclose(o[t, 0], St.T @ q[t, 0], atol=1e-12, rtol=1e-12)
    assert np.allclose(S[0, 0], np.exp(cum[-1])[:, None] * S0[0, 0], atol=1e-12, rtol=1e-12)


def pin_constant_state(lib):
    """g = 0 and beta = 0: the state never changes, so O = Q S_0 (one matrix product)."""
    rng = _rng(15)
    T, dk, dv = 9, 4, 6
    q, k, v, g, beta = _random_chain(rng, T, dk, dv)
    g[:] = 0.0
    beta[:] = 0.0
    S0 = rng.standard_normal((1, 1, dk, dv))
    o, S, _ = oracle.run(q, k, v, g, beta, [0, T], S0=S0, lib=lib)
    assert np.allclose(o[:, 0], q[:, 0] @ S0[0, 0], atol=1e-13)
    assert np.array_equal(S[0, 0], S0[0, 0])


def pin_first_token_from_zero(lib):
    """S_0 = 0, one token: S_1 = beta k v^T and o_1 = beta (q . k) v."""
    rng = _rng(16)
    dk, dv = 7, 3
    q, k, v, g, beta = _random_chain(rng, 1, dk, dv, unit_k=False)
    o, S, _ = oracle.run(q, k, v, g, beta, [0, 1], lib=lib)
    b = beta[0, 0]
    assert np.allclose(S[0, 0], b * np.outer(k[0, 0], v[0, 0]), atol=1e-14)
    assert np.allclose(o[0, 0], b * (q[0, 0] @ k[0, 0]) * v[0, 0], atol=1e-14)


def pin_extreme_gates(lib):
    """Log-decay -10 nearly resets the state (x 4.54e-5); -1e-4 nearly keeps it."""
    rng = _rng(17)
    dk, dv = 4, 4
    q, k, v, g, beta = _random_chain(rng, 1, dk, dv)
    beta[:] = 0.0
    S0 = rng.standard_normal((1, 1, dk, dv))
    g[:] = -10.0
    _, S, _ = oracle.run(q, k, v, g, beta, [0, 1], S0=S0, lib=lib)
    assert np.allclose(S[0, 0], np.exp(-10.0) * S0[0, 0], rtol=1e-14, atol=0)
    g[:] = -1e-4
    _, S, _ = oracle.run(q, k, v, g, beta, [0, 1], S0=S0, lib=lib)
    assert np.allclose(S[0, 0], S0[0, 0], rtol=1.01e-4, atol=0)


def pin_prefix_continuation(lib):
    """One pass == prefix then continuation from the carried state (bit for bit).

    Lecture 11, section 3: one prefill pass, several chunks and a cached
    continuation lead to the same state and outputs.
    """
    rng = _rng(18)
    T, dk, dv = 40, 6, 6
    q, k, v, g, beta = _random_chain(rng, T, dk, dv)
    S0 = rng.standard_normal((1, 1, dk, dv))
    o, S, snaps = oracle.run(q, k, v, g, beta, [0, T], S0=S0, snap_t=[17], lib=lib)
    for split in (1, 17, 39):
        o1, S1, _ = oracle.run(q[:split], k[:split], v[:split], g[:split], beta[:split], [0, split], S0=S0, lib=lib)
        o2, S2, _ = oracle.run(q[split:], k[split:], v[split:], g[split:], beta[split:], [0, T - split], S0=S1,
                               lib=lib)
        assert np.array_equal(np.concatenate([o1, o2]), o)
        assert np.array_equal(S2, S)
        if split == 17:
            assert np.array_equal(S1[0, 0], snaps[0, 0, 0])


def pin_packed_documents(lib):
    """Packed documents == each document run alone (no state crosses a boundary)."""
    rng = _rng(19)
    lens = [5, 1, 0, 13, 7]
    T, H, dk, dv = sum(lens), 2, 4, 3
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk)) * 0.5
    v = rng.standard_normal((T, H, dv))
    g = -np.abs(rng.standard_normal((T, H, dk)))
    beta = rng.uniform(0, 1, (T, H))
    S0 = rng.standard_normal((len(lens), H, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    o, S, _ = oracle.run(q, k, v, g, beta, cu, S0=S0, lib=lib)
    for i, n in enumerate(lens):
        a, b = cu[i], cu[i + 1]
        oi, Si, _ = oracle.run(q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b], [0, n], S0=S0[i:i + 1], lib=lib)
        assert np.array_equal(o[a:b], oi)
        assert np.array_equal(S[i], Si[0])


def pin_stability_bound(lib):
    """||k|| <= 1, beta in [0, 1], D <= I: ||S_t||_2 <= ||S_{t-1}||_2 + beta ||k|| ||v||."""
    rng = _rng(20)
    T, dk, dv = 30, 6, 6
    q, k, v, g, beta = _random_chain(rng, T, dk, dv, unit_k=True)
    S0 = rng.standard_normal((1, 1, dk, dv))
    _, _, snaps = oracle.run(q, k, v, g, beta, [0, T], S0=S0, snap_t=list(range(T + 1)), lib=lib)
    for t in range(T):
        lhs = np.linalg.norm(snaps[t + 1, 0, 0], 2)
        rhs = np.linalg.norm(snaps[t, 0, 0], 2) + beta[t, 0] * np.linalg.norm(k[t, 0]) * np.linalg.norm(v[t, 0])
        assert lhs <= rhs * (1 + 1e-12), (t, lhs, rhs)


def pin_affine_in_initial_state(lib):
    """The final state and outputs are affine in S_0 (the chunk's composed A, B do not depend on S_0)."""
    rng = _rng(21)
    T, dk, dv = 20, 5, 4
    q, k, v, g, beta = _random_chain(rng, T, dk, dv)
    Sa = rng.standard_normal((1, 1, dk, dv))
    Sb = rng.standard_normal((1, 1, dk, dv))
    a = 0.3
    oa, Fa, _ = oracle.run(q, k, v, g, beta, [0, T], S0=Sa, lib=lib)
    ob, Fb, _ = oracle.run(q, k, v, g, beta, [0, T], S0=Sb, lib=lib)
    om, Fm, _ = oracle.run(q, k, v, g, beta, [0, T], S0=a * Sa + (1 - a) * Sb, lib=lib)
    assert np.allclose(Fm, a * Fa + (1 - a) * Fb, atol=1e-12)
    assert np.allclose(om, a * oa + (1 - a) * ob, atol=1e-12)


def pin_multihead_layout(lib):
    """Heads are independent and indexed [T, H, d]: a head run inside H=3 equals it run alone."""
    rng = _rng(22)
    T, H, dk, dv = 11, 3, 4, 5
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk)) * 0.5
    v = rng.standard_normal((T, H, dv))
    g = -np.abs(rng.standard_normal((T, H, dk)))
    beta = rng.uniform(0, 1, (T, H))
    S0 = rng.standard_normal((1, H, dk, dv))
    o, S, _ = oracle.run(q, k, v, g, beta, [0, T], S0=S0, lib=lib)
    for h in range(H):
        oh, Sh, _ = oracle.run(q[:, h:h + 1], k[:, h:h + 1], v[:, h:h + 1], g[:, h:h + 1], beta[:, h:h + 1],
                               [0, T], S0=S0[:, h:h + 1], lib=lib)
        assert np.array_equal(o[:, h], oh[:, 0])
        assert np.array_equal(S[0, h], Sh[0, 0])


ALL_PINS = [
    pin_hand_step,
    pin_dense_affine_composition,
    pin_write_identity,
    pin_unit_write_recalls_value,
    pin_pure_decay,
    pin_constant_state,
    pin_first_token_from_zero,
    pin_extreme_gates,
    pin_prefix_continuation,
    pin_packed_documents,
    pin_stability_bound,
    pin_affine_in_initial_state,
    pin_multihead_layout,
]
