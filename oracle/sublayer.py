"""fp64 references of the sublayer steps on either side of the recurrence.

TEST INFRASTRUCTURE ONLY: tests, the smoke check and the benchmark's CPU legs
may use this module; the library path never does, and nothing here is shared
with the CUDA code.

Lecture 04, section 3 ("The sublayer is bigger than the recurrence") names the
stages around the recurrence -- a short causal convolution on Q, K and/or V, a
Q/K normalisation before it and a gated normalisation on its output -- but
prints no formula for any of them.  These are the plainest readings, written
out as their definitions:

  l2norm(x, eps)               x / sqrt(sum_c x_c^2 + eps) over the last axis
  gated_rmsnorm(o, z, w, eps)  o / sqrt(mean_c o_c^2 + eps) * w_c * sigmoid(z_c)
  short_conv(x, w, cu, state)  y_t = sum_{j < W} w[c, j] x_{t-j} per channel c,
                               causal within each document; positions before a
                               document's first token read that document's
                               carried convolution state (its previous W - 1
                               inputs, oldest first), zeros when none is given
"""
from __future__ import annotations

import numpy as np


def l2norm(x, eps: float):
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def sigmoid(z):
    z = np.asarray(z, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-z))


def gated_rmsnorm(o, z, w, eps: float):
    o = np.asarray(o, dtype=np.float64)
    w = np.ones(o.shape[-1]) if w is None else np.asarray(w, dtype=np.float64)
    rms = np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    return o / rms * w * sigmoid(z)


def short_conv(x, w, cu_seqlens, state=None):
    """Causal depthwise convolution per document.

    x [T, C], w [C, W], cu_seqlens [N + 1], state [N, W - 1, C] or None.
    Returns (y [T, C], new_state [N, W - 1, C]): the new state of a document
    is its last W - 1 inputs (older carried entries when it has fewer tokens).
    """
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    C, W = w.shape
    N = len(cu_seqlens) - 1
    y = np.zeros_like(x)
    new_state = np.zeros((N, W - 1, C))
    for n in range(N):
        a, b = int(cu_seqlens[n]), int(cu_seqlens[n + 1])
        past = np.zeros((W - 1, C)) if state is None else np.asarray(state[n], dtype=np.float64)
        seq = np.concatenate([past, x[a:b]], axis=0)  # seq[W - 1 + i] is token a + i
        for i in range(b - a):
            for j in range(W):
                y[a + i] += w[:, j] * seq[W - 1 + i - j]
        new_state[n] = seq[len(seq) - (W - 1):] if W > 1 else new_state[n]
    return y, new_state
