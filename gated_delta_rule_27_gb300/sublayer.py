"""The KDA sublayer around libkda's recurrence, with synthetic weights, for whole-sublayer timing.

Lecture 04, section 3 lists the executed sublayer: x -> Q/K/V projections ->
short causal convolution -> Q/K normalisation -> decay gate (D_t) -> write
gate (beta_t) -> the recurrence -> gated normalisation on the output ->
output projection, and warns that the stages around the recurrence can take
a large share of the sublayer's time.  This module runs that sequence so the
share can be measured:

  * projections: plain bf16 GEMMs (torch.matmul, i.e. cuBLAS) with random
    weights -- no trained weights are involved;
  * gate activations: small torch elementwise ops on the projection outputs
    (the pages give no formulas; read here as log-decay g = -softplus(x W_a)
    per channel and beta = sigmoid(x W_b) per head);
  * short convolution (width 4) on q, k and v, the q / k L2 normalisation,
    the recurrence and the gated output normalisation: libkda's kernels
    (kda_short_conv_*, kda_prefill_chunked_ex / kda_decode_step_ex).

Hidden size: H * d (the pages give none for the model).
"""
from __future__ import annotations

import dataclasses

import torch

from . import libkda

CONV_W = 4


@dataclasses.dataclass
class Weights:
    W_q: torch.Tensor   # [D, H d] bf16
    W_k: torch.Tensor
    W_v: torch.Tensor
    W_a: torch.Tensor   # decay gate [D, H d]
    W_b: torch.Tensor   # write gate [D, H]
    W_z: torch.Tensor   # output gate [D, H d]
    W_o: torch.Tensor   # [H d, D]
    conv_q: torch.Tensor  # [H d, CONV_W] fp32
    conv_k: torch.Tensor
    conv_v: torch.Tensor
    out_weight: torch.Tensor  # [d] fp32


def synthetic_weights(D: int, H: int, d: int, seed: int, device) -> Weights:
    gen = torch.Generator(device="cpu").manual_seed(seed)
    mat = lambda r, c: (torch.randn((r, c), generator=gen) / r ** 0.5).to(torch.bfloat16).to(device)
    conv = lambda: (0.5 * torch.randn((H * d, CONV_W), generator=gen)).to(device)
    return Weights(mat(D, H * d), mat(D, H * d), mat(D, H * d), mat(D, H * d), mat(D, H), mat(D, H * d),
                   mat(H * d, D), conv(), conv(), conv(), (1.0 + 0.1 * torch.randn(d, generator=gen)).to(device))


def _mark(events, i):
    if events is not None:
        events[i].record()


def prefill_forward(x, cu_seqlens, w: Weights, H: int, d: int, events=None, qk_eps=1e-6, out_eps=1e-6):
    """x [T, D] bf16 -> (y [T, D] bf16, S [N, H, d, d], convolution states of q, k, v [N, CONV_W - 1, H d])
    for packed documents (zero initial states).  With `events` (five torch.cuda.Event), the stage boundaries
    are recorded: projections | convolution | recurrence | output."""
    T = x.shape[0]
    N = cu_seqlens.numel() - 1
    conv_state = [torch.empty((N, CONV_W - 1, H * d), dtype=torch.float32, device=x.device) for _ in range(3)]
    _mark(events, 0)
    q, k, v = x @ w.W_q, x @ w.W_k, x @ w.W_v
    g = -torch.nn.functional.softplus((x @ w.W_a).float())
    beta = torch.sigmoid((x @ w.W_b).float())
    z = x @ w.W_z
    _mark(events, 1)
    qc, kc, vc = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    for src, cw, dst, st in ((q, w.conv_q, qc, conv_state[0]), (k, w.conv_k, kc, conv_state[1]),
                             (v, w.conv_v, vc, conv_state[2])):
        libkda.kda_short_conv_prefill(src, cw, cu_seqlens, dst, conv_state_out=st)
    _mark(events, 2)
    o = torch.empty((T, H, d), dtype=torch.bfloat16, device=x.device)
    S = torch.empty((N, H, d, d), dtype=torch.float32, device=x.device)
    libkda.kda_prefill_chunked_ex(qc.view(T, H, d), kc.view(T, H, d), vc.view(T, H, d), g.view(T, H, d).contiguous(),
                                  beta.contiguous(), cu_seqlens, o, S_final=S, qk_l2norm=True, qk_eps=qk_eps,
                                  out_gate=z.view(T, H, d), out_weight=w.out_weight, out_eps=out_eps)
    _mark(events, 3)
    y = o.view(T, H * d) @ w.W_o
    _mark(events, 4)
    return y, S, conv_state


def decode_forward(x, S, conv_state, w: Weights, H: int, d: int, events=None, qk_eps=1e-6, out_eps=1e-6):
    """One token per sequence: x [N, D] bf16, S [N, H, d, d] and conv_state (q, k, v states, each
    [N, CONV_W - 1, H d]) updated in place; returns y [N, D]."""
    N = x.shape[0]
    _mark(events, 0)
    q, k, v = x @ w.W_q, x @ w.W_k, x @ w.W_v
    g = -torch.nn.functional.softplus((x @ w.W_a).float())
    beta = torch.sigmoid((x @ w.W_b).float())
    z = x @ w.W_z
    _mark(events, 1)
    qc, kc, vc = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    for src, cw, st, dst in ((q, w.conv_q, conv_state[0], qc), (k, w.conv_k, conv_state[1], kc),
                             (v, w.conv_v, conv_state[2], vc)):
        libkda.kda_short_conv_decode(src, cw, st, dst)
    _mark(events, 2)
    o = torch.empty((N, H, d), dtype=torch.bfloat16, device=x.device)
    libkda.kda_decode_step_ex(qc.view(N, H, d), kc.view(N, H, d), vc.view(N, H, d), g.view(N, H, d).contiguous(),
                              beta.contiguous(), S, o, qk_l2norm=True, qk_eps=qk_eps, out_gate=z.view(N, H, d),
                              out_weight=w.out_weight, out_eps=out_eps)
    _mark(events, 3)
    y = o.view(N, H * d) @ w.W_o
    _mark(events, 4)
    return y
