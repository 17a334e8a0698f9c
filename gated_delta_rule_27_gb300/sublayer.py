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


class Buffers:
    """Every intermediate of one sublayer step with R rows (tokens, or sequences in decode), allocated once so
    that repeated steps allocate nothing and keep their addresses (libkda then reuses its encoded tensor
    maps)."""

    def __init__(self, R: int, N: int, H: int, d: int, device):
        bf, f32 = torch.bfloat16, torch.float32
        HD = H * d
        self.q, self.k, self.v, self.z = (torch.empty((R, HD), dtype=bf, device=device) for _ in range(4))
        self.qc, self.kc, self.vc = (torch.empty((R, HD), dtype=bf, device=device) for _ in range(3))
        self.a = torch.empty((R, HD), dtype=bf, device=device)
        self.b = torch.empty((R, H), dtype=bf, device=device)
        self.g = torch.empty((R, HD), dtype=f32, device=device)
        self.beta = torch.empty((R, H), dtype=f32, device=device)
        self.o = torch.empty((R, H, d), dtype=bf, device=device)
        self.S = torch.empty((N, H, d, d), dtype=f32, device=device)
        self.conv_state = [torch.empty((N, CONV_W - 1, HD), dtype=f32, device=device) for _ in range(3)]


def _project(x, w: Weights, bufs: Buffers):
    torch.matmul(x, w.W_q, out=bufs.q)
    torch.matmul(x, w.W_k, out=bufs.k)
    torch.matmul(x, w.W_v, out=bufs.v)
    torch.matmul(x, w.W_a, out=bufs.a)
    torch.matmul(x, w.W_b, out=bufs.b)
    torch.matmul(x, w.W_z, out=bufs.z)
    torch.nn.functional.softplus(bufs.a.float(), out=bufs.g)
    bufs.g.neg_()
    torch.sigmoid(bufs.b.float(), out=bufs.beta)


def prefill_forward(x, cu_seqlens, w: Weights, H: int, d: int, events=None, qk_eps=1e-6, out_eps=1e-6,
                    bufs: Buffers = None):
    """x [T, D] bf16 -> (y [T, D] bf16, S [N, H, d, d], convolution states of q, k, v [N, CONV_W - 1, H d])
    for packed documents (zero initial states).  With `events` (five torch.cuda.Event), the stage boundaries
    are recorded: projections | convolution | recurrence | output.  `bufs` (Buffers for T rows) avoids every
    allocation; the results then live in it."""
    T = x.shape[0]
    N = cu_seqlens.numel() - 1
    if bufs is None:
        bufs = Buffers(T, N, H, d, x.device)
    _mark(events, 0)
    _project(x, w, bufs)
    _mark(events, 1)
    for src, cw, dst, st in ((bufs.q, w.conv_q, bufs.qc, bufs.conv_state[0]), (bufs.k, w.conv_k, bufs.kc,
                                                                               bufs.conv_state[1]),
                             (bufs.v, w.conv_v, bufs.vc, bufs.conv_state[2])):
        libkda.kda_short_conv_prefill(src, cw, cu_seqlens, dst, conv_state_out=st)
    _mark(events, 2)
    libkda.kda_prefill_chunked_ex(bufs.qc.view(T, H, d), bufs.kc.view(T, H, d), bufs.vc.view(T, H, d),
                                  bufs.g.view(T, H, d), bufs.beta, cu_seqlens, bufs.o, S_final=bufs.S,
                                  qk_l2norm=True, qk_eps=qk_eps, out_gate=bufs.z.view(T, H, d),
                                  out_weight=w.out_weight, out_eps=out_eps)
    _mark(events, 3)
    y = bufs.o.view(T, H * d) @ w.W_o
    _mark(events, 4)
    return y, bufs.S, bufs.conv_state


def decode_forward(x, S, conv_state, w: Weights, H: int, d: int, events=None, qk_eps=1e-6, out_eps=1e-6,
                   bufs: Buffers = None):
    """One token per sequence: x [N, D] bf16, S [N, H, d, d] and conv_state (q, k, v states, each
    [N, CONV_W - 1, H d]) updated in place; returns y [N, D].  `bufs` (Buffers for N rows) avoids every
    allocation."""
    N = x.shape[0]
    if bufs is None:
        bufs = Buffers(N, N, H, d, x.device)
    _mark(events, 0)
    _project(x, w, bufs)
    _mark(events, 1)
    for src, cw, st, dst in ((bufs.q, w.conv_q, conv_state[0], bufs.qc), (bufs.k, w.conv_k, conv_state[1], bufs.kc),
                             (bufs.v, w.conv_v, conv_state[2], bufs.vc)):
        libkda.kda_short_conv_decode(src, cw, st, dst)
    _mark(events, 2)
    libkda.kda_decode_step_ex(bufs.qc.view(N, H, d), bufs.kc.view(N, H, d), bufs.vc.view(N, H, d),
                              bufs.g.view(N, H, d), bufs.beta, S, bufs.o, qk_l2norm=True, qk_eps=qk_eps,
                              out_gate=bufs.z.view(N, H, d), out_weight=w.out_weight, out_eps=out_eps)
    _mark(events, 3)
    y = bufs.o.view(N, H * d) @ w.W_o
    _mark(events, 4)
    return y
