"""The fused prologue (q / k L2 normalisation) and epilogue (gated output RMS normalisation) against fp64
references, on the GPU through the C ABI.

Lecture 04, section 3 puts a Q/K normalisation before the recurrence and a gated normalisation on its
output.  The kernels read raw (unnormalised) bf16 or fp32 q and k and a gate input z, and must match the fp64
chain  l2norm -> oracle recurrence -> gated_rmsnorm  (oracle/sublayer.py) within the tolerances of the
parity contract (max|x - ref| / max|ref| <= 2e-2 bf16, <= 1e-4 fp32), on outputs and final states.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gated_delta_rule_27_gb300 import libkda, workloads
from oracle import oracle, sublayer
from tests.gpu_helpers import TOL, dev, f64, rel

pytestmark = pytest.mark.gpu

EPS_QK, EPS_OUT = 1e-6, 1e-6


def _raw_inputs(lengths, H, d, dtype, seed):
    """Prefill inputs with q, k left unnormalised (N(0, 1)), a gate input z and a weight w."""
    inp = workloads.prefill_inputs(lengths, H=H, d=d, dtype=dtype, seed=seed, s0_std=0.1)
    gen = torch.Generator().manual_seed(seed + 1)
    T = inp.total_tokens
    q = torch.randn((T, H, d), generator=gen).to(dtype)
    k = (2.0 * torch.randn((T, H, d), generator=gen)).to(dtype)
    z = torch.randn((T, H, d), generator=gen).to(dtype)
    w = 1.0 + 0.1 * torch.randn(d, generator=gen)
    return inp, q, k, z, w


def _reference(inp, q, k, z, w):
    qn, kn = sublayer.l2norm(f64(q), EPS_QK), sublayer.l2norm(f64(k), EPS_QK)
    o, S, _ = oracle.run(qn, kn, f64(inp.v), f64(inp.g), f64(inp.beta), inp.cu_seqlens.numpy(),
                         S0=f64(inp.S0))
    return sublayer.gated_rmsnorm(o, f64(z), f64(w), EPS_OUT), S


@pytest.mark.parametrize("dtype,d,chunk,plan,weight", [
    (torch.bfloat16, 128, 64, "three", True), (torch.bfloat16, 128, 64, "chain", True),
    (torch.bfloat16, 128, 64, "pipe", True), (torch.bfloat16, 128, 64, "chain", False),
    (torch.float32, 64, 32, "auto", True), (torch.bfloat16, 16, 16, "auto", True)],
    ids=["tc-three", "tc-chain", "tc-pipe", "tc-chain-no-weight", "simt-f32", "simt-bf16-d16"])
def test_prefill_with_fused_norms(dtype, d, chunk, plan, weight):
    inp, q, k, z, w = _raw_inputs([150, 77, 300], H=2, d=d, dtype=dtype, seed=131)
    if not weight:
        w = torch.ones(d)  # the reference's weight when out_weight is null
    o_ref, S_ref = _reference(inp, q, k, z, w)
    x = [t.to(dev()) for t in (q, k, inp.v, inp.g, inp.beta, inp.cu_seqlens)]
    T, H = inp.total_tokens, 2
    o = torch.empty((T, H, d), dtype=dtype, device=dev())
    S = torch.empty((3, H, d, d), device=dev())
    libkda.testing_set_plan({"three": libkda.PLAN_THREE, "chain": libkda.PLAN_CHAIN, "pipe": libkda.PLAN_PIPE,
                             "auto": libkda.PLAN_AUTO}[plan])
    try:
        libkda.kda_prefill_chunked_ex(*x, o, S0=inp.S0.to(dev()), S_final=S, chunk_size=chunk, qk_l2norm=True,
                                      qk_eps=EPS_QK, out_gate=z.to(dev()), out_weight=w.to(dev()) if weight else None,
                                      out_eps=EPS_OUT)
        torch.cuda.synchronize()
    finally:
        libkda.testing_set_plan(libkda.PLAN_AUTO)
    assert rel(o, o_ref, "o fused") <= TOL[dtype], rel(o, o_ref)
    assert rel(S, S_ref, "S fused") <= TOL[dtype], rel(S, S_ref)


def test_fused_options_are_checked():
    inp, q, k, z, w = _raw_inputs([64], H=1, d=128, dtype=torch.bfloat16, seed=133)
    x = [t.to(dev()) for t in (q, k, inp.v, inp.g, inp.beta, inp.cu_seqlens)]
    o = torch.empty((64, 1, 128), dtype=torch.bfloat16, device=dev())
    w_off = torch.empty(129, device=dev())[1:]  # 4 bytes past a 16-byte boundary
    with pytest.raises(libkda.KdaError) as err:
        libkda.kda_prefill_chunked_ex(*x, o, out_gate=z.to(dev()), out_weight=w_off, out_eps=EPS_OUT)
    assert err.value.status == libkda.KDA_ERR_INVALID_ARG
    with pytest.raises(libkda.KdaError):
        libkda.kda_prefill_chunked_ex(*x, o, out_gate=z.to(dev()), out_eps=0.0)  # out_eps must be positive
    with pytest.raises(libkda.KdaError):
        libkda.kda_prefill_chunked_ex(*x, o, out_gate=o, out_eps=EPS_OUT)  # the gate may not alias o


def test_prefill_ex_without_options_is_the_plain_call():
    inp = workloads.prefill_inputs([300, 77], H=4, d=128, dtype=torch.bfloat16, seed=132, s0_std=0.1)
    x = [t.to(dev()) for t in (inp.q, inp.k, inp.v, inp.g, inp.beta, inp.cu_seqlens)]
    o1, S1 = libkda.prefill(*x, S0=inp.S0.to(dev()))
    o2 = torch.empty_like(o1)
    S2 = torch.empty_like(S1)
    libkda.kda_prefill_chunked_ex(*x, o2, S0=inp.S0.to(dev()), S_final=S2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(S1, S2)


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 16), (torch.float32, 64)],
                         ids=["bf16-128", "f32-16", "f32-64"])
def test_decode_with_fused_norms(dtype, d):
    N, H, steps = 5, 3, 6
    gen = torch.Generator().manual_seed(140 + d)
    dec = workloads.decode_inputs(steps, N, H, d, dtype, seed=141 + d)
    q = torch.randn((steps, N, H, d), generator=gen).to(dtype)
    k = (3.0 * torch.randn((steps, N, H, d), generator=gen)).to(dtype)
    z = torch.randn((steps, N, H, d), generator=gen).to(dtype)
    w = 1.0 + 0.1 * torch.randn(d, generator=gen)
    S = dec.S0.to(dev())
    outs = []
    for t in range(steps):
        o = torch.empty((N, H, d), dtype=dtype, device=dev())
        libkda.kda_decode_step_ex(q[t].to(dev()), k[t].to(dev()), dec.v[t].to(dev()), dec.g[t].to(dev()),
                                  dec.beta[t].to(dev()), S, o, qk_l2norm=True, qk_eps=EPS_QK, out_gate=z[t].to(dev()),
                                  out_weight=w.to(dev()), out_eps=EPS_OUT)
        outs.append(o)
    torch.cuda.synchronize()
    # the oracle over each (sequence, head) chain as one document of `steps` tokens
    tr = lambda x: f64(x).transpose(1, 0, *range(2, x.dim())).reshape(N * steps, H, *x.shape[3:])
    qn, kn = sublayer.l2norm(tr(q), EPS_QK), sublayer.l2norm(tr(k), EPS_QK)
    o_ref, S_ref, _ = oracle.run(qn, kn, tr(dec.v), tr(dec.g), tr(dec.beta), np.arange(N + 1) * steps,
                                 S0=f64(dec.S0))
    o_ref = sublayer.gated_rmsnorm(o_ref, tr(z), f64(w), EPS_OUT)
    o_gpu = torch.stack(outs).transpose(0, 1).reshape(N * steps, H, d)
    assert rel(o_gpu, o_ref, "o fused decode") <= TOL[dtype], rel(o_gpu, o_ref)
    assert rel(S, S_ref, "S fused decode") <= TOL[dtype], rel(S, S_ref)
