"""The short causal convolution (prefill over packed documents with carried states, and the rolling decode
step) against the fp64 definition in oracle/sublayer.py, on the GPU through the C ABI.

Tolerance as in the parity contract (max|x - ref| / max|ref|: 1e-4 for fp32, 2e-2 for bf16 outputs); the
carried states are copies of inputs and must match exactly.  The state-carry invariant (Lecture 11, section 3:
one pass, several passes with the state carried, and a prefill continued by decode steps must agree) is
checked on the GPU results themselves.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gated_delta_rule_27_gb300 import libkda, workloads
from oracle import sublayer
from tests.gpu_helpers import TOL, dev, f64, rel

pytestmark = pytest.mark.gpu


def _setup(lengths, C, W, dtype, seed):
    gen = torch.Generator().manual_seed(seed)
    T = sum(lengths)
    x = torch.randn((T, C), generator=gen).to(dtype)
    w = 0.5 * torch.randn((C, W), generator=gen)
    st = torch.randn((len(lengths), max(W - 1, 0), C), generator=gen).to(dtype).float()  # exact in in_dtype
    return x, w, st, workloads.cu_from_lengths(lengths)


@pytest.mark.parametrize("C", [2 * 128 + 8, 2 * 128 + 6], ids=["C264", "C262"])
@pytest.mark.parametrize("dtype,W", [(torch.bfloat16, 4), (torch.float32, 4), (torch.float32, 1), (torch.bfloat16, 8)],
                         ids=["bf16-W4", "f32-W4", "f32-W1", "bf16-W8"])
def test_prefill_against_the_definition(dtype, W, C):
    """C = 264 takes the four-channel kernel, C = 262 (not a multiple of 4) the one-channel kernel; neither is a
    multiple of the block width."""
    lengths = [150, 0, 2, 64, 1, 300, 65]  # empty and shorter-than-window documents, tile-straddling ones
    x, w, st, cu = _setup(lengths, C, W, dtype, seed=11 + W)
    y = torch.empty_like(x, device=dev())
    st_out = torch.full((len(lengths), W - 1, C), float("nan"), device=dev())
    libkda.kda_short_conv_prefill(x.to(dev()), w.to(dev()), cu.to(dev()), y, conv_state=st.to(dev()),
                                  conv_state_out=st_out if W > 1 else None)
    torch.cuda.synchronize()
    y_ref, st_ref = sublayer.short_conv(f64(x), f64(w), cu.numpy(), state=f64(st))
    assert rel(y, y_ref, "y") <= TOL[dtype], rel(y, y_ref)
    if W > 1:
        assert np.array_equal(f64(st_out), st_ref)


def test_state_carry_and_decode_continuation():
    """One pass over a document == two passes with the state carried == a prefill continued by decode steps."""
    C, W, T, split, tail = 512, 4, 200, 77, 9
    x, w, _, _ = _setup([T], C, W, torch.bfloat16, seed=21)
    xd, wd = x.to(dev()), w.to(dev())
    cu = lambda n: workloads.cu_from_lengths([n], device=dev())
    y_all = torch.empty_like(xd)
    s_all = torch.empty((1, W - 1, C), device=dev())
    libkda.kda_short_conv_prefill(xd, wd, cu(T), y_all, conv_state_out=s_all)
    y1, y2 = torch.empty_like(xd[:split]), torch.empty_like(xd[split:])
    s1, s2 = torch.empty_like(s_all), torch.empty_like(s_all)
    libkda.kda_short_conv_prefill(xd[:split].contiguous(), wd, cu(split), y1, conv_state_out=s1)
    libkda.kda_short_conv_prefill(xd[split:].contiguous(), wd, cu(T - split), y2, conv_state=s1, conv_state_out=s2)
    y3 = torch.empty_like(xd[:T - tail])
    s3 = torch.empty_like(s_all)
    libkda.kda_short_conv_prefill(xd[:T - tail].contiguous(), wd, cu(T - tail), y3, conv_state_out=s3)
    ys = []
    for t in range(T - tail, T):
        yt = torch.empty_like(xd[t:t + 1])
        libkda.kda_short_conv_decode(xd[t:t + 1].contiguous(), wd, s3, yt)
        ys.append(yt)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([y1, y2]), y_all) and torch.equal(s2, s_all)
    assert torch.equal(s3, s_all)  # the rolled state is the last W - 1 inputs
    assert torch.equal(torch.cat([y3] + ys), y_all)  # the same fp32 sums in the same order
    y_ref, _ = sublayer.short_conv(f64(x), f64(w), [0, T])
    assert rel(y_all, y_ref, "y one pass") <= TOL[torch.bfloat16]


def _offset_copy(x):
    """x's values in a buffer that starts one element past a 4-element boundary (the one-channel kernels)."""
    buf = torch.empty(x.numel() + 1, dtype=x.dtype, device=dev())
    v = buf[1:].view(x.shape)
    v.copy_(x)
    return v


@pytest.mark.parametrize("dtype,W", [(torch.bfloat16, 4), (torch.float32, 3), (torch.bfloat16, 8), (torch.float32, 1),
                                     (torch.bfloat16, 2)])
def test_four_channel_and_one_channel_kernels_agree_bitwise(dtype, W):
    """The same inputs through the four-channel kernels (aligned) and the one-channel kernels (x and y one element
    off the 4-element alignment): identical outputs and states, prefill and decode."""
    lengths = [150, 0, 2, 64, 1, 300, 65, 17]
    C = 264
    x, w, st, cu = _setup(lengths, C, W, dtype, seed=41 + W)
    xd, wd, cud, std = x.to(dev()), w.to(dev()), cu.to(dev()), st.to(dev())
    ys = []
    states = []
    for xin in (xd, _offset_copy(xd)):
        y = _offset_copy(torch.zeros_like(xd)) if xin.data_ptr() % 8 else torch.empty_like(xd)
        so = torch.full((len(lengths), W - 1, C), float("nan"), device=dev()) if W > 1 else None
        libkda.kda_short_conv_prefill(xin, wd, cud, y, conv_state=std, conv_state_out=so)
        ys.append(y.clone())
        states.append(so)
    assert torch.equal(ys[0], ys[1])
    if W > 1:
        assert torch.equal(states[0], states[1])
    N = len(lengths)
    xt = x[:N].to(dev()).contiguous()  # one token per sequence
    outs = []
    for xin in (xt, _offset_copy(xt)):
        s = std.clone()
        y = _offset_copy(torch.zeros_like(xt)) if xin.data_ptr() % 8 else torch.empty_like(xt)
        libkda.kda_short_conv_decode(xin, wd, s if W > 1 else None, y)
        outs.append((y.clone(), s))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_conv_rejects_bad_arguments():
    x = torch.zeros((4, 8), device=dev())
    w = torch.zeros((8, 4), device=dev())
    cu = torch.tensor([0, 4], dtype=torch.int32, device=dev())
    st = torch.zeros((1, 3, 8), device=dev())
    with pytest.raises(libkda.KdaError):
        libkda.kda_short_conv_prefill(x, w, cu, x)  # y aliases x
    with pytest.raises(libkda.KdaError):
        libkda.kda_short_conv_prefill(x, w, cu, torch.empty_like(x), conv_state=st, conv_state_out=st)
    with pytest.raises(libkda.KdaError) as err:
        libkda.kda_short_conv_prefill(x, torch.zeros((8, 9), device=dev()), cu, torch.empty_like(x))
    assert err.value.status == libkda.KDA_ERR_UNSUPPORTED
