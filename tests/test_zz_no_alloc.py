"""kda_prefill_chunked_noalloc against kda_prefill_chunked, through the C ABI (GPU).

The no-allocation entry point exists for callers that cannot hand the library
device scratch (stream capture, fixed memory pools, plugins that only receive
their inputs and outputs).  Both entry points run the same deterministic
kernels, so the no-allocation call must reproduce the regular call's outputs
and final states bit for bit -- any difference would mean that stale scratch
from an earlier call was read.  The first call of each pair is the larger one,
so leftover records cannot match the second call's by chance.  It must also
refuse sizes whose scratch exceeds the array, and report invalid cu_seqlens
through kda_prefill_noalloc_check.  This file is collected last so that a
failure here cannot stop a run before the other tests.
"""
import ctypes

import pytest
import torch

from gated_delta_rule_27_gb300 import libkda, workloads
from tests.gpu_helpers import dev

pytestmark = pytest.mark.gpu


def _regular(inp, S0, chunk):
    q, k, v, g, beta, cu = (x.to(dev()) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta, inp.cu_seqlens))
    return libkda.prefill(q, k, v, g, beta, cu, S0=S0, chunk_size=chunk)


def _noalloc_raw(inp, S0, chunk):
    """Direct ctypes call of the C entry point (no Python-side allocation of scratch)."""
    fn = libkda.load().kda_prefill_chunked_noalloc
    q, k, v, g, beta, cu = (x.to(dev()) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta, inp.cu_seqlens))
    T, H, d = q.shape
    N = cu.numel() - 1
    o = torch.full((T, H, d), float("nan"), dtype=v.dtype, device=dev())
    S = torch.full((N, H, d, d), float("nan"), device=dev())
    dt = libkda.KDA_BF16 if q.dtype == torch.bfloat16 else libkda.KDA_F32
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    rc = fn(ptr(q), ptr(k), ptr(v), ptr(g), ptr(beta), ptr(cu), N, T, H, d, d, dt, chunk, ptr(S0), ptr(o), ptr(S),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return rc, o, S


@pytest.mark.parametrize("dtype,d,chunk", [(torch.bfloat16, 128, 64), (torch.float32, 64, 32)], ids=["bf16", "f32"])
def test_noalloc_matches_regular_on_two_calls_in_a_row(dtype, d, chunk):
    first = workloads.prefill_inputs([300, 77], H=4, d=d, dtype=dtype, seed=71, s0_std=0.1)
    second = workloads.prefill_inputs([45, 0, 190], H=4, d=d, dtype=dtype, seed=72, s0_std=0.1)
    assert first.total_tokens > second.total_tokens
    for inp in (first, second):
        S0 = inp.S0.to(dev())
        o_ref, S_ref = _regular(inp, S0, chunk)
        rc, o, S = _noalloc_raw(inp, S0, chunk)
        assert rc == libkda.KDA_OK, libkda.status_string(rc)
        assert libkda.kda_prefill_noalloc_check() == libkda.KDA_OK
        assert torch.equal(o, o_ref), (o.float() - o_ref.float()).abs().max().item()
        assert torch.equal(S, S_ref), (S - S_ref).abs().max().item()


def test_noalloc_reports_invalid_cu_seqlens_and_writes_nothing():
    inp = workloads.prefill_inputs([40, 30], H=2, d=128, dtype=torch.bfloat16, seed=73)
    q, k, v, g, beta = (x.to(dev()) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta))
    bad = torch.tensor([0, 50, 40], dtype=torch.int32, device=dev())
    o = torch.full((70, 2, 128), 7.0, dtype=torch.bfloat16, device=dev())
    S = torch.full((2, 2, 128, 128), 7.0, device=dev())
    libkda.kda_prefill_chunked_noalloc(q, k, v, g, beta, bad, o, S_final=S)
    assert libkda.kda_prefill_noalloc_check() == libkda.KDA_ERR_INVALID_ARG
    assert bool((o == 7.0).all()) and bool((S == 7.0).all())
    libkda.kda_prefill_chunked_noalloc(q, k, v, g, beta, inp.cu_seqlens.to(dev()), o, S_final=S)
    assert libkda.kda_prefill_noalloc_check() == libkda.KDA_OK


def test_noalloc_refuses_sizes_beyond_its_scratch():
    T, N, H, d = 65536, 1, 32, 128
    need = libkda.kda_prefill_workspace_size(T, N, H, d, d, libkda.KDA_BF16, 64)
    assert need > libkda.NOALLOC_SCRATCH_BYTES
    x = torch.zeros((T, H, d), dtype=torch.bfloat16, device=dev())
    g = torch.zeros((T, H, d), device=dev())
    beta = torch.zeros((T, H), device=dev())
    cu = torch.tensor([0, T], dtype=torch.int32, device=dev())
    o = torch.full((T, H, d), 3.0, dtype=torch.bfloat16, device=dev())
    with pytest.raises(libkda.KdaError) as err:
        libkda.kda_prefill_chunked_noalloc(x, x, x, g, beta, cu, o)
    assert err.value.status == libkda.KDA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((o == 3.0).all())
