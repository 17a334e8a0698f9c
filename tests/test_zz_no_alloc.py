"""kda_prefill_chunked_noalloc against kda_prefill_chunked, through the C ABI (GPU).

The no-allocation entry point exists for callers that cannot hand the library
device scratch (stream capture, fixed memory pools, plugins that only receive
their inputs and outputs).  It must give the same outputs and final states as
the regular entry point with caller-provided scratch, on consecutive calls
that share its static scratch array, and must refuse sizes whose scratch
exceeds the array.  This file is collected last so that a failure here cannot
stop a run before the other tests.
"""
import ctypes

import pytest
import torch

from gated_delta_rule_27_gb300 import libkda, workloads
from tests.gpu_helpers import TOL, dev, rel

pytestmark = pytest.mark.gpu


def _regular(inp, S0, chunk):
    q, k, v, g, beta, cu = (x.to(dev()) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta, inp.cu_seqlens))
    return libkda.prefill(q, k, v, g, beta, cu, S0=S0, chunk_size=chunk)


def _noalloc_raw(inp, S0, chunk):
    """Direct ctypes call of the C entry point (no Python-side allocation of scratch)."""
    lib = libkda.load()
    fn = lib.kda_prefill_chunked_noalloc
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    fn.restype = ctypes.c_int
    fn.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_int, i32, vp, vp, vp, vp]
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
    for inp in (first, second):
        S0 = inp.S0.to(dev())
        o_ref, S_ref = _regular(inp, S0, chunk)
        rc, o, S = _noalloc_raw(inp, S0, chunk)
        assert rc == libkda.KDA_OK, libkda.status_string(rc)
        assert rel(o, o_ref.double().cpu().numpy()) <= TOL[dtype]
        assert rel(S, S_ref.double().cpu().numpy()) <= TOL[dtype]


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
