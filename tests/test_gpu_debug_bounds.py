"""The bounds-checking build of the library (libkda_debug.so, -DKDA_DEBUG_BOUNDS), on the GPU.

Its kernels test every data-dependent index -- record addresses from the chunk table, token rows, state
slots, the shared-memory offsets derived from them -- before the access; a failed check skips the access
and records KDA_ERR_BOUNDS, with the failing source line, in the call's status word.  On valid inputs no
check may fail and the results must be the release build's bit for bit (the checks only add branches).
"""
from __future__ import annotations

import ctypes

import pytest
import torch

from gated_delta_rule_27_gb300 import libkda, workloads
from tests.gpu_helpers import dev

pytestmark = pytest.mark.gpu


def _prefill(lib, inp, chunk, plan=libkda.PLAN_AUTO):
    """kda_prefill_chunked through `lib`; returns o, S_final, the workspace's two status words."""
    q, k, v, g, beta, cu = (x.to(dev()) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta, inp.cu_seqlens))
    T, H, d = q.shape
    N = cu.numel() - 1
    dt = libkda.KDA_BF16 if q.dtype == torch.bfloat16 else libkda.KDA_F32
    n = lib.kda_prefill_workspace_size(T, N, H, d, d, dt, chunk)
    ws = torch.full((n,), 0x5A, dtype=torch.uint8, device=dev())
    o = torch.full((T, H, d), float("nan"), dtype=v.dtype, device=dev())
    S = torch.full((N, H, d, d), float("nan"), device=dev())
    S0 = None if inp.S0 is None else inp.S0.to(dev())
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    assert lib.kda_testing_set_plan(plan) == 0
    try:
        rc = lib.kda_prefill_chunked(p(q), p(k), p(v), p(g), p(beta), p(cu), N, T, H, d, d, dt, chunk, p(S0), p(o),
                                     p(S), p(ws), n, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        torch.cuda.synchronize()
    finally:
        lib.kda_testing_set_plan(libkda.PLAN_AUTO)
    assert rc == libkda.KDA_OK
    words = ws[:8].view(torch.int32).cpu().tolist()
    return o, S, words[0], words[1]


CASES = [("bf16-tc", [300, 77, 0, 64], 4, 128, torch.bfloat16, 64),
         ("f32-simt", [150, 40], 2, 64, torch.float32, 32)]


@pytest.mark.parametrize("name,lengths,H,d,dtype,chunk", CASES, ids=[c[0] for c in CASES])
def test_debug_build_passes_every_check_and_matches_the_release_build(name, lengths, H, d, dtype, chunk):
    dbg = libkda.load_debug()
    rel = libkda.load()
    inp = workloads.prefill_inputs(lengths, H=H, d=d, dtype=dtype, seed=171, s0_std=0.1)
    plans = [libkda.PLAN_THREE, libkda.PLAN_CHAIN, libkda.PLAN_PIPE] if d == 128 else \
        [libkda.PLAN_AUTO]
    for plan in plans:
        o_d, S_d, st, line = _prefill(dbg, inp, chunk, plan)
        o_r, S_r, st_r, _ = _prefill(rel, inp, chunk, plan)
        assert st == 0 and line == 0, (plan, st, line)
        assert st_r == 0
        assert torch.equal(o_d, o_r) and torch.equal(S_d, S_r), plan
