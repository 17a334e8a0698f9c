"""Failure detection on the GPU, without a GPU fault.

Every wait of one CTA on another in libkda's kernels is bounded in time; when
a bound runs out, the waiting kernel records KDA_ERR_TIMEOUT in the call's
status word, stops touching the outputs it cannot finish, and returns, so
that the context stays usable and kda_prefill_check can report the failure.
Here the test hook kda_testing_set_fault stops the state chains of the chain
and pipe plans from publishing their state images, with a short (20 ms)
bound on the output units' waits for them: nothing hangs, nothing faults,
the wait simply runs out.
"""
from __future__ import annotations

import time

import pytest
import torch

from gated_delta_rule_27_gb300 import libkda, workloads
from tests.gpu_helpers import TOL, dev, oracle_prefill, rel, to_device

pytestmark = pytest.mark.gpu


def _call(q, k, v, g, beta, cu, ws, S0):
    T, H, d = q.shape
    N = cu.numel() - 1
    o = torch.full((T, H, d), float("nan"), dtype=v.dtype, device=dev())
    S = torch.full((N, H, d, d), float("nan"), device=dev())
    libkda.kda_prefill_chunked(q, k, v, g, beta, cu, o, S0=S0, S_final=S, workspace=ws, chunk_size=64)
    return o, S


@pytest.mark.parametrize("plan", ["chain", "pipe"])
def test_wait_that_runs_out_is_reported_and_the_next_call_is_correct(plan):
    inp = workloads.prefill_inputs([300, 77], H=4, d=128, dtype=torch.bfloat16, seed=41, s0_std=0.1)
    q, k, v, g, beta, cu = to_device(inp)
    S0 = inp.S0.to(dev())
    T, H, d = q.shape
    ws = libkda.new_workspace(T, 2, H, d, d, libkda.KDA_BF16, 64, dev())
    libkda.testing_set_plan({"chain": libkda.PLAN_CHAIN, "pipe": libkda.PLAN_PIPE}[plan])
    libkda.testing_set_fault(libkda.FAULT_NO_PUBLISH, 20_000_000)
    try:
        t0 = time.perf_counter()
        _call(q, k, v, g, beta, cu, ws, S0)
        status = libkda.kda_prefill_check(ws)
        elapsed = time.perf_counter() - t0
    finally:
        libkda.testing_set_fault(libkda.FAULT_NONE, 0)
        libkda.testing_set_plan(libkda.PLAN_AUTO)
    assert status == libkda.KDA_ERR_TIMEOUT, libkda.status_string(status)
    assert elapsed < 10.0, elapsed  # the 20 ms bound, not a hang
    # the same context and workspace take a normal call afterwards, and its results are right
    o, S = _call(q, k, v, g, beta, cu, ws, S0)
    assert libkda.kda_prefill_check(ws) == libkda.KDA_OK
    o_ref, S_ref, _ = oracle_prefill(inp, S0=inp.S0)
    assert rel(o, o_ref) <= TOL[torch.bfloat16], rel(o, o_ref)
    assert rel(S, S_ref) <= TOL[torch.bfloat16], rel(S, S_ref)


def test_testing_hooks_reject_unknown_values():
    with pytest.raises(libkda.KdaError):
        libkda.testing_set_plan(7)
    with pytest.raises(libkda.KdaError):
        libkda.testing_set_fault(9, 0)
    with pytest.raises(libkda.KdaError):
        libkda.testing_set_fault(libkda.FAULT_NONE, -1)
