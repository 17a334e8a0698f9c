"""The two launch plans of the tensor-core prefill agree with the oracle and with each other.

bf16 inputs with d = 128 and 64-token chunks take the tensor-core path.  It runs
either as three kernels (preparation, state pass, output) or, for calls with few
(document, head, column tile) chains, as one cooperative launch that overlaps
them; KDA_TC_FUSED=0 / 1 forces one plan.  Both perform the same arithmetic in
the same order, so their results must be bitwise identical, and both must meet
the bf16 tolerance against the fp64 oracle.
"""
from __future__ import annotations

import os

import pytest
import torch

from gated_delta_rule_27_gb300 import libkda, workloads
from tests.gpu_helpers import TOL, dev, oracle_prefill, rel, to_device

pytestmark = pytest.mark.gpu


def _run(inp, plan, S0=None, poison=0x7F):
    """One call under the given launch plan, on a workspace whose every byte is `poison` beforehand, so that
    nothing a call reads before writing it can pass for a result."""
    old = os.environ.get("KDA_TC_FUSED")
    os.environ["KDA_TC_FUSED"] = plan
    try:
        q, k, v, g, beta, cu = to_device(inp)
        T, H, d = q.shape
        N = cu.numel() - 1
        ws = libkda.new_workspace(T, N, H, d, d, libkda.KDA_BF16, 64, dev())
        ws.fill_(poison)
        o = torch.empty_like(v)
        S = torch.empty((N, H, d, d), device=dev())
        libkda.kda_prefill_chunked(q, k, v, g, beta, cu, o, S0=None if S0 is None else S0.to(dev()), S_final=S,
                                   workspace=ws, chunk_size=64)
        torch.cuda.synchronize()
        assert libkda.kda_prefill_check(ws) == 0
    finally:
        if old is None:
            del os.environ["KDA_TC_FUSED"]
        else:
            os.environ["KDA_TC_FUSED"] = old
    return o, S


CASES = {
    # one document, the bench's head count, a ragged tail
    "one_doc": dict(lengths=[1000], H=16, s0=0.0),
    # three documents (one shorter than a chunk), initial states
    "three_docs": dict(lengths=[300, 40, 777], H=4, s0=0.1),
    # an empty document between two others
    "empty_doc": dict(lengths=[130, 0, 64], H=2, s0=0.1),
    # a first document of a single partial chunk
    "short_first": dict(lengths=[40, 777], H=4, s0=0.1),
    # many short documents, 64 chains
    "many_docs": dict(lengths=[1, 5, 0, 64, 65, 0, 200, 3, 100, 7, 0, 129, 64, 2, 33, 90], H=1, s0=0.2),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_fused_and_three_kernel_plans_agree(case):
    c = CASES[case]
    inp = workloads.prefill_inputs(c["lengths"], H=c["H"], d=128, dtype=torch.bfloat16, seed=300 + len(case),
                                   s0_std=c["s0"] or None)
    S0 = inp.S0
    o3, S3 = _run(inp, "0", S0, poison=0x00)
    of, Sf = _run(inp, "1", S0, poison=0x7F)
    assert torch.equal(o3, of), (o3.float() - of.float()).abs().max().item()
    assert torch.equal(S3, Sf), (S3 - Sf).abs().max().item()
    o_ref, S_ref, _ = oracle_prefill(inp, S0=S0)
    assert rel(of, o_ref) <= TOL[torch.bfloat16], rel(of, o_ref)
    assert rel(Sf, S_ref) <= TOL[torch.bfloat16], rel(Sf, S_ref)


def test_fused_plan_on_the_prefill_workload_twice():
    """The prefill workload (which picks the single launch by itself) twice on one workspace: the progress
    flags start from zero every call, so both calls match bit for bit and the three-kernel plan."""
    inp = workloads.workload_prefill("prefill")
    q, k, v, g, beta, cu = to_device(inp)
    T, H, d = q.shape
    ws = libkda.new_workspace(T, 1, H, d, d, libkda.KDA_BF16, 64, dev())
    outs = []
    for _ in range(2):
        o = torch.empty_like(v)
        S = torch.empty((1, H, d, d), device=dev())
        libkda.kda_prefill_chunked(q, k, v, g, beta, cu, o, S_final=S, workspace=ws)
        torch.cuda.synchronize()
        assert libkda.kda_prefill_check(ws) == 0
        outs.append((o, S))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    o3, S3 = _run(inp, "0")
    assert torch.equal(o3, outs[0][0]) and torch.equal(S3, outs[0][1])
