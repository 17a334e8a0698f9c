"""The launch plans of the tensor-core prefill agree with the oracle and with each other.

bf16 inputs with d = 128 and 64-token chunks take the tensor-core path.  It runs
as the preparation followed by a state pass whose chains also form the outputs
("three"; with the gated output normalisation fused, state pass and output
pass); as the preparation followed by one cooperative launch running the state
chains with output units alongside, which form the outputs from the chains'
state images (chain); or as one cooperative launch in which chains run beside
groups that prepare the records in chunk order and then form the outputs
(pipe: chains of 32 columns while there are at most 32 of them, else of 64);
the test hook kda_testing_set_plan forces a plan.
All perform the same arithmetic in the same order, so their results must be
bitwise identical, and they must meet the bf16 tolerance against the fp64
oracle.
"""
from __future__ import annotations

import pytest
import torch

from gated_delta_rule_27_gb300 import libkda, workloads
from tests.gpu_helpers import TOL, dev, oracle_prefill, rel, to_device

pytestmark = pytest.mark.gpu


def _run(inp, plan, S0=None, poison=0x7F):
    """One call under the given launch plan, on a workspace whose every byte is `poison` beforehand, so that
    nothing a call reads before writing it can pass for a result."""
    libkda.testing_set_plan({"auto": libkda.PLAN_AUTO, "three": libkda.PLAN_THREE, "chain": libkda.PLAN_CHAIN,
                             "pipe": libkda.PLAN_PIPE}[plan])
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
        libkda.testing_set_plan(libkda.PLAN_AUTO)
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
def test_chain_and_three_kernel_plans_agree(case):
    c = CASES[case]
    inp = workloads.prefill_inputs(c["lengths"], H=c["H"], d=128, dtype=torch.bfloat16, seed=300 + len(case),
                                   s0_std=c["s0"] or None)
    S0 = inp.S0
    o3, S3 = _run(inp, "three", S0, poison=0x00)
    oc, Sc = _run(inp, "chain", S0, poison=0x5A)
    assert torch.equal(o3, oc), (o3.float() - oc.float()).abs().max().item()
    assert torch.equal(S3, Sc), (S3 - Sc).abs().max().item()
    for plan in ("pipe",):
        op, Sp = _run(inp, plan, S0, poison=0x7F)
        assert torch.equal(o3, op), (plan, (o3.float() - op.float()).abs().max().item())
        assert torch.equal(S3, Sp), (plan, (S3 - Sp).abs().max().item())
    o_ref, S_ref, _ = oracle_prefill(inp, S0=S0)
    assert rel(oc, o_ref) <= TOL[torch.bfloat16], rel(oc, o_ref)
    assert rel(Sc, S_ref) <= TOL[torch.bfloat16], rel(Sc, S_ref)


def test_automatic_plan_on_the_prefill_workload_twice():
    """The prefill workload twice on one workspace with the automatic plan: the progress flags start from zero
    every call, so both calls match bit for bit and the three-kernel plan."""
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
    o3, S3 = _run(inp, "three")
    assert torch.equal(o3, outs[0][0]) and torch.equal(S3, outs[0][1])


@pytest.mark.parametrize("plan", ["three", "chain", "pipe"])
def test_full_prefill_workload_on_poisoned_workspaces(plan):
    """The prefill workload under each launch plan on a workspace poisoned with two different patterns: the
    kernels overlap at their boundaries (and, in the chain and pipe plans, hand data over through flags), so any
    read of a record before it is written would show up as a difference."""
    inp = workloads.workload_prefill("prefill")
    o_a, S_a = _run(inp, plan, poison=0x00)
    o_b, S_b = _run(inp, plan, poison=0x7F)
    assert torch.equal(o_a, o_b) and torch.equal(S_a, S_b)
    o_ref, S_ref, _ = oracle_prefill(inp, heads=[0, 7, 15])
    assert rel(o_a[:, [0, 7, 15]], o_ref) <= TOL[torch.bfloat16]
    assert rel(S_a[:, [0, 7, 15]], S_ref) <= TOL[torch.bfloat16]


def test_varlen_workload_on_poisoned_workspaces():
    """The packed-varlen workload (1024 chains, so three kernels) on two differently poisoned workspaces."""
    inp = workloads.workload_prefill("varlen")
    o_a, S_a = _run(inp, "auto", poison=0x00)
    o_b, S_b = _run(inp, "auto", poison=0x7F)
    assert torch.equal(o_a, o_b) and torch.equal(S_a, S_b)


def _kernel_names(inp, S0):
    """The kernels the automatic plan launches for `inp` (from the profiled entry point)."""
    q, k, v, g, beta, cu = to_device(inp)
    T, H, d = q.shape
    N = cu.numel() - 1
    ws = libkda.new_workspace(T, N, H, d, d, libkda.KDA_BF16, 64, dev())
    o = torch.empty_like(v)
    S = torch.empty((N, H, d, d), device=dev())
    events = [torch.cuda.Event(enable_timing=True) for _ in range(libkda.PREFILL_MAX_KERNELS + 1)]
    for e in events:
        e.record()
    names = libkda.kda_prefill_chunked_profiled(q, k, v, g, beta, cu, o, events, S0=S0.to(dev()), S_final=S,
                                                workspace=ws, chunk_size=64)
    torch.cuda.synchronize()
    return names


@pytest.mark.parametrize("extra_heads", [0, 1])
def test_beyond_the_pipe_plan_the_state_pass_forms_the_outputs(extra_heads):
    """One document with 25 heads (one past the pipe plan's 48 chains of 64 columns) and with as many heads as
    leave 48 SMs beside chains of 32 columns, plus one: without the gated output normalisation the automatic
    plan is the preparation and the state pass that forms the outputs itself (two kernels), which matches the
    chain plan, whose output groups form them from the state images, bit for bit, and meets the bf16 tolerance
    against the oracle."""
    sms = torch.cuda.get_device_properties(dev()).multi_processor_count
    H = 25 if extra_heads == 0 else (sms - 48) // 4 + 1
    inp = workloads.prefill_inputs([300], H=H, d=128, dtype=torch.bfloat16, seed=77 + extra_heads, s0_std=0.1)
    names = _kernel_names(inp, inp.S0)
    assert names == ["chunk_index", "prefill_prepare_tc", "prefill_state_fold_tc"], names
    o_a, S_a = _run(inp, "auto", inp.S0, poison=0x00)
    o_c, S_c = _run(inp, "chain" if extra_heads == 0 else "three", inp.S0, poison=0x7F)
    assert torch.equal(o_a, o_c) and torch.equal(S_a, S_c)
    o_ref, S_ref, _ = oracle_prefill(inp, S0=inp.S0)
    assert rel(o_a, o_ref) <= TOL[torch.bfloat16], rel(o_a, o_ref)
    assert rel(S_a, S_ref) <= TOL[torch.bfloat16], rel(S_a, S_ref)


@pytest.mark.parametrize("H", [8, 9, 24, 25])
def test_pipe_plan_at_its_thresholds(H):
    """One document with 8 heads (the most whose chains run 32 columns wide in the pipe plan) and 9 (64 wide),
    with 24 heads (48 chains of 64 columns, the most the automatic pipe plan takes) and with 25 heads (the
    two-kernel plan then): the automatic choice is the expected plan, matches the three-kernel plan bit for bit
    and meets the bf16 tolerance against the oracle."""
    extra_heads = 1 if H == 25 else 0
    inp = workloads.prefill_inputs([300], H=H, d=128, dtype=torch.bfloat16, seed=97 + H, s0_std=0.1)
    names = _kernel_names(inp, inp.S0)
    assert ("prefill_pipe_tc" in names) == (extra_heads == 0), names
    o_a, S_a = _run(inp, "auto", inp.S0, poison=0x00)
    o_3, S_3 = _run(inp, "three", inp.S0, poison=0x7F)
    assert torch.equal(o_a, o_3) and torch.equal(S_a, S_3)
    o_ref, S_ref, _ = oracle_prefill(inp, S0=inp.S0)
    assert rel(o_a, o_ref) <= TOL[torch.bfloat16], rel(o_a, o_ref)
    assert rel(S_a, S_ref) <= TOL[torch.bfloat16], rel(S_a, S_ref)


@pytest.mark.parametrize("plan", ["pipe", "three", "chain"])
@pytest.mark.parametrize("lengths,bad", [([300], [0, 301]), ([300], [1, 300]), ([200, 100], [0, 250, 240])])
def test_invalid_cu_seqlens_write_nothing_on_the_tensor_core_paths(plan, lengths, bad):
    """cu_seqlens that fail the chunk index checks (not starting at 0, not ending at the token count,
    decreasing) leave o and S_final untouched under every plan, the pipe plan's self-indexed launch for a single
    document (which makes those checks itself) included, and are reported; a valid call on the same workspace
    afterwards is right."""
    inp = workloads.prefill_inputs(lengths, H=4, d=128, dtype=torch.bfloat16, seed=71)
    q, k, v, g, beta, cu_ok = to_device(inp)
    T, H, d = q.shape
    N = len(lengths)
    ws = libkda.new_workspace(T, N, H, d, d, libkda.KDA_BF16, 64, dev())
    libkda.testing_set_plan({"three": libkda.PLAN_THREE, "chain": libkda.PLAN_CHAIN, "pipe": libkda.PLAN_PIPE}[plan])
    try:
        o = torch.full_like(v, 7.0)
        S = torch.full((N, H, d, d), 7.0, device=dev())
        cu = torch.tensor(bad, dtype=torch.int32, device=dev())
        libkda.kda_prefill_chunked(q, k, v, g, beta, cu, o, S_final=S, workspace=ws, chunk_size=64)
        assert libkda.kda_prefill_check(ws) == libkda.KDA_ERR_INVALID_ARG
        assert bool((o == 7.0).all()) and bool((S == 7.0).all())
        libkda.kda_prefill_chunked(q, k, v, g, beta, cu_ok, o, S_final=S, workspace=ws, chunk_size=64)
        assert libkda.kda_prefill_check(ws) == libkda.KDA_OK
    finally:
        libkda.testing_set_plan(libkda.PLAN_AUTO)
    o_ref, S_ref, _ = oracle_prefill(inp)
    assert rel(o, o_ref) <= TOL[torch.bfloat16]
    assert rel(S, S_ref) <= TOL[torch.bfloat16]
