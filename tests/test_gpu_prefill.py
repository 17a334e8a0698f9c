"""Parity of kda_prefill_chunked (through the C ABI) with the fp64 oracle, on the GPU."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gated_delta_rule_27_gb300 import libkda, workloads
from tests.gpu_helpers import TOL, dev, f64, oracle_prefill, rel, to_device

pytestmark = pytest.mark.gpu


def _run(inp, chunk, S0=None, want_state=True):
    q, k, v, g, beta, cu = to_device(inp)
    s0 = None if S0 is None else S0.to(dev())
    o, S = libkda.prefill(q, k, v, g, beta, cu, S0=s0, chunk_size=chunk, want_state=want_state)
    torch.cuda.synchronize()
    return o, S


def _prefix(inp, t):
    """The first t tokens of a single-document input."""
    return workloads.PrefillInputs(inp.q[:t], inp.k[:t], inp.v[:t], inp.g[:t], inp.beta[:t],
                                   workloads.cu_from_lengths([t]), None)


def test_tiny_workload_every_boundary():
    """Tiny workload (fp32, d = 16, chunk 16): outputs, final state and the state at every chunk boundary."""
    w = workloads.WORKLOADS["tiny"]
    inp = workloads.workload_prefill("tiny")
    o_ref, S_ref, snaps = oracle_prefill(inp, snap_t=list(range(16, 65, 16)))
    for chunk in (16, 32, 64):
        o, S = _run(inp, chunk)
        assert rel(o, o_ref, "o chunk %d" % chunk) <= TOL[torch.float32], chunk
        assert rel(S, S_ref, "S chunk %d" % chunk) <= TOL[torch.float32], chunk
    for j, t in enumerate(range(16, 65, 16)):
        _, S = _run(_prefix(inp, t), w["chunk"])
        assert rel(S, snaps[j], "S at %d" % t) <= TOL[torch.float32], t


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 64, 128])
def test_chunk_sizes_and_ragged_tails(d, dtype):
    """Chunk sizes 16/32/64 on a length none of them divides, with an initial state; boundary states too."""
    T = 150
    inp = workloads.prefill_inputs([T], H=2, d=d, dtype=dtype, seed=100 + d, s0_std=0.1)
    snap = [16, 32, 48, 64, 96, 128, 149]
    o_ref, S_ref, snaps = oracle_prefill(inp, S0=inp.S0, snap_t=snap)
    for chunk in (16, 32, 64):
        o, S = _run(inp, chunk, S0=inp.S0)
        assert rel(o, o_ref) <= TOL[dtype], (chunk, rel(o, o_ref))
        assert rel(S, S_ref) <= TOL[dtype], (chunk, rel(S, S_ref))
        for j, t in enumerate(snap):
            if t % chunk and t != 149:
                continue
            p = _prefix(inp, t)
            _, St = _run(p, chunk, S0=inp.S0)
            assert rel(St, snaps[j]) <= TOL[dtype], (chunk, t)


def test_prefill_workload_full():
    """The prefill workload at full size (H = 16, T = 4096, d = 128, bf16, chunk 64), every output."""
    inp = workloads.workload_prefill("prefill")
    bounds = [64, 128, 1024, 2048, 4032]
    o_ref, S_ref, snaps = oracle_prefill(inp, snap_t=bounds)
    o, S = _run(inp, 64)
    assert rel(o, o_ref, "o") <= TOL[torch.bfloat16]
    assert rel(S, S_ref, "S") <= TOL[torch.bfloat16]
    for j, t in enumerate(bounds):
        _, St = _run(_prefix(inp, t), 64)
        assert rel(St, snaps[j], "S at %d" % t) <= TOL[torch.bfloat16], t


def test_varlen_workload_and_document_isolation():
    """Packed documents (8 docs, H = 32): oracle parity on sampled heads, and bit-exact isolation."""
    inp = workloads.workload_prefill("varlen")
    o, S = _run(inp, 64)
    heads = [0, 13, 31]
    o_ref, S_ref, _ = oracle_prefill(inp, heads=heads)
    assert rel(o[:, heads], o_ref, "o heads 0,13,31") <= TOL[torch.bfloat16]
    assert rel(S[:, heads], S_ref, "S heads 0,13,31") <= TOL[torch.bfloat16]
    cu = inp.cu_seqlens.tolist()
    for i in (0, 3, 7):
        a, b = cu[i], cu[i + 1]
        alone = workloads.PrefillInputs(inp.q[a:b], inp.k[a:b], inp.v[a:b], inp.g[a:b], inp.beta[a:b],
                                        workloads.cu_from_lengths([b - a]), None)
        oi, Si = _run(alone, 64)
        assert torch.equal(oi, o[a:b]), i
        assert torch.equal(Si[0], S[i]), i
    # re-randomising every other document leaves document 3's bits unchanged
    other = workloads.prefill_inputs([cu[-1]], H=32, d=128, dtype=torch.bfloat16, seed=999)
    mixed = workloads.PrefillInputs(other.q.clone(), other.k.clone(), other.v.clone(), other.g.clone(),
                                    other.beta.clone(), inp.cu_seqlens, None)
    a, b = cu[3], cu[4]
    for src, dst in ((inp.q, mixed.q), (inp.k, mixed.k), (inp.v, mixed.v), (inp.g, mixed.g), (inp.beta, mixed.beta)):
        dst[a:b] = src[a:b]
    om, Sm = _run(mixed, 64)
    assert torch.equal(om[a:b], o[a:b])
    assert torch.equal(Sm[3], S[3])


def test_long_workload_three_paths():
    """B = 2, H = 32, T = 65536: one pass == 32768 + 32768 continuation == 65472 prefill + 64 decode steps."""
    w = workloads.WORKLOADS["long"]
    inp = workloads.workload_prefill("long", device=dev())
    T, split, tail = w["T"], w["split"], w["decode_tail"]
    cu = inp.cu_seqlens
    q, k, v, g, beta = inp.q, inp.k, inp.v, inp.g, inp.beta

    o1, S1 = libkda.prefill(q, k, v, g, beta, cu, chunk_size=64)

    def halves(lo, hi):
        idx = torch.cat([torch.arange(lo, hi, device=dev()), torch.arange(T + lo, T + hi, device=dev())])
        return [x[idx].contiguous() for x in (q, k, v, g, beta)], idx

    (xa, ia), (xb, ib) = halves(0, split), halves(split, T)
    cu_a = workloads.cu_from_lengths([split, split], device=dev())
    cu_b = workloads.cu_from_lengths([T - split, T - split], device=dev())
    oa, Sa = libkda.prefill(*xa, cu_a, chunk_size=64)
    ob, Sb = libkda.prefill(*xb, cu_b, S0=Sa, chunk_size=64)
    o2 = torch.empty_like(o1)
    o2[ia], o2[ib] = oa, ob

    xp, ip = halves(0, T - tail)
    cu_p = workloads.cu_from_lengths([T - tail, T - tail], device=dev())
    op, Sp = libkda.prefill(*xp, cu_p, chunk_size=64)
    o3 = torch.empty_like(o1)
    o3[ip] = op
    Sd = Sp.clone()
    for j in range(tail):
        rows = torch.tensor([T - tail + j, 2 * T - tail + j], device=dev())
        od = libkda.decode_step(*(x[rows].contiguous() for x in (q, k, v, g, beta)), Sd)
        o3[rows] = od
    torch.cuda.synchronize()

    tol = TOL[torch.bfloat16]
    for name, o_x, S_x in (("continuation", o2, Sb), ("prefill+decode", o3, Sd)):
        assert rel(o_x, f64(o1), "o %s vs one pass" % name) <= tol
        assert rel(S_x, f64(S1), "S %s vs one pass" % name) <= tol
    # each path against the oracle on two sampled chains (seq 0 head 5, seq 1 head 20), one oracle call
    chains = ((0, 5), (1, 20))
    parts = [[x[seq * T:(seq + 1) * T, h:h + 1].cpu() for x in (q, k, v, g, beta)] for seq, h in chains]
    both = workloads.PrefillInputs(*(torch.cat([p[i] for p in parts]) for i in range(5)),
                                   workloads.cu_from_lengths([T, T]), None)
    o_ref, S_ref, _ = oracle_prefill(both)
    for c, (seq, h) in enumerate(chains):
        sl = slice(seq * T, (seq + 1) * T)
        for name, o_x, S_x in (("one pass", o1, S1), ("continuation", o2, Sb), ("prefill+decode", o3, Sd)):
            assert rel(o_x[sl, h:h + 1], o_ref[c * T:(c + 1) * T], "o %s vs oracle" % name) <= tol
            assert rel(S_x[seq, h], S_ref[c, 0], "S %s vs oracle" % name) <= tol


def test_empty_and_degenerate_documents():
    lens = [0, 1, 5, 0, 64, 65, 0]
    for dtype, d in ((torch.float32, 64), (torch.bfloat16, 128)):
        inp = workloads.prefill_inputs(lens, H=2, d=d, dtype=dtype, seed=5, s0_std=0.2)
        o_ref, S_ref, _ = oracle_prefill(inp, S0=inp.S0)
        o, S = _run(inp, 64, S0=inp.S0)
        assert rel(o, o_ref) <= TOL[dtype]
        assert rel(S, S_ref) <= TOL[dtype]
        assert torch.equal(S[0].cpu(), inp.S0[0]) and torch.equal(S[3].cpu(), inp.S0[3])
    # no tokens at all: S_final = S0 (zeros when S0 is absent)
    inp = workloads.prefill_inputs([0, 0], H=1, d=16, dtype=torch.float32, seed=6, s0_std=1.0)
    _, S = _run(inp, 16, S0=inp.S0)
    assert torch.equal(S.cpu(), inp.S0)
    _, S = _run(inp, 16)
    assert not S.any()
    # no documents at all
    inp = workloads.prefill_inputs([], H=1, d=16, dtype=torch.float32, seed=6)
    o, S = _run(inp, 16)
    assert o.numel() == 0 and S.numel() == 0


def test_invalid_cu_seqlens_writes_nothing():
    inp = workloads.prefill_inputs([40, 30], H=1, d=64, dtype=torch.float32, seed=8)
    q, k, v, g, beta, _ = to_device(inp)
    for bad in ([0, 50, 40], [0, 30, 69], [1, 30, 70]):
        cu = torch.tensor(bad, dtype=torch.int32, device=dev())
        o = torch.full((70, 1, 64), 7.0, device=dev())
        S = torch.full((2, 1, 64, 64), 7.0, device=dev())
        ws = libkda.new_workspace(70, 2, 1, 64, 64, libkda.KDA_F32, 64, dev())
        libkda.kda_prefill_chunked(q, k, v, g, beta, cu, o, S_final=S, workspace=ws, chunk_size=64)
        assert libkda.kda_prefill_check(ws) == libkda.KDA_ERR_INVALID_ARG
        assert bool((o == 7.0).all()) and bool((S == 7.0).all())
    cu = inp.cu_seqlens.to(dev())
    ws = libkda.new_workspace(70, 2, 1, 64, 64, libkda.KDA_F32, 64, dev())
    libkda.kda_prefill_chunked(q, k, v, g, beta, cu, torch.empty((70, 1, 64), device=dev()), workspace=ws)
    assert libkda.kda_prefill_check(ws) == libkda.KDA_OK


def test_deterministic_inplace_and_guarded():
    """Same bits twice; S_final may alias S0; nothing is written outside o and S_final."""
    inp = workloads.prefill_inputs([300, 77], H=4, d=128, dtype=torch.bfloat16, seed=9, s0_std=0.1)
    q, k, v, g, beta, cu = to_device(inp)
    S0 = inp.S0.to(dev())
    T, H, d = inp.q.shape
    guard = 4096
    o_buf = torch.full((guard * 2 + T * H * d,), float("nan"), dtype=torch.bfloat16, device=dev())
    S_buf = torch.full((guard * 2 + 2 * H * d * d,), float("nan"), device=dev())
    o = o_buf[guard:guard + T * H * d].view(T, H, d)
    S = S_buf[guard:guard + 2 * H * d * d].view(2, H, d, d)
    libkda.kda_prefill_chunked(q, k, v, g, beta, cu, o, S0=S0, S_final=S, chunk_size=64)
    o_first, S_first = o.clone(), S.clone()
    libkda.kda_prefill_chunked(q, k, v, g, beta, cu, o, S0=S0, S_final=S, chunk_size=64)
    torch.cuda.synchronize()
    assert torch.equal(o, o_first) and torch.equal(S, S_first)
    for buf in (o_buf, S_buf):
        assert bool(torch.isnan(buf[:guard]).all()) and bool(torch.isnan(buf[-guard:]).all())
    S_in = S0.clone()
    libkda.kda_prefill_chunked(q, k, v, g, beta, cu, o, S0=S_in, S_final=S_in, chunk_size=64)
    torch.cuda.synchronize()
    assert torch.equal(S_in, S_first)


@pytest.mark.parametrize("channels", ["all", "one"])
def test_extreme_gates(channels):
    """Runs of log-decay -10 (the extreme-gate values) inside a chunk, and write strengths 0 or 1.

    A chunk whose cumulative log-decay spans more than the tensor-core form's
    bounded range (here about 400 on one side of the chunk's middle token)
    must still match the oracle; so must the chunks around it.
    """
    T, H, d = 200, 2, 128
    inp = workloads.prefill_inputs([T], H=H, d=d, dtype=torch.bfloat16, seed=77, s0_std=0.1)
    sel = slice(None) if channels == "all" else slice(5, 6)
    inp.g[70:111, :, sel] = -10.0
    inp.g[140:142, :, sel] = -1e-4
    inp.beta[75:80] = 1.0
    inp.beta[80:85] = 0.0
    o_ref, S_ref, _ = oracle_prefill(inp, S0=inp.S0)
    for chunk in (64, 32):
        o, S = _run(inp, chunk, S0=inp.S0)
        assert rel(o, o_ref) <= TOL[torch.bfloat16], (chunk, rel(o, o_ref))
        assert rel(S, S_ref) <= TOL[torch.bfloat16], (chunk, rel(S, S_ref))
