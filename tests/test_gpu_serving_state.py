"""Serving-state paths on the GPU: decode over an active-sequence list into a state pool, and state snapshot /
restore for rollback, against the fp64 oracle.

A serving batch mixes request phases (Lecture 04, section 2): some sequences run their chunked prefill while
others generate one token at a time.  Here the states of all sequences live in one pool; prefills start from
pool slots (snapshot) and put their final states back (restore); decode steps update only the listed slots;
a speculative run of three tokens is rolled back by restoring a snapshot and replaying the accepted token
(Lecture 11, section 2, "Serving state" row; section 3: a path after rollback must equal a from-scratch run).
Every slot's token history is then replayed by the oracle from the slot's initial state, and all outputs
and final states must meet the tolerance (max|x - ref| / max|ref|: 1e-4 fp32, 2e-2 bf16).  Copies are bit
exact, and slots that no call listed keep their bits.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gated_delta_rule_27_gb300 import libkda, workloads
from oracle import oracle
from tests.gpu_helpers import TOL, dev, f64, rel

pytestmark = pytest.mark.gpu


class History:
    """Per-slot token inputs, and the GPU's output for each, in the order the slot saw them."""

    def __init__(self, num_slots):
        self.tokens = {s: [] for s in range(num_slots)}

    def add(self, slot, q, k, v, g, beta, o):
        self.tokens[slot].append((q, k, v, g, beta, o))


def _tokens(n, H, d, dtype, seed):
    q, k, v, g, beta = workloads.random_qkvgb(n, H, d, dtype, seed)
    return [x.to(dev()) for x in (q, k, v, g, beta)]


def _decode(pool, slots, hist, H, d, dtype, seed, record=True):
    q, k, v, g, beta = _tokens(len(slots), H, d, dtype, seed)
    idx = torch.tensor(slots, dtype=torch.int32, device=dev())
    o = torch.empty_like(v)
    libkda.kda_decode_step_indexed(q, k, v, g, beta, idx, pool, o)
    if record:
        for i, s in enumerate(slots):
            hist.add(s, *(x[i:i + 1] for x in (q, k, v, g, beta, o)))
    return (q, k, v, g, beta), idx


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 64)], ids=["bf16-d128", "f32-d64"])
def test_mixed_phases_and_rollback_against_the_oracle(dtype, d):
    num_slots, H = 10, 3
    gen = torch.Generator().manual_seed(5)
    pool0 = (0.1 * torch.randn((num_slots, H, d, d), generator=gen)).to(dev())
    pool = pool0.clone()
    hist = History(num_slots)

    # prefill of three new requests into slots 2, 5, 9: initial states from the pool (snapshot), final states
    # back into it (restore)
    pre_slots, lengths = [2, 5, 9], [70, 130, 33]
    inp = workloads.prefill_inputs(lengths, H=H, d=d, dtype=dtype, seed=61)
    q, k, v, g, beta, cu = (x.to(dev()) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta, inp.cu_seqlens))
    idx = torch.tensor(pre_slots, dtype=torch.int32, device=dev())
    S0 = torch.empty((3, H, d, d), device=dev())
    libkda.kda_state_snapshot(pool, idx, S0)
    o, S_fin = libkda.prefill(q, k, v, g, beta, cu, S0=S0, chunk_size=64 if d == 128 else 32)
    libkda.kda_state_restore(S_fin, idx, pool)
    cuh = inp.cu_seqlens.tolist()
    for j, s in enumerate(pre_slots):
        for t in range(cuh[j], cuh[j + 1]):
            hist.add(s, *(x[t:t + 1] for x in (q, k, v, g, beta, o)))

    # decode steps over an active list that mixes prefilled slots and a slot that only decodes (0)
    for step in range(4):
        _decode(pool, [5, 2, 9, 0], hist, H, d, dtype, seed=70 + step)

    # speculation on slots 9 and 2: snapshot, three tokens, roll back, replay the accepted first token
    spec = [9, 2]
    sidx = torch.tensor(spec, dtype=torch.int32, device=dev())
    saved = torch.empty((2, H, d, d), device=dev())
    libkda.kda_state_snapshot(pool, sidx, saved)
    first, _ = _decode(pool, spec, hist, H, d, dtype, seed=80, record=False)
    after_first = torch.empty_like(saved)
    libkda.kda_state_snapshot(pool, sidx, after_first)
    for step in range(2):
        _decode(pool, spec, hist, H, d, dtype, seed=81 + step, record=False)
    libkda.kda_state_restore(saved, sidx, pool)
    torch.cuda.synchronize()
    assert torch.equal(pool[spec], saved)  # the rollback is exact
    o_replay = torch.empty_like(first[2])
    libkda.kda_decode_step_indexed(*first, sidx, pool, o_replay)
    torch.cuda.synchronize()
    assert torch.equal(pool[spec], after_first)  # the replay gives the speculative step's bits again
    for i, s in enumerate(spec):
        hist.add(s, *(x[i:i + 1] for x in first), o_replay[i:i + 1])
    _decode(pool, [0, 9], hist, H, d, dtype, seed=90)
    torch.cuda.synchronize()

    # slots nobody listed keep their bits
    untouched = [s for s in range(num_slots) if not hist.tokens[s]]
    assert untouched == [1, 3, 4, 6, 7, 8]
    assert torch.equal(pool[untouched], pool0[untouched])

    # the oracle replays each slot's history from its initial state, every slot as one document
    used = [s for s in range(num_slots) if hist.tokens[s]]
    cat = lambda i: torch.cat([tok[i] for s in used for tok in hist.tokens[s]])
    qh, kh, vh, gh, bh, oh = (cat(i) for i in range(6))
    cu_h = np.cumsum([0] + [len(hist.tokens[s]) for s in used])
    o_ref, S_ref, _ = oracle.run(f64(qh), f64(kh), f64(vh), f64(gh), f64(bh), cu_h, S0=f64(pool0[used]))
    assert rel(oh, o_ref) <= TOL[dtype], rel(oh, o_ref)
    assert rel(pool[used], S_ref) <= TOL[dtype], rel(pool[used], S_ref)


def test_indexed_decode_equals_dense_decode_bitwise():
    """Listing every slot in order is the dense decode step: same bits."""
    N, H, d = 6, 4, 128
    dec = workloads.decode_inputs(2, N, H, d, torch.bfloat16, seed=17, device=dev())
    Sa, Sb = dec.S0.clone(), dec.S0.clone()
    idx = torch.arange(N, dtype=torch.int32, device=dev())
    for t in range(2):
        oa = libkda.decode_step(dec.q[t], dec.k[t], dec.v[t], dec.g[t], dec.beta[t], Sa)
        ob = torch.empty_like(oa)
        libkda.kda_decode_step_indexed(dec.q[t], dec.k[t], dec.v[t], dec.g[t], dec.beta[t], idx, Sb, ob)
        torch.cuda.synchronize()
        assert torch.equal(oa, ob) and torch.equal(Sa, Sb)


def test_slots_out_of_range_are_skipped_and_reported():
    num_slots, H, d = 4, 2, 64
    pool = torch.randn((num_slots, H, d, d), device=dev())
    before = pool.clone()
    q, k, v, g, beta = _tokens(3, H, d, torch.float32, seed=3)
    idx = torch.tensor([1, 4, -1], dtype=torch.int32, device=dev())
    o = torch.full_like(v, 5.0)
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    libkda.kda_decode_step_indexed(q, k, v, g, beta, idx, pool, o, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == libkda.KDA_ERR_INVALID_ARG
    assert bool((o[1:] == 5.0).all()) and not bool((o[0] == 5.0).all())
    assert torch.equal(pool[[0, 2, 3]], before[[0, 2, 3]]) and not torch.equal(pool[1], before[1])
    saved = torch.full((2, H, d, d), 9.0, device=dev())
    status.zero_()
    libkda.kda_state_snapshot(pool, torch.tensor([2, 7], dtype=torch.int32, device=dev()), saved, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == libkda.KDA_ERR_INVALID_ARG
    assert torch.equal(saved[0], pool[2]) and bool((saved[1] == 9.0).all())
