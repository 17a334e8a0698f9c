"""Parity of kda_decode_step (through the C ABI) with the fp64 oracle, on the GPU."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gated_delta_rule_27_gb300 import libkda, workloads
from oracle import oracle
from tests.gpu_helpers import TOL, dev, f64, rel

pytestmark = pytest.mark.gpu


def _oracle_steps(dec, chains, S0, snap_t=None):
    """Oracle over `steps` tokens of the listed (seq, head) chains, each chain one document."""
    steps = dec.q.shape[0]
    pick = lambda x: torch.stack([x[:, n, h] for n, h in chains], dim=1)  # [steps, C, ...]
    q, k, v, g = (pick(x).transpose(0, 1).reshape(-1, 1, x.shape[-1]) for x in (dec.q, dec.k, dec.v, dec.g))
    beta = pick(dec.beta).transpose(0, 1).reshape(-1, 1)
    s0 = torch.stack([S0[n, h] for n, h in chains])[:, None]
    cu = np.arange(len(chains) + 1) * steps
    o, S, snaps = oracle.run(f64(q), f64(k), f64(v), f64(g), f64(beta), cu, S0=f64(s0), snap_t=snap_t)
    return o.reshape(len(chains), steps, -1), S[:, 0], snaps


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 64, 128])
def test_decode_steps_small(d, dtype):
    N, H, steps = 5, 3, 20
    dec = workloads.decode_inputs(steps, N, H, d, dtype, seed=40 + d, extreme_frac=0.1)
    S = dec.S0.to(dev())
    outs = []
    for t in range(steps):
        outs.append(libkda.decode_step(dec.q[t].to(dev()), dec.k[t].to(dev()), dec.v[t].to(dev()),
                                       dec.g[t].to(dev()), dec.beta[t].to(dev()), S))
    torch.cuda.synchronize()
    chains = [(n, h) for n in range(N) for h in range(H)]
    o_ref, S_ref, _ = _oracle_steps(dec, chains, dec.S0)
    o = torch.stack(outs)  # [steps, N, H, d]
    o = torch.stack([o[:, n, h] for n, h in chains])
    assert rel(o, o_ref) <= TOL[dtype]
    assert rel(torch.stack([S[n, h] for n, h in chains]), S_ref) <= TOL[dtype]


def test_decode_workload_full():
    """256 sequences x 32 heads, 1000 steps with 5% extreme-gate steps; sampled chains against the oracle."""
    w = workloads.WORKLOADS["decode"]
    N, H, d, steps = w["N"], w["H"], w["d"], w["steps"]
    dec = workloads.decode_inputs(steps, N, H, d, w["dtype"], seed=workloads.workload_seed("decode"), device=dev())
    assert dec.extreme_steps.numel() == 50
    chains = [(0, 0), (17, 3), (100, 31), (255, 16), (128, 8), (64, 25), (200, 1), (3, 30)]
    idx_n = torch.tensor([n for n, _ in chains], device=dev())
    idx_h = torch.tensor([h for _, h in chains], device=dev())
    S = dec.S0.clone()
    S0_cpu = dec.S0.cpu()
    o_all = torch.empty((steps, len(chains), d), dtype=w["dtype"], device=dev())
    snap_steps = [50, 500, 999]
    snaps_gpu = {}
    for t in range(steps):
        o = libkda.decode_step(dec.q[t], dec.k[t], dec.v[t], dec.g[t], dec.beta[t], S)
        o_all[t] = o[idx_n, idx_h]
        if t + 1 in snap_steps:
            snaps_gpu[t + 1] = S[idx_n, idx_h].clone()
    torch.cuda.synchronize()
    o_ref, S_ref, snaps = _oracle_steps(dec, chains, S0_cpu, snap_t=snap_steps)
    tol = TOL[w["dtype"]]
    assert rel(o_all.transpose(0, 1), o_ref, "o 1000 steps") <= tol
    assert rel(S[idx_n, idx_h], S_ref, "S after 1000 steps") <= tol
    for j, t in enumerate(snap_steps):
        ref = np.stack([snaps[j, c, 0] for c in range(len(chains))])
        assert rel(snaps_gpu[t], ref, "S at step %d" % t) <= tol, t


def test_decode_deterministic_and_guarded():
    dec = workloads.decode_inputs(1, 7, 2, 128, torch.bfloat16, seed=3)
    guard = 1024
    buf = torch.full((guard * 2 + 7 * 2 * 128 * 128,), float("nan"), device=dev())
    S = buf[guard:-guard].view(7, 2, 128, 128)
    S.copy_(dec.S0)
    args = [x[0].to(dev()) for x in (dec.q, dec.k, dec.v, dec.g, dec.beta)]
    o1 = libkda.decode_step(*args, S)
    S1 = S.clone()
    S.copy_(dec.S0)
    o2 = libkda.decode_step(*args, S)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(S, S1)
    assert bool(torch.isnan(buf[:guard]).all()) and bool(torch.isnan(buf[-guard:]).all())
