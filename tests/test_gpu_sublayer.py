"""The whole KDA sublayer (synthetic weights) against an fp64 composition of the same steps.

The GPU side (gated_delta_rule_27_gb300/sublayer.py) runs bf16 GEMMs and libkda's kernels; the reference runs
the same sequence in fp64 (oracle/sublayer.py for the convolution and the normalisations, the oracle for the
recurrence), rounding to bf16 where the GPU side stores bf16 tensors, so that only arithmetic error is
compared.  Tolerance: the bf16 contract, max|x - ref| / max|ref| <= 2e-2, on the sublayer output and the final
states, for a prefill and for decode steps continuing it.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gated_delta_rule_27_gb300 import sublayer, workloads
from oracle import oracle
from oracle import sublayer as ref
from tests.gpu_helpers import TOL, dev, f64, rel

pytestmark = pytest.mark.gpu


def _bf16(a):
    return torch.from_numpy(np.asarray(a)).to(torch.bfloat16).double().numpy()


def _reference_prefill(x, cu, w, H, d):
    T = x.shape[0]
    X = f64(x)
    proj = lambda W: X @ f64(W)
    q, k, v, z = (_bf16(proj(W)) for W in (w.W_q, w.W_k, w.W_v, w.W_z))
    g = -np.logaddexp(0.0, proj(w.W_a))
    beta = 1.0 / (1.0 + np.exp(-proj(w.W_b)))
    conv = lambda a, cw: ref.short_conv(a, f64(cw), cu)
    (qc, sq), (kc, sk), (vc, sv) = conv(q, w.conv_q), conv(k, w.conv_k), conv(v, w.conv_v)
    qc, kc, vc = (_bf16(a).reshape(T, H, d) for a in (qc, kc, vc))
    o, S, _ = oracle.run(ref.l2norm(qc, 1e-6), ref.l2norm(kc, 1e-6), vc, g.reshape(T, H, d), beta, cu)
    o = _bf16(ref.gated_rmsnorm(o, z.reshape(T, H, d), f64(w.out_weight), 1e-6))
    return o.reshape(T, H * d) @ f64(w.W_o), S, (sq, sk, sv)


def test_sublayer_prefill_then_decode_against_fp64():
    H, d, D = 2, 128, 256
    lengths = [150, 77]
    T = sum(lengths)
    w = sublayer.synthetic_weights(D, H, d, seed=5, device=dev())
    gen = torch.Generator().manual_seed(6)
    x = torch.randn((T, D), generator=gen).to(torch.bfloat16)
    cu = workloads.cu_from_lengths(lengths)
    y, S, conv_state = sublayer.prefill_forward(x.to(dev()), cu.to(dev()), w, H, d)
    torch.cuda.synchronize()
    y_ref, S_ref, _ = _reference_prefill(x, cu.numpy(), w, H, d)
    assert rel(y, y_ref, "y prefill") <= TOL[torch.bfloat16], rel(y, y_ref)
    assert rel(S, S_ref, "S prefill") <= TOL[torch.bfloat16], rel(S, S_ref)

    # three decode steps continuing both documents: the reference replays the whole sequences
    steps = 3
    xs = torch.randn((steps, 2, D), generator=gen).to(torch.bfloat16)
    Sd = S.clone()
    ys = [sublayer.decode_forward(xs[t].to(dev()), Sd, conv_state, w, H, d) for t in range(steps)]
    torch.cuda.synchronize()
    # reference: the documents with their decode tokens appended
    x_full = torch.cat([torch.cat([x[a:b], xs[:, n]]) for n, (a, b) in
                        enumerate(zip(cu.tolist()[:-1], cu.tolist()[1:]))])
    cu_full = workloads.cu_from_lengths([n + steps for n in lengths])
    y_full, S_full, _ = _reference_prefill(x_full, cu_full.numpy(), w, H, d)
    ends = cu_full.tolist()[1:]
    y_dec_ref = np.stack([y_full[[e - steps + t for e in ends]] for t in range(steps)])
    assert rel(torch.stack(ys), y_dec_ref, "y decode") <= TOL[torch.bfloat16], rel(torch.stack(ys), y_dec_ref)
    assert rel(Sd, S_full, "S decode") <= TOL[torch.bfloat16], rel(Sd, S_full)
