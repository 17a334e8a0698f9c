"""Shared helpers of the GPU parity tests: run libkda, run the oracle on the same inputs, compare.

Tolerance contract (fixed before measuring): max|x - ref| / max|ref|, taken
separately over all outputs o and over all states S, must be <= 1e-4 for
fp32 inputs and <= 2e-2 for bf16 inputs.
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

from oracle import oracle

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def dev():
    return torch.device("cuda:0")


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def oracle_prefill(inp, S0=None, heads=None, snap_t=None, threads=None):
    """Oracle over all (or the listed) heads of a PrefillInputs on the CPU."""
    q, k, v, g, beta = inp.q, inp.k, inp.v, inp.g, inp.beta
    if heads is not None:
        sel = list(heads)
        q, k, v, g, beta = (x[:, sel] for x in (q, k, v, g, beta))
        if S0 is not None:
            S0 = S0[:, sel]
    cu = inp.cu_seqlens.cpu().numpy()
    return oracle.run(f64(q), f64(k), f64(v), f64(g), f64(beta), cu,
                      S0=None if S0 is None else f64(S0), snap_t=snap_t, threads=threads)


def to_device(inp):
    d = dev()
    return [x.to(d) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta, inp.cu_seqlens)]


def rel(x, ref, label: str = ""):
    """max|x - ref| / max|ref|.  With KDA_PARITY_LOG set, every measured error is appended there as one JSON
    line with the running test's name, so that the margin under the tolerance can be tabulated."""
    err = oracle.rel_err(f64(x) if torch.is_tensor(x) else x, ref)
    path = os.environ.get("KDA_PARITY_LOG")
    if path:
        with open(path, "a") as fh:
            fh.write(json.dumps({"test": os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0], "label": label,
                                 "err": err}) + "\n")
    return err
