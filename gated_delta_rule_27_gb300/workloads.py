"""Seeded synthetic inputs for the KDA recurrence.

This module only draws random tensors with the shapes, dtypes and
distributions of the five workloads the library is checked and measured on.
It holds none of the recurrence's arithmetic, so the CUDA path's tests and
the fp64 oracle can both take their inputs from it.

Distributions (per the workload descriptions):
  * q, k : N(0, 1) per element, then L2-normalised per (token, head) in fp32,
    then rounded to the input dtype (bf16 or fp32);
  * v    : N(0, 1), rounded to the input dtype;
  * beta : sigmoid(N(0, 1)) in fp32;
  * g    : log-decay, -exp(N(-1, 0.5)) per channel in fp32, so that the
    decay exp(g) lies in (0, 1);
  * decode state S0 : N(0, 0.1) in fp32 (0.1 is the standard deviation).
Each tensor has its own torch.Generator, seeded from the workload seed and
the tensor's position in the fixed order (q, k, v, g, beta, S0, lengths).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

BASE_SEED = 20261202

_ORDER = {"q": 0, "k": 1, "v": 2, "g": 3, "beta": 4, "S0": 5, "lengths": 6, "extreme": 7}


def _gen(seed: int, name: str, device) -> torch.Generator:
    gen = torch.Generator(device=device)
    gen.manual_seed(seed * 16 + _ORDER[name])
    return gen


@dataclasses.dataclass
class PrefillInputs:
    q: torch.Tensor          # [T, H, d] in_dtype
    k: torch.Tensor          # [T, H, d] in_dtype
    v: torch.Tensor          # [T, H, d] in_dtype
    g: torch.Tensor          # [T, H, d] fp32
    beta: torch.Tensor       # [T, H] fp32
    cu_seqlens: torch.Tensor  # [N + 1] int32
    S0: Optional[torch.Tensor]  # [N, H, d, d] fp32 or None

    @property
    def num_seqs(self) -> int:
        return self.cu_seqlens.numel() - 1

    @property
    def total_tokens(self) -> int:
        return self.q.shape[0]


def _l2_normalised(shape, gen, device, dtype):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    x = x / torch.linalg.vector_norm(x, dim=-1, keepdim=True).clamp_min(1e-12)
    return x.to(dtype)


def random_qkvgb(T: int, H: int, d: int, dtype: torch.dtype, seed: int, device="cpu"):
    """q, k, v, g, beta with the workload distributions."""
    q = _l2_normalised((T, H, d), _gen(seed, "q", device), device, dtype)
    k = _l2_normalised((T, H, d), _gen(seed, "k", device), device, dtype)
    v = torch.randn((T, H, d), generator=_gen(seed, "v", device), device=device, dtype=torch.float32).to(dtype)
    g = -torch.exp(torch.normal(-1.0, 0.5, (T, H, d), generator=_gen(seed, "g", device), device=device))
    beta = torch.sigmoid(torch.randn((T, H), generator=_gen(seed, "beta", device), device=device))
    return q, k, v, g.float().contiguous(), beta.float().contiguous()


def cu_from_lengths(lengths, device="cpu") -> torch.Tensor:
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32, device=device)


def prefill_inputs(lengths, H: int, d: int, dtype: torch.dtype, seed: int, device="cpu",
                   s0_std: Optional[float] = None) -> PrefillInputs:
    """Packed prefill inputs for documents of the given lengths."""
    T = int(sum(int(n) for n in lengths))
    q, k, v, g, beta = random_qkvgb(T, H, d, dtype, seed, device)
    S0 = None
    if s0_std is not None:
        S0 = torch.normal(0.0, s0_std, (len(lengths), H, d, d), generator=_gen(seed, "S0", device),
                          device=device).float()
    return PrefillInputs(q, k, v, g, beta, cu_from_lengths(lengths, device), S0)


def varlen_lengths(num_docs: int, lo: int, hi: int, seed: int):
    """Document lengths drawn uniformly from [lo, hi] (inclusive)."""
    gen = _gen(seed, "lengths", "cpu")
    return [int(x) for x in torch.randint(lo, hi + 1, (num_docs,), generator=gen)]


@dataclasses.dataclass
class DecodeInputs:
    q: torch.Tensor      # [steps, N, H, d] in_dtype
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor      # [steps, N, H, d] fp32
    beta: torch.Tensor   # [steps, N, H] fp32
    S0: torch.Tensor     # [N, H, d, d] fp32
    extreme_steps: torch.Tensor  # indices of the steps with extreme gates


def decode_inputs(steps: int, N: int, H: int, d: int, dtype: torch.dtype, seed: int, device="cpu",
                  s0_std: float = 0.1, extreme_frac: float = 0.05) -> DecodeInputs:
    """Inputs of `steps` successive single-token steps over N sequences.

    A seeded `extreme_frac` share of the steps uses extreme gates: beta drawn
    uniformly from {0, 1} per (seq, head) and log-decay drawn uniformly from
    {-10, -1e-4} per channel.
    """
    q, k, v, g, beta = random_qkvgb(steps * N, H, d, dtype, seed, device)
    q, k, v, g = (x.view(steps, N, H, d) for x in (q, k, v, g))
    beta = beta.view(steps, N, H)
    n_ext = int(round(extreme_frac * steps))
    gen = _gen(seed, "extreme", "cpu")
    ext = torch.randperm(steps, generator=gen)[:n_ext].sort().values
    if n_ext:
        gen_d = _gen(seed, "extreme", device)
        b_bits = torch.randint(0, 2, (n_ext, N, H), generator=gen_d, device=device).float()
        g_bits = torch.randint(0, 2, (n_ext, N, H, d), generator=gen_d, device=device)
        g_ext = torch.where(g_bits.bool(), torch.tensor(-10.0, device=device), torch.tensor(-1e-4, device=device))
        idx = ext.to(device)
        beta[idx] = b_bits
        g[idx] = g_ext
    S0 = torch.normal(0.0, s0_std, (N, H, d, d), generator=_gen(seed, "S0", device), device=device).float()
    return DecodeInputs(q.contiguous(), k.contiguous(), v.contiguous(), g.contiguous(), beta.contiguous(), S0, ext)


# The five workloads, by name.  Sizes follow the workload descriptions; the
# seed of workload i is BASE_SEED + i.
WORKLOADS = {
    "tiny": dict(index=0, B=1, H=1, T=64, d=16, chunk=16, dtype=torch.float32),
    "prefill": dict(index=1, B=1, H=16, T=4096, d=128, chunk=64, dtype=torch.bfloat16),
    "varlen": dict(index=2, docs=8, len_lo=128, len_hi=8192, H=32, d=128, chunk=64, dtype=torch.bfloat16),
    "decode": dict(index=3, N=256, H=32, d=128, steps=1000, dtype=torch.bfloat16),
    "long": dict(index=4, B=2, H=32, T=65536, d=128, chunk=64, dtype=torch.bfloat16, split=32768,
                 decode_tail=64),
}


def workload_seed(name: str) -> int:
    return BASE_SEED + WORKLOADS[name]["index"]


def workload_prefill(name: str, device="cpu", head_block: int = 0) -> PrefillInputs:
    """Prefill inputs of the tiny / prefill / varlen / long workloads (zero S0).

    `head_block` b > 0 draws the inputs of heads [b H, (b + 1) H) of a larger problem made of several such
    blocks side by side (block 0 is the workload itself): the same documents, inputs from their own seed.
    """
    w = WORKLOADS[name]
    seed = workload_seed(name)
    if head_block:
        lengths_seed = seed
        seed = seed + 1000 * head_block
        if name == "varlen":
            lengths = varlen_lengths(w["docs"], w["len_lo"], w["len_hi"], lengths_seed)
            return prefill_inputs(lengths, w["H"], w["d"], w["dtype"], seed, device)
    if name == "varlen":
        lengths = varlen_lengths(w["docs"], w["len_lo"], w["len_hi"], seed)
    else:
        lengths = [w["T"]] * w["B"]
    return prefill_inputs(lengths, w["H"], w["d"], w["dtype"], seed, device)
