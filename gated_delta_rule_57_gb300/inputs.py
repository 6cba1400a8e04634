"""Seeded synthetic inputs for KDA prefill and decode.

This module is shared by the tests, the benchmark and the smoke check. It
draws random tensors and nothing else: it holds none of KDA's arithmetic.

Recipe (all draws from one ``torch.Generator`` seeded per workload, in the
order q, k, v, beta-logit, g-logit, initial state):
  q, k   ~ N(0, 1), then L2-normalised per (b, t, h) vector in fp32, then cast
           to the I/O type;
  v      ~ N(0, 1), cast to the I/O type;
  beta   = sigmoid(N(0, 1))  (fp32);
  g      = -5 * sigmoid(N(0, 1)) per channel (fp32), i.e. inside (-5, 0);
  h0 / S ~ N(0, 0.02^2) fp32 where the workload has an initial state.
The log-decay bound g >= -5 is the one stated on the orkas.ai page "Kimi K3
architecture", section "A lower bound that deleted a GPU code path".
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class PrefillWorkload:
    name: str
    B: int
    T: int
    H: int
    dk: int
    dv: int
    io: str  # "bf16" or "f32"
    seed: int
    h0_std: Optional[float] = None  # None: zero initial state (h0 = NULL)
    stress_heads: bool = False  # heads H/2..H-1 get g = -4.99 everywhere


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    name: str
    N: int
    H: int
    dk: int
    dv: int
    io: str
    seed: int
    steps: int
    S_std: float = 0.02


# The five workloads of the benchmark spec, by what they are.
TINY_F32 = PrefillWorkload("prefill_tiny_f32_b1_t256_h2_d64", 1, 256, 2, 64, 64, "f32", 0)
PREFILL_T4K = PrefillWorkload("prefill_bf16_b1_t4096_h32_d128_stress", 1, 4096, 32, 128, 128,
                              "bf16", 1, stress_heads=True)
PREFILL_B8_T8K = PrefillWorkload("prefill_bf16_b8_t8192_h32_d128", 8, 8192, 32, 128, 128,
                                 "bf16", 2, h0_std=0.02)
PREFILL_T1M = PrefillWorkload("prefill_bf16_b1_t1048576_h32_d128", 1, 1 << 20, 32, 128, 128,
                              "bf16", 3)
DECODE_N256 = DecodeWorkload("decode_bf16_n256_h32_d128", 256, 32, 128, 128, "bf16", 4, 1000)

WORKLOADS = {w.name: w for w in (TINY_F32, PREFILL_T4K, PREFILL_B8_T8K, PREFILL_T1M, DECODE_N256)}

_IO = {"bf16": torch.bfloat16, "f32": torch.float32}


def io_dtype(io: str) -> torch.dtype:
    return _IO[io]


def _unit(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True)


def prefill_inputs(w: PrefillWorkload, device="cpu", *, B: Optional[int] = None,
                   T: Optional[int] = None, H: Optional[int] = None, seed: Optional[int] = None):
    """Draw one prefill batch. B, T, H, seed override the workload's (for small cases)."""
    B = w.B if B is None else B
    T = w.T if T is None else T
    H = w.H if H is None else H
    seed = w.seed if seed is None else seed
    dt = io_dtype(w.io)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    kw = dict(generator=gen, device=device, dtype=torch.float32)
    q = _unit(torch.randn(B, T, H, w.dk, **kw)).to(dt)
    k = _unit(torch.randn(B, T, H, w.dk, **kw)).to(dt)
    v = torch.randn(B, T, H, w.dv, **kw).to(dt)
    beta = torch.sigmoid(torch.randn(B, T, H, **kw))
    g = torch.randn(B, T, H, w.dk, **kw)
    g = torch.sigmoid(g).mul_(-5.0)
    if w.stress_heads:
        g[:, :, H // 2:, :] = -4.99
    h0 = None
    if w.h0_std is not None:
        h0 = torch.randn(B, H, w.dk, w.dv, **kw).mul_(w.h0_std)
    return dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0)


def decode_inputs(w: DecodeWorkload, device="cpu", *, N: Optional[int] = None,
                  H: Optional[int] = None, steps: Optional[int] = None,
                  seed: Optional[int] = None):
    """Draw the initial state and `steps` fresh tokens per sequence.

    Returns q, k [steps, N, H, dk], v [steps, N, H, dv], g [steps, N, H, dk],
    beta [steps, N, H] and S [N, H, dk, dv].
    """
    N = w.N if N is None else N
    H = w.H if H is None else H
    steps = w.steps if steps is None else steps
    seed = w.seed if seed is None else seed
    dt = io_dtype(w.io)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    kw = dict(generator=gen, device=device, dtype=torch.float32)
    q = _unit(torch.randn(steps, N, H, w.dk, **kw)).to(dt)
    k = _unit(torch.randn(steps, N, H, w.dk, **kw)).to(dt)
    v = torch.randn(steps, N, H, w.dv, **kw).to(dt)
    beta = torch.sigmoid(torch.randn(steps, N, H, **kw))
    g = torch.sigmoid(torch.randn(steps, N, H, w.dk, **kw)).mul_(-5.0)
    S = torch.randn(N, H, w.dk, w.dv, **kw).mul_(w.S_std)
    return dict(q=q, k=k, v=v, g=g, beta=beta, S=S)
