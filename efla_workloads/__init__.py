"""Seeded synthetic workloads for the EFLA token mixer.

This module only draws random inputs; it holds none of the method's arithmetic.
It is the one piece of code that both the CUDA path's callers and the oracle's
callers use, so that both see bit-identical inputs.

The five workloads mirror the layer shapes of the language models the EFLA
summary pages report on (340M- and 1.3B-parameter models, page es,
"Resultados Experimentales" item 1) plus a stiff long-context case (the
large-key-norm regime of page es, "Enunciado del Problema") and a recurrent
decode step.  No dataset or trained weight is involved: every tensor is drawn
from a torch CPU generator seeded with the workload index.

Draw order within a workload: q, k direction, k norm, v, beta, S0, dO.
  q      ~ N(0,1), times 1/sqrt(d_k) where the workload says so
  k      = direction/||direction|| * norm, norm from the workload's law
  v      ~ N(0,1)
  beta   = sigmoid(N(mu_beta, 1))
  S0     = 0, or N(0, sigma_S0^2) (fp32)
  dO     ~ N(0,1)
q, k, v, dO are rounded to the workload's input dtype before anyone sees them.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int            # seed
    B: int
    H: int
    L: int
    dk: int
    dv: int
    chunk: int
    dtype: torch.dtype    # q, k, v, dO
    q_scaled: bool        # q times 1/sqrt(dk)
    knorm: str            # "lognormal" (LogNormal(0, 0.5)) or "uniform" (U[0.01, 10])
    beta_mu: float        # beta = sigmoid(N(beta_mu, 1))
    s0_std: float         # 0 -> S0 = zeros
    with_grad: bool       # draw dO
    steps: int = 0        # decode workloads: number of successive tokens


TINY_FP32 = Workload("tiny_fp32_B1H1L64d16", 0, 1, 1, 64, 16, 16, 16, torch.float32,
                     True, "lognormal", 0.0, 0.0, False)
LM340M_FWD = Workload("lm340m_fwd_B8H8L2048d128", 1, 8, 8, 2048, 128, 128, 64, torch.bfloat16,
                      True, "lognormal", 0.0, 0.0, False)
LM1P3B_FWDBWD = Workload("lm1p3b_fwdbwd_B4H16L4096d128", 2, 4, 16, 4096, 128, 128, 64,
                         torch.bfloat16, True, "lognormal", 0.0, 0.02, True)
STIFF_LONG = Workload("stiff_long_B1H16L65536d128", 3, 1, 16, 65536, 128, 128, 64, torch.bfloat16,
                      False, "uniform", 2.0, 0.0, False)
DECODE = Workload("decode_B256H16d128x1024", 4, 256, 16, 1, 128, 128, 1, torch.bfloat16,
                  False, "lognormal", 0.0, 0.0, False, steps=1024)

ALL = (TINY_FP32, LM340M_FWD, LM1P3B_FWDBWD, STIFF_LONG, DECODE)


def resized(w: Workload, **kw) -> Workload:
    """Same distributions, other sizes (parity cases the oracle finishes in seconds)."""
    return dataclasses.replace(w, **kw)


def _keys(g: torch.Generator, shape, knorm: str) -> torch.Tensor:
    kdir = torch.randn(shape, generator=g, dtype=torch.float64)
    n = shape[:-1]
    if knorm == "lognormal":
        r = torch.exp(0.5 * torch.randn(n, generator=g, dtype=torch.float64))
    elif knorm == "uniform":
        r = 0.01 + (10.0 - 0.01) * torch.rand(n, generator=g, dtype=torch.float64)
    else:
        raise ValueError(knorm)
    nrm = kdir.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    return kdir / nrm * r.unsqueeze(-1)


def make_inputs(w: Workload, seed: Optional[int] = None) -> dict:
    """Chunked-forward/backward inputs of workload ``w`` as torch CPU tensors.

    Keys: q, k, v (w.dtype), beta (fp32), S0 (fp32 or None), dO (w.dtype or None)."""
    g = torch.Generator().manual_seed(w.index if seed is None else seed)
    B, H, L, dk, dv = w.B, w.H, w.L, w.dk, w.dv
    q = torch.randn((B, H, L, dk), generator=g, dtype=torch.float64)
    if w.q_scaled:
        q = q / math.sqrt(dk)
    k = _keys(g, (B, H, L, dk), w.knorm)
    v = torch.randn((B, H, L, dv), generator=g, dtype=torch.float64)
    beta = torch.sigmoid(w.beta_mu + torch.randn((B, H, L), generator=g, dtype=torch.float64))
    S0 = None
    if w.s0_std > 0:
        S0 = (w.s0_std * torch.randn((B, H, dk, dv), generator=g, dtype=torch.float64)).float()
    dO = None
    if w.with_grad:
        dO = torch.randn((B, H, L, dv), generator=g, dtype=torch.float64).to(w.dtype)
    return dict(q=q.to(w.dtype), k=k.to(w.dtype), v=v.to(w.dtype), beta=beta.float(),
                S0=S0, dO=dO)


class DecodeStream:
    """Successive single-token inputs for a decode workload (one draw per step)."""

    def __init__(self, w: Workload, seed: Optional[int] = None):
        self.w = w
        self.g = torch.Generator().manual_seed(w.index if seed is None else seed)

    def next(self) -> dict:
        w, g = self.w, self.g
        B, H, dk, dv = w.B, w.H, w.dk, w.dv
        q = torch.randn((B, H, dk), generator=g, dtype=torch.float64)
        if w.q_scaled:
            q = q / math.sqrt(dk)
        k = _keys(g, (B, H, dk), w.knorm)
        v = torch.randn((B, H, dv), generator=g, dtype=torch.float64)
        beta = torch.sigmoid(w.beta_mu + torch.randn((B, H), generator=g, dtype=torch.float64))
        return dict(q=q.to(w.dtype), k=k.to(w.dtype), v=v.to(w.dtype), beta=beta.float())


def decode_inputs_device(w: Workload, steps: int, device, seed: Optional[int] = None) -> dict:
    """All ``steps`` decode tokens drawn at once with a device generator (benchmark use).

    Same distributions as DecodeStream, different stream of numbers.
    Shapes: q,k [steps,B,H,dk], v [steps,B,H,dv], beta [steps,B,H]."""
    g = torch.Generator(device=device).manual_seed(1000 + (w.index if seed is None else seed))
    B, H, dk, dv = w.B, w.H, w.dk, w.dv
    q = torch.randn((steps, B, H, dk), generator=g, device=device)
    if w.q_scaled:
        q = q / math.sqrt(dk)
    kdir = torch.randn((steps, B, H, dk), generator=g, device=device)
    if w.knorm == "lognormal":
        r = torch.exp(0.5 * torch.randn((steps, B, H), generator=g, device=device))
    else:
        r = 0.01 + 9.99 * torch.rand((steps, B, H), generator=g, device=device)
    k = kdir / kdir.norm(dim=-1, keepdim=True).clamp_min(1e-30) * r.unsqueeze(-1)
    v = torch.randn((steps, B, H, dv), generator=g, device=device)
    beta = torch.sigmoid(w.beta_mu + torch.randn((steps, B, H), generator=g, device=device))
    return dict(q=q.to(w.dtype), k=k.to(w.dtype), v=v.to(w.dtype), beta=beta.float())


def fwd_inputs_device(w: Workload, device, seed: Optional[int] = None) -> dict:
    """Chunked-forward inputs drawn directly on ``device`` (benchmark use at full size).

    Same distributions as make_inputs, different stream of numbers."""
    g = torch.Generator(device=device).manual_seed(2000 + (w.index if seed is None else seed))
    B, H, L, dk, dv = w.B, w.H, w.L, w.dk, w.dv
    q = torch.randn((B, H, L, dk), generator=g, device=device)
    if w.q_scaled:
        q = q / math.sqrt(dk)
    kdir = torch.randn((B, H, L, dk), generator=g, device=device)
    if w.knorm == "lognormal":
        r = torch.exp(0.5 * torch.randn((B, H, L), generator=g, device=device))
    else:
        r = 0.01 + 9.99 * torch.rand((B, H, L), generator=g, device=device)
    k = kdir / kdir.norm(dim=-1, keepdim=True).clamp_min(1e-30) * r.unsqueeze(-1)
    v = torch.randn((B, H, L, dv), generator=g, device=device)
    beta = torch.sigmoid(w.beta_mu + torch.randn((B, H, L), generator=g, device=device))
    S0 = None
    if w.s0_std > 0:
        S0 = w.s0_std * torch.randn((B, H, dk, dv), generator=g, device=device)
    dO = None
    if w.with_grad:
        dO = torch.randn((B, H, L, dv), generator=g, device=device).to(w.dtype)
    return dict(q=q.to(w.dtype), k=k.to(w.dtype), v=v.to(w.dtype), beta=beta, S0=S0, dO=dO)


# ------------------------------------------------------------- token mixer
@dataclasses.dataclass(frozen=True)
class MixerWorkload:
    """Input projections of one EFLA layer: tokens x [B, L, D] and the stacked weight
    [Wq; Wk; Wv; Wb] of 3 H dk + H output features."""
    name: str
    index: int            # seed
    B: int
    L: int
    D: int                # d_model
    H: int
    dk: int = 128


MIXER_340M = MixerWorkload("mixer340m_B8L2048D1024H8", 11, 8, 2048, 1024, 8)
MIXER_1P3B = MixerWorkload("mixer1p3b_B4L4096D2048H16", 12, 4, 4096, 2048, 16)


def mixer_inputs(w: MixerWorkload, device="cpu", seed: Optional[int] = None) -> dict:
    """x ~ N(0, 1) and weights ~ N(0, 1/D) (unit-variance outputs), both rounded to bf16;
    drawn on `device` (a CPU generator for CPU tensors)."""
    g = torch.Generator(device=device).manual_seed(w.index if seed is None else seed)
    x = torch.randn((w.B, w.L, w.D), generator=g, device=device)
    wt = torch.randn((3 * w.H * w.dk + w.H, w.D), generator=g, device=device) / math.sqrt(w.D)
    return dict(x=x.to(torch.bfloat16), w=wt.to(torch.bfloat16))
