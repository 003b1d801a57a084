"""Seeded synthetic inputs for the chunk-level gated delta rule.

This module holds the input recipe only (distributions, shapes, chunk
boundaries): none of the method's arithmetic. Both the CUDA tests and the CPU
oracle are fed from it.

Recipe (per token and head):
  q, k ~ N(0, 1), each L2-normalised over its head dimension
  v    ~ N(0, 1)
  beta = sigmoid(N(0, 1))                 (write strength, already in (0, 1))
  g    = -softplus(N(0, 1) + 2)           (log-decay, alpha = exp(g) ~ 0.16)
  do   ~ N(0, 1) * do_scale               (upstream gradient of o)
  dS_out = 0 at the end of the sequence
Values are drawn in fp32 with a torch generator seeded per workload, then cast
to the workload's dtype. A "weak" decay variant g = -0.1 * softplus(N(0,1) - 5)
(alpha ~ 0.9995) keeps the boundary state alive across long spans, so that
S_in, S_out and dS_in carry weight in tests.

The workloads stand in for the long-context training runs of the StateFlow
pages (256K context, N chunks per sequence, hybrid alpha partition); no
dataset is involved.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

from .partition import hybrid_boundaries

BLOCK = 64


@dataclass
class Workload:
    name: str
    B: int
    T: int
    H: int
    dk: int
    dv: int
    dtype: str                      # "f32" or "bf16"
    chunks: list = field(default_factory=list)   # chunk lengths (fixed-length API)
    seqlens: list | None = None     # varlen sequence lengths (B == 1)
    do_scale: float = 1.0
    seed: int = 1234

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


def varlen_lengths(total: int = 131072, seed: int = 0, mu: float = math.log(4096),
                   sigma: float = 1.2, lo: int = 64, hi: int = 65536, mult: int = 64):
    """Lognormal sequence lengths, clipped, rounded to multiples of 64, packed to `total`."""
    rng = np.random.default_rng(seed)
    out, acc = [], 0
    while acc < total:
        x = float(np.exp(rng.normal(mu, sigma)))
        L = int(min(hi, max(lo, round(x / mult) * mult)))
        L = min(L, total - acc)
        out.append(L)
        acc += L
    return out


def workloads():
    """The five workloads: a tiny fp32 exactness case and four bf16 cases."""
    return [
        Workload("tiny_fp32_exactness_B1_H2_T256_d64", 1, 256, 2, 64, 64, "f32",
                 chunks=[128, 128], seed=1234),
        Workload("mid_bf16_B1_H16_T8192_d128_4x2048", 1, 8192, 16, 128, 128, "bf16",
                 chunks=[2048] * 4, seed=1235),
        Workload("long_bf16_B1_H16_T262144_d128_8x32768", 1, 262144, 16, 128, 128, "bf16",
                 chunks=[32768] * 8, do_scale=0.02, seed=1236),
        Workload("hybrid_bf16_B1_H32_T131072_d128_alpha0.5", 1, 131072, 32, 128, 128, "bf16",
                 chunks=[int(x) for x in np.diff(hybrid_boundaries(131072, 8, 0.5))],
                 seed=1237),
        Workload("varlen_bf16_H16_T131072_dk128_dv256", 1, 131072, 16, 128, 256, "bf16",
                 seqlens=varlen_lengths(), seed=1238),
    ]


def workload(i: int) -> Workload:
    return workloads()[i]


def cu_seqlens(seqlens) -> torch.Tensor:
    cu = np.zeros(len(seqlens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(seqlens)
    return torch.from_numpy(cu)


def make_inputs(B, T, H, dk, dv, dtype=torch.bfloat16, seed=1234, device="cpu",
                decay="default", do_scale=1.0, with_state=False, state_batch=None):
    """Draw one problem. Returns a dict of tensors on `device`.

    decay: "default" (-softplus(N+2)), "weak" (-0.1 softplus(N-5)) or "zero" (g = 0).
    with_state: also draw S_in ~ N(0,1) * 0.1 and dS_out ~ N(0,1) * 0.1
    (fp32, [state_batch or B, H, dk, dv]); otherwise they are absent (zero).
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)

    def randn(*shape):
        return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)

    q = randn(B, T, H, dk)
    k = randn(B, T, H, dk)
    q = q / q.norm(dim=-1, keepdim=True).clamp_min(1e-6)
    k = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-6)
    v = randn(B, T, H, dv)
    beta = torch.sigmoid(randn(B, T, H))
    z = randn(B, T, H)
    if decay == "default":
        g = -torch.nn.functional.softplus(z + 2.0)
    elif decay == "weak":
        g = -0.1 * torch.nn.functional.softplus(z - 5.0)
    elif decay == "zero":
        g = torch.zeros_like(z)
    else:
        raise ValueError(decay)
    do = randn(B, T, H, dv) * do_scale
    out = {k_: t.to(dtype) for k_, t in
           dict(q=q, k=k, v=v, g=g, beta=beta, do=do).items()}
    if with_state:
        nb = state_batch or B
        out["S_in"] = randn(nb, H, dk, dv) * 0.1
        out["dS_out"] = randn(nb, H, dk, dv) * 0.1
    return out


def make_workload_inputs(w: Workload, device="cpu", **kw):
    return make_inputs(w.B, w.T, w.H, w.dk, w.dv, dtype=w.torch_dtype, seed=w.seed,
                       device=device, do_scale=w.do_scale, **kw)


# ---------------------------------------------------------------- short convolution
# Recipe for the causal short convolution carried across chunks (the auxiliary
# local-convolution states): x ~ N(0, 1), weights ~ N(0, 1) / sqrt(W),
# bias ~ 0.1 N(0, 1), incoming state ~ N(0, 1) (zeros at a sequence start),
# dy ~ N(0, 1), dstate_out ~ N(0, 1). The benchmark's case is a Gated DeltaNet
# layer's q / k / v convolution on the 256K-token workload: C = 16 heads x
# (128 + 128 + 128) channels, W = 4, SiLU, 8 chained chunks of 32768 tokens.
CONV_BENCH = dict(B=1, T=262144, C=16 * 384, W=4, chunks=[32768] * 8, act="silu")


def make_conv_inputs(B, T, C, W, dtype=torch.bfloat16, seed=4321, device="cpu",
                     with_state=True, with_bias=True):
    gen = torch.Generator().manual_seed(seed)
    r = lambda *shape: torch.randn(*shape, generator=gen, dtype=torch.float32)
    out = {
        "x": r(B, T, C).to(dtype),
        "w": r(C, W) / math.sqrt(W),
        "b": 0.1 * r(C) if with_bias else None,
        "dy": r(B, T, C).to(dtype),
        "state_in": r(B, W - 1, C).to(dtype) if with_state else None,
        "dstate_out": r(B, W - 1, C).to(dtype) if with_state else None,
    }
    return {k: (v.to(device) if v is not None else None) for k, v in out.items()}
