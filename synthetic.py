"""Seeded synthetic inputs shared by the tests, the smoke check and bench.py.

This module draws random tensors and nothing else: it holds none of the
recurrence's arithmetic.  Both the CUDA path and the fp64 oracle consume the
tensors it returns (the oracle through ``to_oracle``, which only re-interprets
bits).

Workloads (value distributions as the pages' experiments and the task fix them):

  taylor_fp32_small   Taylor linear attention, fp32: B=1, H=2, N=256, d'=16,
                      d_v=64; q, k ~ N(0,1)/sqrt(d'), v ~ N(0,1); seed 0.
  based_prefill       BASED Taylor prefill, bf16 in / fp32 state: B=8, H=16,
                      N=4096, d'=16, d_v=64; same distributions; seed 1.
  gdn_prefill         Gated DeltaNet prefill, bf16 in / fp32 state: B=4,
                      H=16, N=16384, d_k=d_v=128; q, k L2-normalised Gaussian
                      (normalised in fp32, then rounded to bf16), v ~ N(0,1),
                      beta = sigmoid(N(0,1)), alpha = exp(-U(0.001, 0.1)); seed 2.
  gdn_prefill_long    as gdn_prefill with B=1, H=16, N=1,048,576; seed 3.
  decode              256 sequences x 16 heads, one token per step, 1000 steps;
                      GDN inputs as gdn_prefill, Taylor inputs as
                      based_prefill, bf16; seed 4.

A generator runs on the device it is given; CPU and CUDA streams of random
numbers differ, so a test draws once and hands the same tensors to both sides.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

TAYLOR_DFEAT = 16
TAYLOR_DV = 64
GDN_D = 128


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str          # "taylor" | "gdn" | "decode"
    B: int
    H: int
    N: int
    dtype: torch.dtype
    seed: int
    description: str


WORKLOADS = {
    "taylor_fp32_small": Workload("taylor_fp32_small", "taylor", 1, 2, 256, torch.float32, 0,
                                  "Taylor linear attention fp32 B=1 H=2 N=256 d'=16 d_v=64"),
    "based_prefill": Workload("based_prefill", "taylor", 8, 16, 4096, torch.bfloat16, 1,
                              "BASED Taylor prefill bf16/fp32-state B=8 H=16 N=4096 d'=16 D=273 d_v=64"),
    "gdn_prefill": Workload("gdn_prefill", "gdn", 4, 16, 16384, torch.bfloat16, 2,
                            "Gated DeltaNet prefill bf16/fp32-state B=4 H=16 N=16384 d_k=d_v=128"),
    "gdn_prefill_long": Workload("gdn_prefill_long", "gdn", 1, 16, 1048576, torch.bfloat16, 3,
                                 "Gated DeltaNet prefill bf16/fp32-state B=1 H=16 N=1048576 d_k=d_v=128"),
    "decode": Workload("decode", "decode", 256, 16, 1000, torch.bfloat16, 4,
                       "recurrent decode 256 seqs x H=16, 1000 steps; GDN 128x128 and Taylor 273x64 fp32 state"),
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(shape, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def taylor_inputs(B, H, N, dtype=torch.bfloat16, seed=0, device="cpu",
                  dfeat=TAYLOR_DFEAT, dv=TAYLOR_DV):
    """q, k ~ N(0,1)/sqrt(d'), v ~ N(0,1); layout [B,H,N,d] contiguous."""
    g = _gen(device, seed)
    scale = 1.0 / math.sqrt(dfeat)
    q = (_randn((B, H, N, dfeat), g, device) * scale).to(dtype)
    k = (_randn((B, H, N, dfeat), g, device) * scale).to(dtype)
    v = _randn((B, H, N, dv), g, device).to(dtype)
    return {"q": q, "k": k, "v": v}


def _l2_normalised(shape, g, device, dtype):
    x = _randn(shape, g, device)
    x = x / x.norm(dim=-1, keepdim=True)
    return x.to(dtype)


def gdn_inputs(B, H, N, dtype=torch.bfloat16, seed=2, device="cpu", dk=GDN_D, dv=GDN_D):
    """q, k L2-normalised Gaussian, v ~ N(0,1), beta = sigmoid(N(0,1)),
    alpha = exp(-U(0.001, 0.1)); alpha, beta fp32 [B,H,N]."""
    g = _gen(device, seed)
    q = _l2_normalised((B, H, N, dk), g, device, dtype)
    k = _l2_normalised((B, H, N, dk), g, device, dtype)
    v = _randn((B, H, N, dv), g, device).to(dtype)
    beta = torch.sigmoid(_randn((B, H, N), g, device))
    u = torch.rand((B, H, N), generator=g, device=device, dtype=torch.float32)
    alpha = torch.exp(-(0.001 + (0.1 - 0.001) * u))
    return {"q": q, "k": k, "v": v, "alpha": alpha.contiguous(), "beta": beta.contiguous()}


def decode_step_inputs(S, H, step, seed=4, device="cpu", dtype=torch.bfloat16):
    """Inputs of decode step `step` (0-based) for both variants; [S,H,d]."""
    base = int(seed) * 1_000_003 + int(step)
    g = gdn_inputs(S, H, 1, dtype=dtype, seed=2 * base, device=device)
    t = taylor_inputs(S, H, 1, dtype=dtype, seed=2 * base + 1, device=device)
    out = {"gdn": {name: x.squeeze(2).contiguous() for name, x in g.items()},
           "taylor": {name: x.squeeze(2).contiguous() for name, x in t.items()}}
    return out


def workload_inputs(name: str, device="cpu", **override):
    w = WORKLOADS[name]
    B, H, N = override.get("B", w.B), override.get("H", w.H), override.get("N", w.N)
    seed = override.get("seed", w.seed)
    if w.kind == "taylor":
        return taylor_inputs(B, H, N, dtype=w.dtype, seed=seed, device=device)
    if w.kind == "gdn":
        return gdn_inputs(B, H, N, dtype=w.dtype, seed=seed, device=device)
    raise ValueError(f"{name} is generated per step: use decode_step_inputs")


def to_oracle(t: torch.Tensor) -> np.ndarray:
    """Hand a tensor to the oracle: fp32 as float32, bf16 as its raw uint16 bits."""
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError(f"unsupported dtype {t.dtype}")
