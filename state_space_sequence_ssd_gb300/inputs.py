"""Seeded synthetic inputs for the SSD forward pass (shared by tests and bench).

This module draws random numbers and names workloads; it holds none of the
method's arithmetic and imports nothing else from this package, so both the
CUDA path and the CPU oracle can be fed from it.

Recipe (one CPU torch.Generator, seeded, fixed draw order x, dt, A, B, C, D, init):
    x, B, C  ~ N(0, 1) drawn in float32, rounded to bfloat16 (round-to-nearest-even)
    dt       = softplus(N(0, 1) - 4)                    float32, always > 0
    A_h      = -exp(U(0, ln 16))                        float32, in [-16, -1]
    D_h      ~ N(0, 1)                                  float32
    init     = 0.1 * N(0, 1) (only for workloads with a non-zero initial state)
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    chunk_size: int
    nonzero_init: bool

    @property
    def nchunks(self) -> int:
        return -(-self.seqlen // self.chunk_size)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The pages' sweep: 1K-256K tokens, state size 64-512, headdim 64, chunk 256.
WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_L512_N64", 1, 512, 4, 64, 64, 1, 64, False),
        Workload("mamba2_1p3b_layer_2x4096_N128", 2, 4096, 64, 64, 128, 1, 256, False),
        Workload("long_L65536_N128", 1, 65536, 32, 64, 128, 1, 256, True),
        Workload("state_sweep_L16384_N64", 1, 16384, 32, 64, 64, 1, 256, False),
        Workload("state_sweep_L16384_N128", 1, 16384, 32, 64, 128, 1, 256, False),
        Workload("state_sweep_L16384_N256", 1, 16384, 32, 64, 256, 1, 256, False),
        Workload("state_sweep_L16384_N512", 1, 16384, 32, 64, 512, 1, 256, False),
        Workload("longest_L262144_N256_G8", 1, 262144, 32, 64, 256, 8, 256, True),
    ]
}

HEADLINE = "long_L65536_N128"


def make_inputs(w: Workload, seed: int = 0) -> dict:
    """CPU torch tensors for workload ``w``; bf16 tensors are torch.bfloat16."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    b, L, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    x = torch.randn((b, L, H, P), generator=g, dtype=torch.float32).to(torch.bfloat16)
    dt = torch.nn.functional.softplus(torch.randn((b, L, H), generator=g, dtype=torch.float32) - 4.0)
    A = -torch.exp(torch.rand((H,), generator=g, dtype=torch.float32) * math.log(16.0))
    B = torch.randn((b, L, G, N), generator=g, dtype=torch.float32).to(torch.bfloat16)
    C = torch.randn((b, L, G, N), generator=g, dtype=torch.float32).to(torch.bfloat16)
    D = torch.randn((H,), generator=g, dtype=torch.float32)
    if w.nonzero_init:
        init = 0.1 * torch.randn((b, H, P, N), generator=g, dtype=torch.float32)
    else:
        init = None
    return {"x": x, "dt": dt, "A": A, "B": B, "C": C, "D": D, "init": init}


def make_layer_options(w: Workload, seed: int = 0) -> dict:
    """Seeded inputs of a whole layer's input-side options for workload ``w`` (CPU torch tensors):
        dt_raw  ~ N(0, 1)                    float32 (batch, L, H): the pre-activation dt
        dt_bias ~ U(-6, -2)                  float32 (H,)
        D_hp    ~ N(0, 1)                    float32 (H, P): one skip weight per channel
        z       ~ N(0, 1) rounded to bf16    (batch, L, H, P): the output gate
        dt_limit = (0.001, 0.1)
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(10_000 + seed)
    b, L, H, P = w.batch, w.seqlen, w.nheads, w.headdim
    dt_raw = torch.randn((b, L, H), generator=g, dtype=torch.float32)
    dt_bias = torch.rand((H,), generator=g, dtype=torch.float32) * 4.0 - 6.0
    D_hp = torch.randn((H, P), generator=g, dtype=torch.float32)
    z = torch.randn((b, L, H, P), generator=g, dtype=torch.float32).to(torch.bfloat16)
    return {"dt_raw": dt_raw, "dt_bias": dt_bias, "D_hp": D_hp, "z": z, "dt_limit": (0.001, 0.1)}


def make_grad_inputs(w: Workload, seed: int = 0, dfinal: bool = True) -> dict:
    """Seeded output gradients for workload ``w`` (CPU torch tensors), the inputs of the backward pass:
        dy     ~ N(0, 1) rounded to bf16        (batch, L, H, P): dLoss/dy
        dfinal ~ N(0, 1)                        float32 (batch, H, P, N): dLoss/dfinal (None if not asked for)
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(20_000 + seed)
    b, L, H, P, N = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate
    dy = torch.randn((b, L, H, P), generator=g, dtype=torch.float32).to(torch.bfloat16)
    df = torch.randn((b, H, P, N), generator=g, dtype=torch.float32) if dfinal else None
    return {"dy": dy, "dfinal": df}


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bfloat16 torch tensor -> numpy uint16 bit patterns (no copy of values' meaning)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def as_numpy(inp: dict) -> dict:
    """Numpy views for the oracle: bf16 tensors as uint16 bits, others float32."""
    out = {}
    for k, v in inp.items():
        if v is None:
            out[k] = None
        elif v.dtype == torch.bfloat16:
            out[k] = bf16_bits(v)
        else:
            out[k] = v.contiguous().numpy()
    return out
