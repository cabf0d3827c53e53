"""Seeded synthetic workloads for DualKV shared-prompt attention.

This module only describes layouts and draws inputs; it holds none of the
attention arithmetic, so both the CUDA path's tests/benchmark and the fp64
oracle can take their inputs from it.

The workloads stand in for the training jobs of the DualKV paper (abstract:
GRPO and DAPO on Qwen3-8B, N=32 responses, 8K context; a Gemma-style hybrid
sliding/global model with head dimension 512).  No model, dataset or weights
are involved: one attention layer's q, k, v and upstream gradient dO are drawn
i.i.d. N(0, 1) in float32 from a seeded CPU generator, in the order q, k, v,
dO, then rounded to bf16 (round to nearest even).  The softmax scale is
1/sqrt(D).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch

# Ragged DAPO-like response lengths: numpy.random.default_rng(20260518)
# .integers(256, 4097, size=32), i.e. uniform on [256, 4096], stored verbatim.
DAPO_R = [666, 568, 1324, 1784, 1600, 1760, 3827, 3350, 3573, 3205, 353, 1333, 3601, 3053, 752, 2281,
          1065, 2648, 430, 3867, 3147, 3535, 4087, 1893, 3449, 3750, 3493, 2554, 3651, 1800, 621, 3774]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    P: int
    R: tuple  # response lengths R_0..R_{N-1}
    Hq: int
    Hkv: int
    D: int
    window: int  # <= 0: global causal; else keys with 0 <= pos_q - pos_k < window
    seed: int

    @property
    def N(self) -> int:
        return len(self.R)

    @property
    def offsets(self) -> List[int]:
        off = [0]
        for r in self.R:
            off.append(off[-1] + int(r))
        return off

    @property
    def T(self) -> int:
        return self.P + sum(self.R)

    @property
    def T_replicated(self) -> int:
        return self.N * self.P + sum(self.R)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def replicated(self) -> "Workload":
        """The same sequences with the prompt copied into every segment (P=0)."""
        return dataclasses.replace(self, name=self.name + "-replicated", P=0,
                                   R=tuple(self.P + r for r in self.R))


WORKLOADS = {
    "tiny": Workload("tiny", 64, (32,) * 4, 2, 2, 64, 0, 20260515),
    "qwen16": Workload("qwen16", 8192, (1024,) * 16, 32, 8, 128, 0, 20260516),
    "grpo32": Workload("grpo32", 6144, (2048,) * 32, 32, 8, 128, 0, 20260517),
    "dapo32": Workload("dapo32", 8192, tuple(DAPO_R), 32, 8, 128, 0, 20260518),
    "gemma_global": Workload("gemma_global", 16384, (3072,) * 16, 8, 2, 512, 0, 20260519),
    "gemma_window": Workload("gemma_window", 16384, (3072,) * 16, 8, 2, 512, 1024, 20260519),
}


def custom(P, R, Hq, Hkv, D, window=0, seed=1234, name="custom") -> Workload:
    return Workload(name, int(P), tuple(int(r) for r in R), int(Hq), int(Hkv), int(D), int(window), int(seed))


def draw_inputs(w: Workload, with_dout: bool = True, device: Optional[str] = None):
    """q [T,Hq,D], k [T,Hkv,D], v [T,Hkv,D], dout [T,Hq,D] as bf16 tensors."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(w.seed)
    T = w.T
    shapes = [(T, w.Hq, w.D), (T, w.Hkv, w.D), (T, w.Hkv, w.D)]
    if with_dout:
        shapes.append((T, w.Hq, w.D))
    out = []
    for shp in shapes:
        x = torch.randn(shp, generator=gen, dtype=torch.float32).to(torch.bfloat16)
        out.append(x.to(device) if device else x)
    if not with_dout:
        out.append(None)
    return tuple(out)


def replicate_rows(w: Workload, x: torch.Tensor) -> torch.Tensor:
    """Copy packed rows into the replicated layout (prompt rows repeated per segment)."""
    off = w.offsets
    parts = []
    for n in range(w.N):
        parts.append(x[: w.P])
        parts.append(x[w.P + off[n]: w.P + off[n + 1]])
    return torch.cat(parts, dim=0)
