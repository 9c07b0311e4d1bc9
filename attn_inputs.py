"""Seeded synthetic inputs for the attention forward.

This module only draws random numbers and names workloads: it holds none of
the attention arithmetic, so both the GPU path and the CPU oracle can take
their inputs from it without sharing any code with each other.

Recipe (one per workload): fp32 standard normals from a CPU
``torch.Generator`` seeded per tensor, rounded to the workload's 16-bit type
(round-to-nearest-even by torch's cast).  The oracle reads the same 16-bit
values upcast to fp64, so both sides see identical inputs.  The peaked
workload multiplies K by 4 in fp32 before the cast, which makes the scaled
logits' standard deviation about 4 and the softmax rows sharply peaked.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str          # "bf16" or "fp16"
    causal: bool
    k_mult: float = 1.0  # K drawn as k_mult * N(0,1)
    index: int = 0      # offsets the seeds so workloads draw different numbers

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float16

    def flops(self) -> float:
        """4*B*H*N^2*d, halved when causal (the metric's own formula)."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def describe(self) -> dict:
        return {"workload": self.name, "B": self.B, "H": self.H, "N": self.N, "d": self.d,
                "dtype": self.dtype, "causal": self.causal, "k_mult": self.k_mult,
                "scale": "1/sqrt(d)"}


# The attention shapes the pages' target is stated on: a tiny single-tile
# case, a d=64 batch, the d=128 N=4096 batch (both masks), a long causal
# sequence with few heads, and a large fp16 batch with peaked rows.
WORKLOADS = {
    "tiny_b1h1n128d64": Workload("tiny_b1h1n128d64", 1, 1, 128, 64, "bf16", False, index=0),
    "b4h16n1024d64": Workload("b4h16n1024d64", 4, 16, 1024, 64, "bf16", False, index=1),
    "b4h16n1024d64_causal": Workload("b4h16n1024d64_causal", 4, 16, 1024, 64, "bf16", True,
                                     index=1),
    "b8h16n4096d128": Workload("b8h16n4096d128", 8, 16, 4096, 128, "bf16", False, index=2),
    "b8h16n4096d128_causal": Workload("b8h16n4096d128_causal", 8, 16, 4096, 128, "bf16", True,
                                      index=2),
    "b1h32n16384d128_causal": Workload("b1h32n16384d128_causal", 1, 32, 16384, 128, "bf16",
                                       True, index=3),
    "b16h32n8192d128_fp16_peaked": Workload("b16h32n8192d128_fp16_peaked", 16, 32, 8192, 128,
                                            "fp16", False, k_mult=4.0, index=4),
    # the same per-head shape and values with 1/8 of the heads (0.5 GiB on the
    # device): a case small enough for a full profiler capture
    "b2h32n8192d128_fp16_peaked": Workload("b2h32n8192d128_fp16_peaked", 2, 32, 8192, 128,
                                           "fp16", False, k_mult=4.0, index=4),
    # d=64 with long items (32 K/V blocks per Q tile), both masks: the
    # head dim's steady state rather than its launch and ramp; not target shapes
    "b4h32n4096d64": Workload("b4h32n4096d64", 4, 32, 4096, 64, "bf16", False, index=6),
    "b4h32n4096d64_causal": Workload("b4h32n4096d64_causal", 4, 32, 4096, 64, "bf16", True,
                                     index=6),
    # a large causal batch (K and V: 2 GiB, far beyond L2): the case the
    # head-by-head causal order is for; not one of the target shapes
    "b16h32n8192d128_causal": Workload("b16h32n8192d128_causal", 16, 32, 8192, 128, "bf16",
                                       True, index=5),
}

BASE_SEED = 0


def make_qkv(B: int, H: int, N: int, d: int, dtype=torch.bfloat16, seed: int = 0,
             k_mult: float = 1.0, q_zero: bool = False):
    """Q, K, V as contiguous CPU tensors [B, H, N, d] of `dtype`.

    Q, K and V come from three generators seeded seed+0, seed+1, seed+2.
    """
    shape = (B, H, N, d)
    out = []
    for t in range(3):
        g = torch.Generator(device="cpu")
        g.manual_seed(seed + t)
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if t == 1 and k_mult != 1.0:
            x.mul_(k_mult)
        if t == 0 and q_zero:
            x.zero_()
        out.append(x.to(dtype).contiguous())
    return tuple(out)


def make_workload_inputs(w: Workload):
    return make_qkv(w.B, w.H, w.N, w.d, w.torch_dtype, seed=BASE_SEED + 10 * w.index,
                    k_mult=w.k_mult)


def sample_rows(B: int, H: int, N: int, n_random: int = 32, seed: int = 1234,
                heads=None) -> np.ndarray:
    """Flat row ids (b*H + h)*N + i to check on large workloads.

    For each selected head: the first and last rows, rows either side of the
    128-row tile boundaries at the start, middle and end of the sequence,
    plus `n_random` seeded random rows.  `heads` limits which (b*H + h)
    heads are sampled (all by default).
    """
    fixed = [0, 1, 127, 128, 255, N // 2, N - 129, N - 128, N - 1]
    fixed = sorted({i for i in fixed if 0 <= i < N})
    rng = np.random.default_rng(seed)
    heads = range(B * H) if heads is None else heads
    rows = []
    for bh in heads:
        rnd = rng.integers(0, N, size=n_random) if n_random else []
        for i in sorted(set(fixed) | {int(x) for x in rnd}):
            rows.append(bh * N + i)
    return np.asarray(rows, dtype=np.int64)
