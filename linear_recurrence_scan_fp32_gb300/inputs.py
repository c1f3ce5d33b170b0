"""Seeded synthetic inputs for the linear-recurrence scan.

This module only draws random numbers.  It holds none of the recurrence's
arithmetic, so both the CUDA path's tests and the CPU oracle's tests can use
it without sharing any part of the method.

Every tensor is fp32, contiguous, row-major (B, L, D) with D contiguous, drawn
on the CPU from ``torch.Generator().manual_seed(seed)`` in the order a, then b.

The five named workloads follow the shapes and distributions of the
linear-recurrence problem on the POPCORNBENCH traces "Kimi-K2.6 l1_p9" and
"FW-GLM-5-1 l1_p9" (problem statement: B=32, L=4096, D=256), widened to a
tiny case, a long-sequence case, a gated wide case and a many-short-scans case.
"""
from __future__ import annotations

import dataclasses
from typing import Callable, Dict, Tuple

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    L: int
    D: int
    seed: int
    a_dist: str   # see _A_DISTS
    b_dist: str   # see _B_DISTS
    about: str

    @property
    def shape(self) -> Tuple[int, int, int]:
        return (self.B, self.L, self.D)

    @property
    def numel(self) -> int:
        return self.B * self.L * self.D

    @property
    def algorithmic_bytes(self) -> int:
        # read a, read b, write h: 4 bytes each, once.
        return 12 * self.numel


def _uniform(lo: float, hi: float) -> Callable:
    def draw(shape, g):
        return lo + (hi - lo) * torch.rand(shape, generator=g, dtype=torch.float32)
    return draw


def _normal(std: float) -> Callable:
    def draw(shape, g):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        return x if std == 1.0 else x * std
    return draw


def _sigmoid_normal(shape, g):
    # gate a = sigmoid(z), z ~ Normal(0, 1); torch's CPU sigmoid, input generation only
    return torch.sigmoid(torch.randn(shape, generator=g, dtype=torch.float32))


def _const(v: float) -> Callable:
    def draw(shape, g):
        return torch.full(shape, v, dtype=torch.float32)
    return draw


def _int_range(lo: int, hi_excl: int) -> Callable:
    # integer-valued fp32; randint never yields -0.0
    def draw(shape, g):
        return torch.randint(lo, hi_excl, shape, generator=g, dtype=torch.int32).to(torch.float32)
    return draw


_A_DISTS: Dict[str, Callable] = {
    "u[0,1)": _uniform(0.0, 1.0),
    "u[0.5,1)": _uniform(0.5, 1.0),
    "u[0.9,1)": _uniform(0.9, 1.0),
    "sigmoid(n(0,1))": _sigmoid_normal,
    "ones": _const(1.0),
    "zeros": _const(0.0),
}

_B_DISTS: Dict[str, Callable] = {
    "n(0,1)": _normal(1.0),
    "n(0,0.5)": _normal(0.5),
    "int[-8,8]": _int_range(-8, 9),
    "u[0,1)": _uniform(0.0, 1.0),
}


WORKLOADS: Dict[str, Workload] = {w.name: w for w in [
    Workload("tiny", 1, 64, 32, 0, "u[0.5,1)", "n(0,1)",
             "tiny scan (1,64,32), a~U[0.5,1), b~N(0,1)"),
    Workload("pages", 32, 4096, 256, 1, "u[0,1)", "n(0,1)",
             "the pages' shape (32,4096,256), a~U[0,1), b~N(0,1)"),
    Workload("long", 1, 1048576, 64, 2, "u[0.9,1)", "n(0,1)",
             "long sequence, few channels (1,1048576,64), a~U[0.9,1), b~N(0,1)"),
    Workload("gated", 64, 2048, 1024, 3, "sigmoid(n(0,1))", "n(0,0.5)",
             "gated wide scan (64,2048,1024), a=sigmoid(z), b~N(0,0.5)"),
    Workload("short", 256, 128, 4096, 4, "u[0,1)", "n(0,1)",
             "many short scans (256,128,4096), a~U[0,1), b~N(0,1)"),
    # long sequences over more channels: 32 slices of 32 channels, the chain mode's shape
    Workload("long32", 4, 65536, 256, 5, "u[0.9,1)", "n(0,1)",
             "long sequences, 32 channel slices (4,65536,256), a~U[0.9,1), b~N(0,1)"),
    # closed-form variants on the many-short-scans shape
    Workload("short_ones", 256, 128, 4096, 4, "ones", "n(0,1)", "a=1: inclusive prefix sum of b"),
    Workload("short_zeros", 256, 128, 4096, 4, "zeros", "n(0,1)", "a=0: h=b"),
    Workload("short_ones_int", 256, 128, 4096, 4, "ones", "int[-8,8]",
             "a=1, integer b: prefix sum, exact in fp32"),
    Workload("short_zeros_int", 256, 128, 4096, 4, "zeros", "int[-8,8]", "a=0, integer b: h=b exactly"),
]}

# The five configurations, in order: tiny, pages' shape, long, gated, short.
CONFIG_ORDER = ("tiny", "pages", "long", "gated", "short")


def generate(B: int, L: int, D: int, seed: int, a_dist: str = "u[0,1)",
             b_dist: str = "n(0,1)") -> Tuple[torch.Tensor, torch.Tensor]:
    """Draw (a, b), each fp32 contiguous (B, L, D) on the CPU, a first then b."""
    if a_dist not in _A_DISTS:
        raise ValueError(f"unknown a distribution {a_dist!r}")
    if b_dist not in _B_DISTS:
        raise ValueError(f"unknown b distribution {b_dist!r}")
    g = torch.Generator().manual_seed(seed)
    shape = (B, L, D)
    a = _A_DISTS[a_dist](shape, g).contiguous()
    b = _B_DISTS[b_dist](shape, g).contiguous()
    return a, b


def generate_workload(w: Workload | str) -> Tuple[torch.Tensor, torch.Tensor]:
    if isinstance(w, str):
        w = WORKLOADS[w]
    return generate(w.B, w.L, w.D, w.seed, w.a_dist, w.b_dist)


STORAGE16 = {"bf16": torch.bfloat16, "f16": torch.float16}


def to_storage16(x: torch.Tensor, kind: str) -> torch.Tensor:
    """The draws stored in 16 bits ("bf16" or "f16"), by torch's conversion: the
    stored words are the test input itself, given to both the CUDA path and the
    oracle (which decodes them by its own definition of the format)."""
    return x.to(STORAGE16[kind]).contiguous()


def to_bdl(x: torch.Tensor) -> torch.Tensor:
    """A (B, L, D) draw laid out (B, D, L), time innermost: the same values, moved."""
    return x.transpose(1, 2).contiguous()
