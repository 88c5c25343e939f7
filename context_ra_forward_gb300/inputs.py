"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module holds no attention arithmetic: it only draws N(0, 1) tensors with a
seeded CPU generator and rounds them to the storage dtype, and it spells out the
ALiBi slope vector that a caller passes in (the head-slope formula of
"长上下文技术综述" §2.1.2, ALiBi: slope of head i = 2^(-8 i / H), i = 1..H).

Every GPU test and the oracle read the same rounded values: bf16 inputs are
generated in fp32, rounded to bf16 (round-to-nearest-even) and then handed to
the oracle upcast to fp64, so both sides see bit-identical inputs.
"""
from __future__ import annotations

import dataclasses

import torch

# Seed offsets per tensor; a workload's seed is added to them.
SEED_Q, SEED_K, SEED_V, SEED_DO = 1000, 2000, 3000, 4000


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention problem: sizes, dtype and the sequence layout."""

    name: str
    B: int
    H: int
    S: int
    D: int
    dtype: str          # "f32" or "bf16"
    causal: bool
    alibi: bool
    N: int              # number of virtual ring shards
    layout: str         # "contiguous" or "zigzag"
    backward: bool = False
    seed: int = 0

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


# The five workloads of the long-context regime the pages discuss
# (256k-token training, 64K sequence-parallel runs, 500k-token OOM case).
WORKLOADS = {
    "C1": Workload("C1", 1, 2, 1024, 64, "f32", True, False, 4, "zigzag", False, 1),
    "C2": Workload("C2", 1, 32, 32768, 128, "bf16", False, False, 8, "contiguous", False, 2),
    "C3": Workload("C3", 1, 32, 65536, 128, "bf16", True, False, 8, "zigzag", False, 3),
    "C4": Workload("C4", 1, 32, 65536, 128, "bf16", True, True, 8, "zigzag", False, 4),
    "C5": Workload("C5", 1, 16, 262144, 128, "bf16", True, False, 16, "zigzag", True, 5),
    # the same causal workloads with the token-strided assignment the Zig-Zag
    # section prints ("GPU 0 gets tokens [0, 4, 8...]")
    "C3S": Workload("C3S", 1, 32, 65536, 128, "bf16", True, False, 8, "strided", False, 3),
    # C3 with the contiguous split, the unbalanced layout the zig-zag one corrects
    "C3C": Workload("C3C", 1, 32, 65536, 128, "bf16", True, False, 8, "contiguous", False, 3),
    "C5S": Workload("C5S", 1, 16, 262144, 128, "bf16", True, False, 16, "strided", True, 5),
}


def randn(shape, seed: int, dtype: torch.dtype) -> torch.Tensor:
    """N(0,1) drawn in fp32 on the CPU with a seeded generator, then rounded to dtype."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    return x.to(dtype)


def make_inputs(w: Workload, B=None, H=None, S=None, D=None, seed=None):
    """Q, K, V (and dO when the workload has a backward) in ORIGINAL sequence order,
    shape [B, H, S, D], on the CPU in the workload's dtype.  Sizes may be overridden
    to build a smaller case of the same recipe."""
    B = w.B if B is None else B
    H = w.H if H is None else H
    S = w.S if S is None else S
    D = w.D if D is None else D
    seed = w.seed if seed is None else seed
    dt = w.torch_dtype
    shape = (B, H, S, D)
    out = {
        "q": randn(shape, SEED_Q + seed, dt),
        "k": randn(shape, SEED_K + seed, dt),
        "v": randn(shape, SEED_V + seed, dt),
    }
    if w.backward:
        out["do"] = randn(shape, SEED_DO + seed, dt)
    return out


def alibi_slopes(H: int) -> torch.Tensor:
    """The per-head ALiBi slope vector, fp32: head index hh (0-based) gets
    2^(-8 (hh+1) / H) ("长上下文技术综述" §2.1.2, slopes listed for i = 1..num_heads)."""
    return torch.tensor([2.0 ** (-8.0 * i / H) for i in range(1, H + 1)], dtype=torch.float32)


def to_f64_numpy(t: torch.Tensor):
    """Exact upcast of a CPU tensor (fp32 or bf16) to a float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).numpy()


E4M3_MAX = 448.0  # largest finite e4m3 value


def quantize_e4m3(x: torch.Tensor):
    """Per-tensor e4m3 quantisation of a CPU tensor: scale = max|x| / 448, returns
    (x8 as torch.float8_e4m3fn, scale as a Python float).  The value an element
    stands for is float(x8) * scale."""
    amax = float(x.float().abs().max())
    scale = amax / E4M3_MAX if amax > 0 else 1.0
    x8 = (x.float() / scale).to(torch.float8_e4m3fn)
    return x8, scale


def dequantize_f64(x8: torch.Tensor, scale: float):
    """Exact value of an e4m3 tensor times its scale, as float64 numpy."""
    return x8.to(torch.float64).numpy() * scale
