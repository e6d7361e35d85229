"""Seeded synthetic inputs for the GEMM workloads.

This module only draws numbers: it holds none of the product's arithmetic and
serves the CUDA path and the CPU oracle alike, so that both see the same bits.

Recipe (the same for every workload):

* one ``torch.Generator('cpu')`` seeded with the workload's seed;
* A (M x K, row-major) is drawn first, then B, drawn directly in its
  column-major storage order as the N x K array ``Bcm`` (``Bcm[j, k] = B[k, j]``);
* ``uniform``: ``2 * U[0, 1) - 1`` in float32, then rounded to the input type
  with round-to-nearest-even (``Tensor.to``);
* ``normal``: ``std * N(0, 1)`` in float32, then rounded the same way;
* ``int8``: ``randint(-128, 128)``, i.e. every integer in [-128, 127];
* ``zeros``: all zero (no random draws), for measurements of how the
  values themselves affect the GPU's clock.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

# dtype pairs of the library boundary: (input element type, output element type)
DTYPE_PAIRS = {
    "f16_f32": ("f16", "f32"),
    "f16_f16": ("f16", "f16"),
    "s8_s32": ("s8", "s32"),
    "bf16_bf16": ("bf16", "bf16"),
    "bf16_f32": ("bf16", "f32"),
}

TORCH_DTYPE = {
    "f16": torch.float16,
    "bf16": torch.bfloat16,
    "s8": torch.int8,
    "f32": torch.float32,
    "s32": torch.int32,
}


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dtype: str          # key of DTYPE_PAIRS
    dist: str           # "uniform", "normal" or "int8"
    scale: float        # std for "normal"; unused otherwise
    seed: int

    @property
    def in_type(self) -> str:
        return DTYPE_PAIRS[self.dtype][0]

    @property
    def out_type(self) -> str:
        return DTYPE_PAIRS[self.dtype][1]

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


# The five workloads of the method's measurements, named by what they are.
WORKLOADS = {
    w.name: w
    for w in (
        Workload("f16_256x256x256_f32out", 256, 256, 256, "f16_f32", "uniform", 1.0, 1),
        Workload("f16_4096x4096x4096_f16out", 4096, 4096, 4096, "f16_f16", "uniform", 1.0, 2),
        Workload("s8_4096x4096x4096_s32out", 4096, 4096, 4096, "s8_s32", "int8", 1.0, 3),
        Workload("bf16_skinny_64x8192x8192_bf16out", 64, 8192, 8192, "bf16_bf16", "normal", 1.0, 4),
        Workload("bf16_8192x8192x16384_f32out", 8192, 8192, 16384, "bf16_f32", "normal", 0.5, 5),
    )
}
WORKLOAD_ORDER = list(WORKLOADS)


def _draw(g: torch.Generator, shape, in_type: str, dist: str, scale: float) -> torch.Tensor:
    if dist == "int8":
        if in_type != "s8":
            raise ValueError("int8 draws need an s8 input type")
        return torch.randint(-128, 128, shape, generator=g, dtype=torch.int8)
    if dist == "zeros":
        return torch.zeros(shape, dtype=TORCH_DTYPE[in_type])
    if dist == "uniform":
        x = torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    elif dist == "normal":
        x = torch.randn(shape, generator=g, dtype=torch.float32) * scale
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return x.to(TORCH_DTYPE[in_type])


def make_inputs(M: int, N: int, K: int, in_type: str, dist: str, seed: int,
                scale: float = 1.0):
    """Returns (A, Bcm) as contiguous CPU tensors of the input type."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    A = _draw(g, (M, K), in_type, dist, scale).contiguous()
    Bcm = _draw(g, (N, K), in_type, dist, scale).contiguous()
    return A, Bcm


def workload_inputs(w: Workload):
    return make_inputs(w.M, w.N, w.K, w.in_type, w.dist, w.seed, w.scale)
