"""Seeded synthetic operands and the named workloads.

This module is shared by the tests, the benchmark and the oracle's checks.
It holds no MatMul arithmetic: it only draws values and casts them.

Input recipe (one reading, applied everywhere):

* a fresh ``torch.Generator('cpu')`` seeded with the workload's seed per
  product; A is drawn first, then B;
* FLOAT, FLOAT16 and BFLOAT16 operands are drawn as float32
  (``uniform`` = ``rand * (hi - lo) + lo``, ``normal`` = ``randn * sigma``,
  ``int`` = ``randint(lo, hi + 1)``) and cast to the storage type with
  round-to-nearest-even; DOUBLE operands are drawn directly in float64;
* the cast CPU tensors are the single source of truth: the device copy is
  made from them, and the oracle reads them.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import torch

TORCH_DTYPES = {
    "float32": torch.float32,
    "float64": torch.float64,
    "float16": torch.float16,
    "bfloat16": torch.bfloat16,
    "float8_e4m3fn": torch.float8_e4m3fn,
    "float8_e5m2": torch.float8_e5m2,
    "float8_e4m3fnuz": torch.float8_e4m3fnuz,
    "float8_e5m2fnuz": torch.float8_e5m2fnuz,
}

# ONNX TensorProto element type codes, as used by the C ABI.
ONNX_CODES = {"float32": 1, "float16": 10, "float64": 11, "bfloat16": 16,
              "float8_e4m3fn": 17, "float8_e4m3fnuz": 18, "float8_e5m2": 19,
              "float8_e5m2fnuz": 20}

ELEMENT_BYTES = {"float32": 4, "float64": 8, "float16": 2, "bfloat16": 2,
                 "float8_e4m3fn": 1, "float8_e5m2": 1, "float8_e4m3fnuz": 1, "float8_e5m2fnuz": 1}

FP8_DTYPES = ("float8_e4m3fn", "float8_e5m2", "float8_e4m3fnuz", "float8_e5m2fnuz")


def output_dtype(dtype: str) -> str:
    """Element type of a product's output: FLOAT for the 8-bit float
    operand types (float32 accumulation, no narrowing), the operand type
    otherwise."""
    return "float32" if dtype in FP8_DTYPES else dtype


@dataclass(frozen=True)
class Dist:
    """A value distribution: kind in {"uniform", "normal", "int"}."""
    kind: str
    lo: float = -1.0
    hi: float = 1.0
    sigma: float = 1.0

    def label(self) -> str:
        if self.kind == "uniform":
            return "U[%g,%g]" % (self.lo, self.hi)
        if self.kind == "normal":
            return "N(0,%g)" % self.sigma
        return "int{%d..%d}" % (int(self.lo), int(self.hi))


UNIFORM = Dist("uniform", -1.0, 1.0)
SMALL_INT = Dist("int", -3, 3)


def normal(sigma: float) -> Dist:
    return Dist("normal", sigma=sigma)


def draw(shape, dist: Dist, dtype: str, gen: torch.Generator) -> torch.Tensor:
    """One operand: drawn on the CPU from ``gen`` and cast to ``dtype``."""
    shape = tuple(int(d) for d in shape)
    wide = torch.float64 if dtype == "float64" else torch.float32
    if dist.kind == "uniform":
        t = torch.rand(shape, generator=gen, dtype=wide) * (dist.hi - dist.lo) + dist.lo
    elif dist.kind == "normal":
        t = torch.randn(shape, generator=gen, dtype=wide) * dist.sigma
    elif dist.kind == "int":
        t = torch.randint(int(dist.lo), int(dist.hi) + 1, shape, generator=gen).to(wide)
    else:
        raise ValueError(dist.kind)
    return t.to(TORCH_DTYPES[dtype]).contiguous()


def operands(a_shape, b_shape, dtype: str, dist_a: Dist, dist_b: Dist,
             seed: int) -> Tuple[torch.Tensor, torch.Tensor]:
    """(A, B) on the CPU for one product, A drawn first."""
    gen = torch.Generator("cpu")
    gen.manual_seed(int(seed))
    a = draw(a_shape, dist_a, dtype, gen)
    b = draw(b_shape, dist_b, dtype, gen)
    return a, b


def chain_operands(shapes: List[Tuple[int, int]], dtype: str, dist: Dist,
                   seed: int) -> List[torch.Tensor]:
    """Inputs of a chain of products: the first activation, then each weight,
    drawn in that order from one generator."""
    gen = torch.Generator("cpu")
    gen.manual_seed(int(seed))
    return [draw(s, dist, dtype, gen) for s in shapes]


def to_numpy_storage(t: torch.Tensor):
    """A CPU tensor as the numpy array the oracle takes: float32 / float64
    values, uint16 bit patterns for the 16-bit types, uint8 bit patterns for
    the 8-bit float types."""
    t = t.detach().cpu().contiguous()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy().view("uint16")
    if t.dtype in (torch.float8_e4m3fn, torch.float8_e5m2, torch.float8_e4m3fnuz,
                   torch.float8_e5m2fnuz):
        return t.view(torch.uint8).numpy()
    return t.numpy()


def from_numpy_storage(arr, dtype: str) -> torch.Tensor:
    """Inverse of ``to_numpy_storage``."""
    import numpy as np
    if dtype in ("float16", "bfloat16"):
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16).copy()).view(
            TORCH_DTYPES[dtype])
    if dtype in FP8_DTYPES:
        return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.uint8).copy()).view(
            TORCH_DTYPES[dtype])
    return torch.from_numpy(np.ascontiguousarray(arr).copy())


# --------------------------------------------------------------------------
# named workloads

@dataclass(frozen=True)
class Product:
    """One MatMul of a workload."""
    name: str
    a_shape: Tuple[int, ...]
    b_shape: Tuple[int, ...]
    dtype: str
    dist_a: Dist
    dist_b: Dist
    seed: int

    def draw(self):
        return operands(self.a_shape, self.b_shape, self.dtype, self.dist_a,
                        self.dist_b, self.seed)


@dataclass(frozen=True)
class Chain:
    """Consecutive products, each output feeding the next as its A."""
    name: str
    shapes: Tuple[Tuple[int, int], ...]   # first activation, then the weights
    dtype: str
    dist: Dist
    seed: int

    def draw(self):
        return chain_operands(list(self.shapes), self.dtype, self.dist, self.seed)


@dataclass(frozen=True)
class Workload:
    name: str
    description: str
    products: Tuple[Product, ...] = field(default_factory=tuple)
    chains: Tuple[Chain, ...] = field(default_factory=tuple)


def _fp32_small() -> Workload:
    return Workload(
        "fp32_64x128x96",
        "FP32 A[64,128] x B[128,96], U[-1,1] seed 0, and the same shapes with "
        "integers in {-3..3} for an exact check",
        products=(
            Product("uniform", (64, 128), (128, 96), "float32", UNIFORM, UNIFORM, 0),
            Product("small_int", (64, 128), (128, 96), "float32", SMALL_INT, SMALL_INT, 0),
        ))


def _fp32_broadcast() -> Workload:
    u = UNIFORM
    return Workload(
        "fp32_broadcast_batch",
        "FP32 A[8,1,128,256] x B[1,4,256,64] (zero batch strides on both sides), "
        "rank-one a[256] x B[4,256,64] and A[4,32,256] x b[256], and an empty "
        "batch A[0,16,32] x B[32,8]; U[-1,1] seed 1",
        products=(
            Product("broadcast", (8, 1, 128, 256), (1, 4, 256, 64), "float32", u, u, 1),
            Product("vector_a", (256,), (4, 256, 64), "float32", u, u, 1),
            Product("vector_b", (4, 32, 256), (256,), "float32", u, u, 1),
            Product("empty_batch", (0, 16, 32), (32, 8), "float32", u, u, 1),
        ))


def _bf16_projection() -> Workload:
    a, w = normal(1.0), normal(0.02)
    return Workload(
        "bf16_transformer_projection",
        "BF16 activations A ~ N(0,1) x weights B ~ N(0,0.02), seed 2: "
        "[8,2048,4096]x[4096,4096], [8,2048,4096]x[4096,14336], "
        "[8,2048,14336]x[14336,4096]; FP32 accumulation, BF16 output",
        products=(
            Product("proj_4096x4096", (8, 2048, 4096), (4096, 4096), "bfloat16", a, w, 2),
            Product("proj_4096x14336", (8, 2048, 4096), (4096, 14336), "bfloat16", a, w, 2),
            Product("proj_14336x4096", (8, 2048, 14336), (14336, 4096), "bfloat16", a, w, 2),
        ))


def _fp8_projection() -> Workload:
    a, w = normal(1.0), normal(0.5)
    return Workload(
        "fp8_transformer_projection",
        "E4M3FN activations A ~ N(0,1) x weights B ~ N(0,0.5) (cast RNE), seed 2: "
        "[8,2048,4096]x[4096,4096], [8,2048,4096]x[4096,14336], "
        "[8,2048,14336]x[14336,4096]; float32 accumulation, FLOAT output",
        products=(
            Product("fp8_proj_4096x4096", (8, 2048, 4096), (4096, 4096), "float8_e4m3fn", a, w, 2),
            Product("fp8_proj_4096x14336", (8, 2048, 4096), (4096, 14336), "float8_e4m3fn", a, w, 2),
            Product("fp8_proj_14336x4096", (8, 2048, 14336), (14336, 4096), "float8_e4m3fn", a, w, 2),
        ))


def _fp16_corners() -> Workload:
    a, w = normal(1.0), normal(0.02)
    return Workload(
        "fp16_skinny_splitk",
        "FP16 skinny-M A[4,8192]xB[8192,28672], skinny-N A[16384,4096]xB[4096,8], "
        "tiny-output long-K A[32,131072]xB[131072,32]; activations N(0,1), "
        "weights N(0,0.02), seed 3",
        products=(
            Product("skinny_m", (4, 8192), (8192, 28672), "float16", a, w, 3),
            Product("skinny_n", (16384, 4096), (4096, 8), "float16", a, w, 3),
            Product("split_k", (32, 131072), (131072, 32), "float16", a, w, 3),
        ))


def _fp8_decode() -> Workload:
    a, w = normal(1.0), normal(0.5)
    return Workload(
        "fp8_skinny_decode",
        "E4M3FN few-row products against one large weight, A ~ N(0,1) x B ~ N(0,0.5) "
        "(cast RNE), seed 3: [1,8192], [4,8192] and [16,8192] x [8192,28672]; "
        "float32 accumulation, FLOAT output",
        products=tuple(
            Product("fp8_rows_%d" % m, (m, 8192), (8192, 28672), "float8_e4m3fn", a, w, 3)
            for m in (1, 4, 16)))


def _square_sweep(dtype: str) -> Workload:
    u = UNIFORM
    return Workload(
        "%s_square_chain" % dtype,
        "%s squares M=N=K in {1024,4096,8192} and the chain "
        "[4096,1024]x[1024,4096] -> x[4096,1024] -> x[1024,4096]; U[-1,1] seed 4" % dtype,
        products=tuple(
            Product("square_%d" % s, (s, s), (s, s), dtype, u, u, 4) for s in (1024, 4096, 8192)),
        chains=(Chain("chain", ((4096, 1024), (1024, 4096), (4096, 1024), (1024, 4096)),
                      dtype, u, 4),),
    )


def workloads():
    """All named workloads, smallest first."""
    return [_fp32_small(), _fp32_broadcast(), _bf16_projection(), _fp16_corners(),
            _square_sweep("float32"), _square_sweep("float64"), _fp8_projection(), _fp8_decode()]


def workload(name: str) -> Workload:
    for w in workloads():
        if w.name == name:
            return w
    raise KeyError(name)
