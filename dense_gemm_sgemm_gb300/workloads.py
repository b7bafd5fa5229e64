"""Seeded synthetic workloads for the GEMM library (inputs only, no GEMM arithmetic).

Each workload names a shape, the operand layout, alpha/beta and a value recipe.  Values
are drawn on the CPU with ``torch.Generator().manual_seed(seed)`` in the fixed order A,
then B, then C_in, so the same seed always gives the same bytes on any machine.  fp16 and
bf16 operands are drawn in fp32 and rounded once (``Tensor.half()`` /
``Tensor.to(torch.bfloat16)``, round to nearest even); consumers receive those 16-bit
values and never see the fp32 draw.

The shapes follow the pages this library is built from: square fp32 problems of the
copecc "GEMM" page benchmark (section "完整优化 Kernel 源码引用"), the ragged
1001 x 513 x 777 problem of the yekq.top "LeetGPU 第二题" page (it exercises the tails of
every tile), the M = N sweep with K = 1024 of the ssxxe.cn page (section "1.2"), the fp16
square problems of the dandandamowang.xyz "GEMM优化（二）" page, and a linear-layer shaped
fp16 problem with B stored N x K.  These synthetic inputs stand in for the pages' own random
inputs and for the public LeetGPU challenge, whose test cases are not reproduced here.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

SWEEP_MN = (128, 256, 512, 1024, 2048, 4096, 8192, 16384)
HGEMM_SQUARE = (2048, 4096, 8192)


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str  # "f32" (SGEMM), "f16" or "bf16" (16-bit inputs, fp32 accumulate and output)
    M: int
    N: int
    K: int
    opA: str = "N"
    opB: str = "N"
    alpha: float = 1.0
    beta: float = 0.0
    seed: int = 0
    dist_a: str = "u11"  # u11 = uniform[-1,1]; int4 = integers in [-4,4]; n01 = N(0,1)
    dist_b: str = "u11"  # n002 = N(0, 0.02)
    dist_c: str = "u11"  # n01_1 = N(0, 0.1)
    pad: tuple = field(default=(0, 0, 0))  # extra elements per row of A, B, C storage

    @property
    def a_shape(self):  # stored shape of A (rows, cols)
        return (self.M, self.K) if self.opA == "N" else (self.K, self.M)

    @property
    def b_shape(self):
        return (self.K, self.N) if self.opB == "N" else (self.N, self.K)

    @property
    def lda(self):
        return self.a_shape[1] + self.pad[0]

    @property
    def ldb(self):
        return self.b_shape[1] + self.pad[1]

    @property
    def ldc(self):
        return self.N + self.pad[2]

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def in_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def algorithmic_bytes(self) -> int:
        """Compulsory traffic: each input read once, C written once, C read when beta != 0."""
        c = 4 * self.M * self.N * (2 if self.beta != 0.0 else 1)
        return self.in_bytes * (self.M * self.K + self.K * self.N) + c


def _draw(g: torch.Generator, rows: int, cols: int, dist: str) -> torch.Tensor:
    shape = (rows, cols)
    if dist == "u11":
        return torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    if dist == "int4":
        return torch.randint(-4, 5, shape, generator=g, dtype=torch.int64).to(torch.float32)
    if dist == "n01":
        return torch.randn(shape, generator=g, dtype=torch.float32)
    if dist == "n002":
        return torch.randn(shape, generator=g, dtype=torch.float32) * 0.02
    if dist == "n01_1":
        return torch.randn(shape, generator=g, dtype=torch.float32) * 0.1
    raise ValueError(f"unknown distribution {dist!r}")


def _padded(x: torch.Tensor, pad: int, fill=float("nan")) -> torch.Tensor:
    if pad == 0:
        return x.contiguous()
    out = torch.full((x.shape[0], x.shape[1] + pad), fill, dtype=x.dtype)
    out[:, : x.shape[1]] = x
    return out


def make_inputs(w: Workload) -> dict:
    """A, B (stored shapes, padded rows if ``w.pad``) and C_in as CPU tensors.

    C_in is always produced (it is the initial content of C); when beta == 0 it is filled
    with NaN, which a correct implementation never reads.
    """
    g = torch.Generator().manual_seed(w.seed)
    a = _draw(g, *w.a_shape, w.dist_a)
    b = _draw(g, *w.b_shape, w.dist_b)
    if w.beta != 0.0:
        c = _draw(g, w.M, w.N, w.dist_c)
    else:
        c = torch.full((w.M, w.N), float("nan"), dtype=torch.float32)
    if w.dtype == "f16":
        a, b = a.half(), b.half()
    elif w.dtype == "bf16":
        a, b = a.to(torch.bfloat16), b.to(torch.bfloat16)
    return {
        "A": _padded(a, w.pad[0]),
        "B": _padded(b, w.pad[1]),
        "C": _padded(c, w.pad[2]),
    }


def sgemm_256(integer: bool = False) -> Workload:
    d = "int4" if integer else "u11"
    return Workload("sgemm_256cube" + ("_int" if integer else ""), "f32", 256, 256, 256,
                    seed=0, dist_a=d, dist_b=d)


def sgemm_ragged() -> Workload:
    return Workload("sgemm_ragged_1001x777x513", "f32", 1001, 777, 513, alpha=1.5,
                    beta=-0.5, seed=1)


def sgemm_sweep(mn: int, K: int = 1024) -> Workload:
    return Workload(f"sgemm_sweep_{mn}x{mn}x{K}", "f32", mn, mn, K, seed=2, dist_a="n01",
                    dist_b="n01")


def sgemm_cube(n: int = 4096) -> Workload:
    return Workload(f"sgemm_{n}cube", "f32", n, n, n, seed=2, dist_a="n01", dist_b="n01")


def hgemm_square(n: int, integer: bool = False, K: int | None = None) -> Workload:
    d = "int4" if integer else "u11"
    k = n if K is None else K
    return Workload(f"hgemm_{n}x{n}x{k}" + ("_int" if integer else ""), "f16", n, n, k,
                    seed=3, dist_a=d, dist_b=d)


def linear_fp16() -> Workload:
    return Workload("linear_16384x4096x4096_opBT", "f16", 16384, 4096, 4096, opB="T",
                    alpha=1.0, beta=1.0, seed=4, dist_a="n01", dist_b="n002",
                    dist_c="n01_1")


def all_named() -> list[Workload]:
    """Every workload the parity tests and the benchmark use."""
    out = [sgemm_256(), sgemm_256(True), sgemm_ragged()]
    out += [sgemm_sweep(mn) for mn in SWEEP_MN]
    out += [sgemm_cube(4096)]
    out += [hgemm_square(n) for n in HGEMM_SQUARE]
    out += [hgemm_square(2048, integer=True, K=1024), linear_fp16()]
    return out


def by_name(name: str) -> Workload:
    for w in all_named():
        if w.name == name:
            return w
    raise KeyError(name)
