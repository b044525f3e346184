"""Seeded synthetic inputs for the FP8 cast-transpose path.

This module only draws random numbers: it holds none of the cast, transpose,
amax, dbias or scale-update arithmetic.  The tests feed the same tensors to
the CUDA library and to the CPU oracle, and the benchmark uses the same
recipes.  Every generator draws in fp32 with a ``torch.Generator`` seeded
explicitly, on the requested device, then rounds to bf16 (torch's RNE
conversion).  The same seed gives the same values only on the same device
type, so a test that compares the two paths always generates once and copies.

Workloads (all row-major bf16):
  * single matrix 256x512, N(0, 1)                          (seed 1001)
  * weight-like 4096x4096, N(0, 0.02), plus copies x*2^k for
    k = -4..3 (multiplying by a power of two is exact in bf16)  (seed 1002)
  * gradient-like dy 8192x12288, N(0, 1e-3), with round(1e-4*M*N) entries at
    seeded random positions set to +-5.0 with seeded signs     (seed 1003)
  * a list of 48 tensors cycling through 6144x12288, 12288x6144, 18432x6144
    and 6144x24576, N(0, 0.02); tensors 7 and 30 all zero, tensors 15 and 44
    rescaled in fp32 so that max|x| = 1e-30 before rounding
    (seed 1004000 + i; shard s of a layer, e.g. on rank s: + 100000 * s)
  * activation 16384x12288, 0.5 * Student-t with 3 degrees of freedom built
    as z0 / sqrt((z1^2 + z2^2 + z3^2) / 3) from four seeded normals (seed 1005)
"""
from __future__ import annotations

import torch

SEED_SINGLE = 1001
SEED_WEIGHT = 1002
SEED_GRADIENT = 1003
SEED_MULTI = 1004
SEED_ACTIVATION = 1005

MULTI_SHAPES = ((6144, 12288), (12288, 6144), (18432, 6144), (6144, 24576))
MULTI_COUNT = 48
MULTI_ZERO = (7, 30)
MULTI_TINY = (15, 44)
WEIGHT_EXPONENTS = tuple(range(-4, 4))


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(seed)
    return g


def normal_bf16(rows: int, cols: int, std: float, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    x = torch.randn(rows, cols, generator=g, device=device, dtype=torch.float32)
    return (x * std).to(torch.bfloat16)


def single_matrix(device="cpu", rows: int = 256, cols: int = 512) -> torch.Tensor:
    return normal_bf16(rows, cols, 1.0, SEED_SINGLE, device)


def weight_matrix(device="cpu", rows: int = 4096, cols: int = 4096) -> torch.Tensor:
    return normal_bf16(rows, cols, 0.02, SEED_WEIGHT, device)


def weight_rescaled(x: torch.Tensor, k: int) -> torch.Tensor:
    """x * 2^k, exact in bf16 for the value ranges used here."""
    return (x.float() * (2.0 ** k)).to(torch.bfloat16)


def gradient_matrix(device="cpu", rows: int = 8192, cols: int = 12288,
                    std: float = 1e-3, outlier_fraction: float = 1e-4,
                    outlier: float = 5.0) -> torch.Tensor:
    g = _gen(SEED_GRADIENT, device)
    x = torch.randn(rows, cols, generator=g, device=device, dtype=torch.float32) * std
    count = int(round(outlier_fraction * rows * cols))
    if count:
        pos = torch.randperm(rows * cols, generator=g, device=device)[:count]
        sign = torch.randint(0, 2, (count,), generator=g, device=device).float() * 2.0 - 1.0
        x.view(-1)[pos] = sign * outlier
    return x.to(torch.bfloat16)


def multi_shape(i: int, shapes=MULTI_SHAPES) -> tuple:
    return shapes[i % len(shapes)]


def multi_tensor(i: int, device="cpu", shapes=MULTI_SHAPES,
                 zero=MULTI_ZERO, tiny=MULTI_TINY, shard: int = 0) -> torch.Tensor:
    """Tensor i of the list; `shard` > 0 draws another shard of the same
    layer (another seed, same shape and recipe), e.g. one per rank."""
    rows, cols = multi_shape(i, shapes)
    if i in zero:
        return torch.zeros(rows, cols, dtype=torch.bfloat16, device=device)
    g = _gen(SEED_MULTI * 1000 + i + 100000 * shard, device)
    x = torch.randn(rows, cols, generator=g, device=device, dtype=torch.float32) * 0.02
    if i in tiny:
        x = x * (1e-30 / x.abs().max())
    return x.to(torch.bfloat16)


def multi_list(device="cpu", count: int = MULTI_COUNT, shapes=MULTI_SHAPES,
               zero=MULTI_ZERO, tiny=MULTI_TINY, shard: int = 0) -> list:
    return [multi_tensor(i, device, shapes, zero, tiny, shard) for i in range(count)]


def activation_matrix(device="cpu", rows: int = 16384, cols: int = 12288,
                      df_scale: float = 0.5) -> torch.Tensor:
    g = _gen(SEED_ACTIVATION, device)
    z = [torch.randn(rows, cols, generator=g, device=device, dtype=torch.float32)
         for _ in range(4)]
    t3 = z[0] / torch.sqrt((z[1] * z[1] + z[2] * z[2] + z[3] * z[3]) / 3.0)
    return (df_scale * t3).to(torch.bfloat16)


def bf16_all_patterns() -> torch.Tensor:
    """All 65536 bf16 bit patterns as a 256x256 matrix (row i holds patterns
    256*i .. 256*i+255)."""
    return torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).reshape(256, 256)
