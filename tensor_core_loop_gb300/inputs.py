"""Seeded synthetic inputs shared by the CUDA path, the oracle, the tests and the benchmark.

This module only draws random numbers and lays them out in memory; it holds
none of the product's arithmetic. Every input is generated on the CPU with a
``torch.Generator`` seeded explicitly, A drawn before B from the same
generator, so the oracle and the GPU receive the identical bytes.

Value distributions follow the workload definitions the library is measured
on:
  * bf16 GEMM: entries uniform in [-1, 1) drawn as fp32, then rounded to bf16
    (round-to-nearest-even; a value may round to exactly +1.0).
  * int8 GEMM: integers uniform in [-128, 127], both ends included.
  * TF32 GEMM: fp32 entries from N(0, 1), passed to the tensor cores as fp32.

A leading dimension larger than the row width pads every row with a fixed
sentinel pattern, so a kernel that reads or writes past the logical width is
caught by the tests.
"""
from __future__ import annotations

import torch

PAD_BF16_BITS = 0x7FC1      # a quiet-NaN bf16 pattern: poisons any product it reaches
PAD_F32 = float("nan")
PAD_S8 = 0x55               # distinct from most random rows; int8 has no NaN


def _padded(t: torch.Tensor, ld: int | None, fill) -> torch.Tensor:
    """Return a row-major view of ``t`` whose rows are ``ld`` elements apart."""
    rows, cols = t.shape
    if ld is None or ld == cols:
        return t.contiguous()
    if ld < cols:
        raise ValueError("leading dimension smaller than the row width")
    buf = torch.empty((rows, ld), dtype=t.dtype)
    if t.dtype == torch.bfloat16:
        buf.view(torch.int16).fill_(fill)
    else:
        buf.fill_(fill)
    buf[:, :cols] = t
    return buf[:, :cols]


def uniform_bf16(gen: torch.Generator, rows: int, cols: int) -> torch.Tensor:
    x = torch.rand((rows, cols), generator=gen, dtype=torch.float32)
    return (x * 2.0 - 1.0).to(torch.bfloat16)


def bf16_pair(M: int, N: int, K: int, seed: int = 0, lda: int | None = None, ldb: int | None = None):
    """A (M×K) and B (K×N), bf16, uniform [-1, 1), row-major on the CPU."""
    g = torch.Generator().manual_seed(seed)
    a = uniform_bf16(g, M, K)
    b = uniform_bf16(g, K, N)
    return _padded(a, lda, PAD_BF16_BITS), _padded(b, ldb, PAD_BF16_BITS)


def s8_pair(M: int, N: int, K: int, seed: int = 0, lda: int | None = None, ldb: int | None = None):
    """A (M×K) and B (K×N), int8, uniform over [-128, 127]."""
    g = torch.Generator().manual_seed(seed)
    a = torch.randint(-128, 128, (M, K), generator=g, dtype=torch.int8)
    b = torch.randint(-128, 128, (K, N), generator=g, dtype=torch.int8)
    return _padded(a, lda, PAD_S8), _padded(b, ldb, PAD_S8)


def tf32_pair(M: int, N: int, K: int, seed: int = 0, lda: int | None = None, ldb: int | None = None):
    """A (M×K) and B (K×N), fp32 from N(0, 1)."""
    g = torch.Generator().manual_seed(seed)
    a = torch.randn((M, K), generator=g, dtype=torch.float32)
    b = torch.randn((K, N), generator=g, dtype=torch.float32)
    return _padded(a, lda, PAD_F32), _padded(b, ldb, PAD_F32)


def bf16_bits(t: torch.Tensor):
    """The uint16 bit patterns of a bf16 CPU tensor, as a numpy view with the same strides."""
    return t.view(torch.int16).numpy().view("uint16")
