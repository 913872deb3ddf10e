"""Element-wise acceptance bounds for the CUDA path against the oracle.

C_ref and S = sum_k |a_ik·b_kj| come from the oracle (fp64). The bounds are
the ones the workload definitions state:
  bf16 in, fp32 out:  |C - C_ref| <= 1e-4·S + 1e-6
  bf16 in, bf16 out:  |C - C_ref| <= 1e-4·S + 1e-6 + 2^-8·|C_ref|
  TF32 in, fp32 out:  |C - C_ref| <= 5e-3·S
  int8 in, int32 out: C == C_ref (bit-exact)
and, for the CUDA-core fp32 GEMM (fp32 FMA chain in k order from 0, one
rounding per step; the classical bound for recursive summation with fused
multiply-adds, u = 2^-24):
  fp32 in, fp32 out:  |C - C_ref| <= K·u / (1 - K·u) · S
"""
from __future__ import annotations

import numpy as np


def bound_for(kind: str, ref: np.ndarray, S: np.ndarray, K: int | None = None) -> np.ndarray:
    if kind == "bf16_f32":
        return 1e-4 * S + 1e-6
    if kind == "bf16_bf16":
        return 1e-4 * S + 1e-6 + 2.0 ** -8 * np.abs(ref)
    if kind == "tf32":
        return 5e-3 * S
    if kind == "f32":
        u = 2.0 ** -24
        return (K * u / (1.0 - K * u)) * S
    raise ValueError(kind)


def assert_within(kind: str, got: np.ndarray, ref: np.ndarray, S: np.ndarray, what: str = "",
                  K: int | None = None) -> float:
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite outputs"
    b = bound_for(kind, ref, S, K)
    err = np.abs(got - ref)
    ratio = err / b
    worst = np.unravel_index(int(np.argmax(ratio)), ratio.shape)
    nbad = int((err > b).sum())
    assert nbad == 0, (f"{what}: {nbad} of {err.size} elements outside the {kind} bound; worst at {worst}: "
                       f"got {got[worst]!r} ref {ref[worst]!r} bound {b[worst]!r}")
    return float(ratio.max())


def assert_exact(got: np.ndarray, ref: np.ndarray, what: str = "") -> None:
    got = np.asarray(got).astype(np.int64)
    assert got.shape == ref.shape
    bad = got != ref
    if bad.any():
        idx = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} mismatches; first at {idx}: got {got[idx]} ref {ref[idx]}")
