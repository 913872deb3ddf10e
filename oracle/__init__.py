"""Plain CPU oracle for C = A·B — test infrastructure, not product code.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never calls it, and it
never calls the CUDA library: the two share no code. Both sides receive the
same input bytes from the seeded generators in
``tensor_core_loop_gb300.inputs``, which hold none of the product's arithmetic.

The arithmetic lives in ``gemm_oracle.c`` (plain C, fp64 / int64 triple loop,
OpenMP over rows); this module compiles it with gcc on first use and passes
numpy arrays to it through ctypes.

Definition followed ("4.1 CUDA GEMM 算子性能优化", §1.1 and §3.1):
    C[i][j] = sum_k A[i][k] · B[k][j],   A: M×K, B: K×N, both row-major.
Inputs are decoded exactly as the tensor cores consume them: bf16 exactly,
fp32 as TF32 (truncated by default, see ``TF32_TRUNCATE``), int8 exactly; the
CUDA-core (SIMT) fp32 GEMM consumes fp32 as is, widened exactly to fp64.

Parity is pinned by the ``-m "not gpu"`` tests in ``tests/test_oracle.py``
(exhaustive decode, exact rational brute force, closed forms, invariants).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

TF32_TRUNCATE = 0
TF32_ROUND_NEAREST = 1

_STATUS = {1: "null pointer", 2: "bad dimensions", 3: "bad leading dimension", 9: "out of memory"}


def build(force: bool = False) -> str:
    """Compile gemm_oracle.c into liboracle.so (gcc, OpenMP, no fp contraction)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        L, P, I = ctypes.c_long, ctypes.c_void_p, ctypes.c_int
        for name in ("oracle_gemm_bf16", "oracle_gemm_f64"):
            fn = getattr(lib, name)
            fn.argtypes = [L, L, L, P, L, P, L, L, L, L, L, P, L, P, L]
            fn.restype = I
        lib.oracle_gemm_tf32.argtypes = [L, L, L, P, L, P, L, L, L, L, L, P, L, P, L, I]
        lib.oracle_gemm_tf32.restype = I
        lib.oracle_gemm_s8.argtypes = [L, L, L, P, L, P, L, L, L, L, L, P, L]
        lib.oracle_gemm_s8.restype = I
        lib.oracle_decode_bf16.argtypes = [P, P, L]
        lib.oracle_decode_tf32.argtypes = [P, P, L, I]
        lib.oracle_num_threads.restype = I
        lib.oracle_set_num_threads.argtypes = [I]
        lib.oracle_set_num_threads.restype = None
        _lib = lib
        return lib


def num_threads() -> int:
    """OpenMP threads the oracle uses (all host cores unless OMP_NUM_THREADS says otherwise)."""
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """OpenMP threads for the following oracle calls (timing on one core uses 1)."""
    _load().oracle_set_num_threads(int(n))


def _as_rows(x: np.ndarray, dtype) -> tuple[np.ndarray, int]:
    """Return (array, leading dimension in elements) for a 2-D row-major view."""
    if x.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {x.dtype}")
    if x.ndim != 2:
        raise ValueError("expected a 2-D array")
    if x.strides[1] != x.itemsize:
        x = np.ascontiguousarray(x)
    ld = x.strides[0] // x.itemsize if x.shape[0] > 1 else x.shape[1]
    return x, max(int(ld), x.shape[1], 1)


def _ranges(M, N, rows, cols):
    i0, i1 = (0, M) if rows is None else rows
    j0, j1 = (0, N) if cols is None else cols
    return int(i0), int(i1), int(j0), int(j1)


def _check(st):
    if st:
        raise ValueError(f"oracle rejected its arguments: {_STATUS.get(st, st)}")


def gemm_bf16(a_bits: np.ndarray, b_bits: np.ndarray, rows=None, cols=None, with_abs=True):
    """C = A·B for bf16 inputs given as uint16 bit patterns; returns (C, S) in fp64.

    ``rows=(i0, i1)`` / ``cols=(j0, j1)`` restrict the output to a block of C;
    ``S`` is sum_k |a_ik·b_kj| over the same block (None if ``with_abs`` is
    False).
    """
    a, lda = _as_rows(a_bits, np.uint16)
    b, ldb = _as_rows(b_bits, np.uint16)
    M, K = a.shape
    K2, N = b.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    i0, i1, j0, j1 = _ranges(M, N, rows, cols)
    C = np.empty((i1 - i0, j1 - j0), np.float64)
    S = np.empty_like(C) if with_abs else None
    _check(_load().oracle_gemm_bf16(M, N, K, a.ctypes.data, lda, b.ctypes.data, ldb, i0, i1, j0, j1,
                                    C.ctypes.data, max(C.shape[1], 1),
                                    S.ctypes.data if with_abs else None, max(C.shape[1], 1)))
    return C, S


def gemm_tf32(a: np.ndarray, b: np.ndarray, rows=None, cols=None, with_abs=True, mode=TF32_TRUNCATE):
    """C = A·B for fp32 inputs consumed as TF32; returns (C, S) in fp64."""
    a, lda = _as_rows(a, np.float32)
    b, ldb = _as_rows(b, np.float32)
    M, K = a.shape
    K2, N = b.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    i0, i1, j0, j1 = _ranges(M, N, rows, cols)
    C = np.empty((i1 - i0, j1 - j0), np.float64)
    S = np.empty_like(C) if with_abs else None
    _check(_load().oracle_gemm_tf32(M, N, K, a.ctypes.data, lda, b.ctypes.data, ldb, i0, i1, j0, j1,
                                    C.ctypes.data, max(C.shape[1], 1),
                                    S.ctypes.data if with_abs else None, max(C.shape[1], 1), int(mode)))
    return C, S


def gemm_f64(a: np.ndarray, b: np.ndarray, rows=None, cols=None, with_abs=True):
    """C = A·B for fp64 inputs (same summation loop, no input decoding)."""
    a, lda = _as_rows(a, np.float64)
    b, ldb = _as_rows(b, np.float64)
    M, K = a.shape
    K2, N = b.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    i0, i1, j0, j1 = _ranges(M, N, rows, cols)
    C = np.empty((i1 - i0, j1 - j0), np.float64)
    S = np.empty_like(C) if with_abs else None
    _check(_load().oracle_gemm_f64(M, N, K, a.ctypes.data, lda, b.ctypes.data, ldb, i0, i1, j0, j1,
                                   C.ctypes.data, max(C.shape[1], 1),
                                   S.ctypes.data if with_abs else None, max(C.shape[1], 1)))
    return C, S


def gemm_f32(a: np.ndarray, b: np.ndarray, rows=None, cols=None, with_abs=True):
    """C = A·B for fp32 inputs taken at full fp32 precision (the SIMT GEMM's operands):
    every fp32 value is exactly a double, so this is the fp64 loop on the widened inputs."""
    if a.dtype != np.float32 or b.dtype != np.float32:
        raise TypeError("expected float32 inputs")
    return gemm_f64(np.asarray(a, np.float64), np.asarray(b, np.float64), rows, cols, with_abs)


def gemm_s8(a: np.ndarray, b: np.ndarray, rows=None, cols=None):
    """C = A·B for int8 inputs, exact int64 result."""
    a, lda = _as_rows(a, np.int8)
    b, ldb = _as_rows(b, np.int8)
    M, K = a.shape
    K2, N = b.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    i0, i1, j0, j1 = _ranges(M, N, rows, cols)
    C = np.empty((i1 - i0, j1 - j0), np.int64)
    _check(_load().oracle_gemm_s8(M, N, K, a.ctypes.data, lda, b.ctypes.data, ldb, i0, i1, j0, j1,
                                  C.ctypes.data, max(C.shape[1], 1)))
    return C


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, np.float64)
    _load().oracle_decode_bf16(bits.ctypes.data, out.ctypes.data, bits.size)
    return out


def decode_tf32(x: np.ndarray, mode=TF32_TRUNCATE) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.float64)
    _load().oracle_decode_tf32(x.ctypes.data, out.ctypes.data, x.size, int(mode))
    return out
