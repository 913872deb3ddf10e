"""Pins for the CPU oracle (no GPU).

The oracle restates the plain definition C[i][j] = sum_k A[i][k]·B[k][j]
("4.1 CUDA GEMM 算子性能优化", §1.1 and the one-thread-per-element kernel of
§3.1). These tests tie it to things other than itself: exhaustive decoding
against torch's own bf16 conversion, exact rational arithmetic on tiny
problems, closed forms, and invariants that a dropped term, a wrong sign, a
wrong index or a transposed operand would break. ``test_planted_mistakes``
compiles altered copies of the oracle and checks that these pins reject them.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import struct
import subprocess
from fractions import Fraction

import numpy as np
import pytest
import torch

from tensor_core_loop_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def bf16_bits_of(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def exact_bf16_values(bits: np.ndarray):
    """Decoded values via torch (independent of the oracle's own decoder)."""
    t = torch.from_numpy(bits.astype(np.uint16).view(np.int16)).view(torch.bfloat16).to(torch.float64)
    return t.numpy()


def tf32_trunc_py(x: float) -> float:
    (u,) = struct.unpack("<I", struct.pack("<f", x))
    (f,) = struct.unpack("<f", struct.pack("<I", u & 0xFFFFE000))
    return f


# ---------------------------------------------------------------- decoding

def test_decode_bf16_exhaustive(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle_mod.decode_bf16(bits)
    ref = exact_bf16_values(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


TF32_CASES = [
    # (fp32 bit pattern, truncated value, round-to-nearest-even value)
    (0x3F800000, 1.0, 1.0),
    (0x3F800001, 1.0, 1.0),                                  # 1 + 2^-23
    (0x3F801000, 1.0, 1.0),                                  # 1 + 2^-11: a tie, kept lsb 0
    (0x3F803000, 1 + 2**-10, 1 + 2**-9),                     # 1 + 2^-10 + 2^-11: a tie, kept lsb 1
    (0x3F801001, 1.0, 1 + 2**-10),                           # just above the tie
    (0x3FFFFFFF, 1 + 1023 / 1024, 2.0),                      # just below 2
    (0xBFC00001, -1.5, -1.5),
    (0x00001FFF, 0.0, 2.0**-136),                            # subnormal below the kept bits
    (0x00002000, 2.0**-136, 2.0**-136),
    (0x7F800000, float("inf"), float("inf")),
]


def test_decode_tf32_patterns(oracle_mod):
    x = np.array([c[0] for c in TF32_CASES], np.uint32).view(np.float32)
    trunc = oracle_mod.decode_tf32(x, oracle_mod.TF32_TRUNCATE)
    rne = oracle_mod.decode_tf32(x, oracle_mod.TF32_ROUND_NEAREST)
    for (pat, t, r), gt, gr in zip(TF32_CASES, trunc, rne):
        assert gt == t, hex(pat)
        assert gr == r, hex(pat)
    nanx = np.array([0x7FC00000], np.uint32).view(np.float32)
    assert np.isnan(oracle_mod.decode_tf32(nanx, 0)[0]) and np.isnan(oracle_mod.decode_tf32(nanx, 1)[0])


# ------------------------------------------------------- exact brute force

def _exact_gemm(a_vals, b_vals):
    M, K = a_vals.shape
    N = b_vals.shape[1]
    C = [[Fraction(0)] * N for _ in range(M)]
    S = [[Fraction(0)] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            c = Fraction(0)
            s = Fraction(0)
            for k in range(K):
                p = Fraction(float(a_vals[i, k])) * Fraction(float(b_vals[k, j]))
                c += p
                s += abs(p)
            C[i][j] = c
            S[i][j] = s
    return C, S


def _assert_close_to_exact(C, S, Cx, Sx, K):
    # fp64 summation of K exact products: |error| <= (K-1)·2^-53·S (first-order bound)
    gamma = Fraction(max(K - 1, 0) * 2 + 1, 2**53)
    M, N = C.shape
    for i in range(M):
        for j in range(N):
            assert abs(Fraction(float(C[i, j])) - Cx[i][j]) <= gamma * Sx[i][j], (i, j)
            assert abs(Fraction(float(S[i, j])) - Sx[i][j]) <= gamma * Sx[i][j], (i, j)


@pytest.mark.parametrize("M,N,K,seed", [(1, 1, 1, 0), (3, 5, 7, 1), (16, 16, 16, 2), (9, 4, 13, 3), (16, 1, 16, 4)])
def test_bruteforce_bf16_against_rationals(oracle_mod, M, N, K, seed):
    a, b = inputs.bf16_pair(M, N, K, seed=seed)
    ab, bb = inputs.bf16_bits(a), inputs.bf16_bits(b)
    C, S = oracle_mod.gemm_bf16(ab, bb)
    Cx, Sx = _exact_gemm(exact_bf16_values(ab), exact_bf16_values(bb))
    _assert_close_to_exact(C, S, Cx, Sx, K)


@pytest.mark.parametrize("M,N,K,seed", [(2, 3, 4, 0), (16, 16, 16, 5), (7, 11, 5, 6)])
def test_bruteforce_tf32_against_rationals(oracle_mod, M, N, K, seed):
    a, b = inputs.tf32_pair(M, N, K, seed=seed)
    an, bn = a.numpy(), b.numpy()
    C, S = oracle_mod.gemm_tf32(an, bn)
    av = np.vectorize(tf32_trunc_py)(an.astype(np.float64))
    bv = np.vectorize(tf32_trunc_py)(bn.astype(np.float64))
    Cx, Sx = _exact_gemm(av, bv)
    _assert_close_to_exact(C, S, Cx, Sx, K)


@pytest.mark.parametrize("M,N,K,seed", [(1, 1, 1, 0), (5, 3, 16, 7), (16, 16, 16, 8)])
def test_bruteforce_s8_exact(oracle_mod, M, N, K, seed):
    a, b = inputs.s8_pair(M, N, K, seed=seed)
    an, bn = a.numpy(), b.numpy()
    C = oracle_mod.gemm_s8(an, bn)
    for i in range(M):
        for j in range(N):
            assert C[i, j] == sum(int(an[i, k]) * int(bn[k, j]) for k in range(K))


# ------------------------------------------------------------ closed forms

def test_identity_and_permutation(oracle_mod):
    n = 24
    a, b = inputs.bf16_pair(n, n, n, seed=11)
    ab, bb = inputs.bf16_bits(a), inputs.bf16_bits(b)
    eye = bf16_bits_of(torch.eye(n))
    C, _ = oracle_mod.gemm_bf16(eye, bb)
    assert np.array_equal(C, exact_bf16_values(bb))
    C, _ = oracle_mod.gemm_bf16(ab, eye)
    assert np.array_equal(C, exact_bf16_values(ab))
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(3))
    P = torch.zeros(n, n)
    P[torch.arange(n), perm] = 1.0           # (P·X)[i] = X[perm[i]]
    C, _ = oracle_mod.gemm_bf16(bf16_bits_of(P), bb)
    assert np.array_equal(C, exact_bf16_values(bb)[perm.numpy()])
    C, _ = oracle_mod.gemm_bf16(ab, bf16_bits_of(P.t()))   # (X·Pᵀ)[:, j] = X[:, perm[j]]
    assert np.array_equal(C, exact_bf16_values(ab)[:, perm.numpy()])
    # int8 identity and permutation
    a8, b8 = inputs.s8_pair(n, n, n, seed=12)
    C = oracle_mod.gemm_s8(np.eye(n, dtype=np.int8), b8.numpy())
    assert np.array_equal(C, b8.numpy().astype(np.int64))
    C = oracle_mod.gemm_s8(P.numpy().astype(np.int8), b8.numpy())
    assert np.array_equal(C, b8.numpy().astype(np.int64)[perm.numpy()])


@pytest.mark.parametrize("K", [1, 2, 17, 300])
def test_all_ones_closed_form(oracle_mod, K):
    M, N = 5, 9
    C, S = oracle_mod.gemm_bf16(bf16_bits_of(torch.ones(M, K)), bf16_bits_of(torch.ones(K, N)))
    assert np.all(C == K) and np.all(S == K)
    C, S = oracle_mod.gemm_bf16(bf16_bits_of(torch.ones(M, K)), bf16_bits_of(-torch.ones(K, N)))
    assert np.all(C == -K) and np.all(S == K)
    C, S = oracle_mod.gemm_tf32(np.ones((M, K), np.float32), np.ones((K, N), np.float32))
    assert np.all(C == K) and np.all(S == K)
    C = oracle_mod.gemm_s8(np.ones((M, K), np.int8), np.ones((K, N), np.int8))
    assert np.all(C == K)


@pytest.mark.parametrize("K", [1, 64, 4096])
def test_int8_extremes_closed_form(oracle_mod, K):
    M, N = 3, 4
    hi = np.full((M, K), 127, np.int8)
    lo = np.full((M, K), -128, np.int8)
    assert np.all(oracle_mod.gemm_s8(hi, np.full((K, N), 127, np.int8)) == 16129 * K)
    assert np.all(oracle_mod.gemm_s8(lo, np.full((K, N), -128, np.int8)) == 16384 * K)
    assert np.all(oracle_mod.gemm_s8(hi, np.full((K, N), -128, np.int8)) == -16256 * K)


def test_rank_one_closed_form(oracle_mod):
    # A[i][k] = x_i, B[k][j] = y_j  ->  C[i][j] = K·x_i·y_j, exact for power-of-two data
    M, N, K = 6, 7, 40
    x = torch.tensor([2.0 ** (-i) * (-1) ** i for i in range(M)])
    y = torch.tensor([2.0 ** (j - 3) for j in range(N)])
    A = x[:, None].expand(M, K)
    B = y[None, :].expand(K, N)
    C, S = oracle_mod.gemm_bf16(bf16_bits_of(A), bf16_bits_of(B))
    ref = (K * x[:, None] * y[None, :]).double().numpy()
    assert np.array_equal(C, ref)
    assert np.array_equal(S, np.abs(ref))


def test_k_dependent_weights(oracle_mod):
    # A[0][k] = k+1, B[k][0] = 1 -> C = K(K+1)/2 ; B[k][1] = (-1)^k -> alternating sum.
    K = 100
    A = torch.arange(1, K + 1, dtype=torch.float32)[None, :]
    B = torch.stack([torch.ones(K), torch.tensor([(-1.0) ** k for k in range(K)])], dim=1)
    C, _ = oracle_mod.gemm_bf16(bf16_bits_of(A), bf16_bits_of(B))
    # bf16 holds the integers 1..100 exactly except those needing more than 8 significant bits
    avals = exact_bf16_values(bf16_bits_of(A))[0]
    assert C[0, 0] == avals.sum()
    assert C[0, 1] == sum(avals[k] * (-1) ** k for k in range(K))
    C = oracle_mod.gemm_s8(np.arange(1, K + 1, dtype=np.int64).clip(max=127).astype(np.int8)[None, :],
                           np.ones((K, 1), np.int8))
    assert C[0, 0] == int(np.arange(1, K + 1).clip(max=127).sum())


# -------------------------------------------------------------- invariants

def test_transpose_invariant_bitwise(oracle_mod):
    M, N, K = 37, 29, 53
    a, b = inputs.bf16_pair(M, N, K, seed=21)
    C, S = oracle_mod.gemm_bf16(inputs.bf16_bits(a), inputs.bf16_bits(b))
    Ct, St = oracle_mod.gemm_bf16(inputs.bf16_bits(b.t().contiguous()), inputs.bf16_bits(a.t().contiguous()))
    assert np.array_equal(C, Ct.T) and np.array_equal(S, St.T)
    a8, b8 = inputs.s8_pair(M, N, K, seed=22)
    C8 = oracle_mod.gemm_s8(a8.numpy(), b8.numpy())
    C8t = oracle_mod.gemm_s8(b8.t().contiguous().numpy(), a8.t().contiguous().numpy())
    assert np.array_equal(C8, C8t.T)


def test_padded_leading_dims_and_blocks(oracle_mod):
    M, N, K = 40, 24, 72
    a, b = inputs.bf16_pair(M, N, K, seed=5)
    ap, bp = inputs.bf16_pair(M, N, K, seed=5, lda=K + 8, ldb=N + 16)
    C, S = oracle_mod.gemm_bf16(inputs.bf16_bits(a), inputs.bf16_bits(b))
    Cp, Sp = oracle_mod.gemm_bf16(inputs.bf16_bits(ap), inputs.bf16_bits(bp))
    assert np.array_equal(C, Cp) and np.array_equal(S, Sp)
    Cb, Sb = oracle_mod.gemm_bf16(inputs.bf16_bits(ap), inputs.bf16_bits(bp), rows=(7, 31), cols=(3, 20))
    assert np.array_equal(Cb, C[7:31, 3:20]) and np.array_equal(Sb, S[7:31, 3:20])
    a8, b8 = inputs.s8_pair(M, N, K, seed=6)
    a8p, b8p = inputs.s8_pair(M, N, K, seed=6, lda=K + 16, ldb=N + 16)
    C8 = oracle_mod.gemm_s8(a8.numpy(), b8.numpy())
    assert np.array_equal(C8, oracle_mod.gemm_s8(a8p.numpy(), b8p.numpy()))
    assert np.array_equal(C8[5:9, 1:2], oracle_mod.gemm_s8(a8p.numpy(), b8p.numpy(), rows=(5, 9), cols=(1, 2)))
    at, bt = inputs.tf32_pair(M, N, K, seed=7)
    atp, btp = inputs.tf32_pair(M, N, K, seed=7, lda=K + 4, ldb=N + 4)
    assert np.array_equal(oracle_mod.gemm_tf32(at.numpy(), bt.numpy())[0],
                          oracle_mod.gemm_tf32(atp.numpy(), btp.numpy())[0])


def test_linearity_exact_on_small_integers(oracle_mod):
    g = torch.Generator().manual_seed(9)
    M, N, K = 12, 10, 33
    A1 = torch.randint(-8, 9, (M, K), generator=g).float()
    A2 = torch.randint(-8, 9, (M, K), generator=g).float()
    B = torch.randint(-8, 9, (K, N), generator=g).float()
    c1, _ = oracle_mod.gemm_bf16(bf16_bits_of(A1), bf16_bits_of(B))
    c2, _ = oracle_mod.gemm_bf16(bf16_bits_of(A2), bf16_bits_of(B))
    c12, _ = oracle_mod.gemm_bf16(bf16_bits_of(A1 + A2), bf16_bits_of(B))
    assert np.array_equal(c12, c1 + c2)
    c3, _ = oracle_mod.gemm_bf16(bf16_bits_of(3 * A1), bf16_bits_of(B))
    assert np.array_equal(c3, 3 * c1)


def test_abs_sum_invariants(oracle_mod):
    M, N, K = 20, 30, 64
    a, b = inputs.bf16_pair(M, N, K, seed=31)
    C, S = oracle_mod.gemm_bf16(inputs.bf16_bits(a), inputs.bf16_bits(b))
    assert np.all(S >= np.abs(C))
    Ca, Sa = oracle_mod.gemm_bf16(inputs.bf16_bits(a.abs()), inputs.bf16_bits(b.abs()))
    assert np.array_equal(Ca, S) and np.array_equal(Sa, S)


def test_f64_entry_matches_numpy_on_exact_data(oracle_mod):
    # small integers: every partial sum is exact, so any correct summation order agrees
    g = np.random.default_rng(4)
    A = g.integers(-50, 51, (17, 23)).astype(np.float64)
    B = g.integers(-50, 51, (23, 19)).astype(np.float64)
    C, S = oracle_mod.gemm_f64(A, B)
    assert np.array_equal(C, A @ B)
    assert np.array_equal(S, np.abs(A) @ np.abs(B))


def test_f32_entry_exact_and_full_precision(oracle_mod):
    # fp32 inputs that are small integers: the exact integer product (brute force)
    g = np.random.default_rng(5)
    A = g.integers(-40, 41, (9, 13)).astype(np.float32)
    B = g.integers(-40, 41, (13, 7)).astype(np.float32)
    C, S = oracle_mod.gemm_f32(A, B)
    exact = [[sum(int(A[i, k]) * int(B[k, j]) for k in range(13)) for j in range(7)] for i in range(9)]
    assert np.array_equal(C, np.array(exact, dtype=np.float64))
    assert np.array_equal(S, np.abs(A).astype(np.float64) @ np.abs(B).astype(np.float64))
    # full fp32 precision, not TF32: 1 + 2^-20 survives (TF32 keeps 10 mantissa bits)
    a = np.full((2, 3), 1.0 + 2.0 ** -20, np.float32)
    b = np.zeros((3, 2), np.float32)
    b[0, :] = 1.0
    C, _ = oracle_mod.gemm_f32(a, b)
    assert np.all(C == 1.0 + 2.0 ** -20)
    # padded rows (a wider leading dimension) give the same result as dense ones
    wide = np.full((9, 16), np.nan, np.float32)
    wide[:, :13] = A
    C2, _ = oracle_mod.gemm_f32(wide[:, :13], B)
    assert np.array_equal(C2, np.array(exact, dtype=np.float64))


def test_f32_bound_admits_fma_chain_and_rejects_a_dropped_term():
    from bounds import bound_for
    g = np.random.default_rng(6)
    K = 300
    a = g.standard_normal(K).astype(np.float32)
    b = g.standard_normal(K).astype(np.float32)
    exact = float(np.dot(a.astype(np.float64), b.astype(np.float64)))
    S = float(np.dot(np.abs(a).astype(np.float64), np.abs(b).astype(np.float64)))
    # an fp32 chain with one rounding per step (the product formed exactly, as an FMA does)
    acc = np.float32(0.0)
    for x, y in zip(a, b):
        acc = np.float32(float(acc) + float(x) * float(y))
    bound = float(bound_for("f32", np.array([exact]), np.array([S]), K)[0])
    assert abs(float(acc) - exact) <= bound
    # losing one product term is caught
    assert abs(float(acc) - float(a[7]) * float(b[7]) - exact) > bound


def test_bad_arguments_rejected(oracle_mod):
    a = np.zeros((4, 8), np.uint16)
    b = np.zeros((7, 4), np.uint16)
    with pytest.raises(ValueError):
        oracle_mod.gemm_bf16(a, b)
    with pytest.raises(ValueError):
        oracle_mod.gemm_bf16(a, np.zeros((8, 4), np.uint16), rows=(2, 9))


# ---------------------------------------------------- planted mistakes

MUTANTS = {
    "dropped_last_k": ("for (long k = 0; k < K; ++k) {\n            const double a", "for (long k = 0; k < K - 1; ++k) {\n            const double a"),
    "wrong_sign": ("c[j] += a * b[j];", "c[j] -= a * b[j];"),
    "transposed_b": ("Bd[k * ncols + j] = dec_bf16(B[k * ldb + j0 + j]);", "Bd[k * ncols + j] = dec_bf16(B[(j0 + j) * ldb + k]);"),
    "a_column_index": ("return dec_bf16(((const uint16_t*)A)[i * lda + k]);", "return dec_bf16(((const uint16_t*)A)[k * lda + i]);"),
    "bf16_shift": ("uint32_t u = ((uint32_t)h) << 16;", "uint32_t u = ((uint32_t)h) << 15;"),
    "abs_missing": ("s[j] += fabs(a * b[j]);", "s[j] += a * b[j];"),
}


def _run_pins_on(lib_path):
    """A subset of the pins above, driven against an arbitrary build of the oracle."""
    lib = ctypes.CDLL(lib_path)
    f = lib.oracle_gemm_bf16
    L, P = ctypes.c_long, ctypes.c_void_p
    f.argtypes = [L, L, L, P, L, P, L, L, L, L, L, P, L, P, L]
    f.restype = ctypes.c_int

    def gemm(ab, bb):
        M, K = ab.shape
        N = bb.shape[1]
        C = np.empty((M, N)); S = np.empty((M, N))
        ab = np.ascontiguousarray(ab); bb = np.ascontiguousarray(bb)
        assert f(M, N, K, ab.ctypes.data, K, bb.ctypes.data, N, 0, M, 0, N, C.ctypes.data, N, S.ctypes.data, N) == 0
        return C, S

    failures = []
    # brute force vs rationals on a non-square problem
    a, b = inputs.bf16_pair(5, 7, 9, seed=2)
    ab, bb = inputs.bf16_bits(a), inputs.bf16_bits(b)
    C, S = gemm(ab, bb)
    Cx, Sx = _exact_gemm(exact_bf16_values(ab), exact_bf16_values(bb))
    try:
        _assert_close_to_exact(C, S, Cx, Sx, 9)
    except AssertionError:
        failures.append("bruteforce")
    # all-ones closed form with a negative operand
    C, S = gemm(bf16_bits_of(torch.ones(3, 6)), bf16_bits_of(-torch.ones(6, 4)))
    if not (np.all(C == -6) and np.all(S == 6)):
        failures.append("closed_form")
    return failures


def test_planted_mistakes_are_caught(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(os.path.join(ROOT, "oracle", "gemm_oracle.c")).read()
    clean = tmp_path / "clean.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-shared", "-fPIC", "-o", str(clean),
                    os.path.join(ROOT, "oracle", "gemm_oracle.c"), "-lm"], check=True)
    assert _run_pins_on(str(clean)) == []
    for name, (old, new) in MUTANTS.items():
        assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
        path = tmp_path / f"{name}.c"
        path.write_text(src.replace(old, new))
        so = tmp_path / f"{name}.so"
        subprocess.run(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-shared", "-fPIC", "-o", str(so),
                        str(path), "-lm"], check=True)
        assert _run_pins_on(str(so)), f"planted mistake '{name}' was not caught"
