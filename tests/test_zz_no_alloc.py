"""gemm_s8_static: the int8 GEMM that allocates nothing.

Some callers cannot let the library call cudaMalloc: a process whose device
memory is already held by another allocator's pool, or code that must not
trigger the device-wide synchronisation gemm_s8 performs when it grows its
scratch. gemm_s8_static writes its packed operands into a fixed 64 MiB array
that is part of the library's device image instead. These tests call it
through the C ABI and compare it with gemm_s8 (the int8 result is exact, so
the comparison is bit for bit), twice in a row on different problems so that
the second call runs over the first call's leftovers in the shared array.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import tensor_core_loop_gb300 as tcl
from tensor_core_loop_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_core_loop_gb300 import _build
    _build.build()
    return tcl.lib()


def _up(x, q):
    return -(-x // q) * q


def _operands(M, N, K, seed):
    a, b = inputs.s8_pair(M, N, K, seed=seed)
    lda, ldb = _up(K, 16), _up(N, 16)
    ad = torch.zeros((M, lda), dtype=torch.int8, device=DEV)
    bd = torch.zeros((K, ldb), dtype=torch.int8, device=DEV)
    ad[:, :K] = a.to(DEV)
    bd[:, :N] = b.to(DEV)
    return ad, lda, bd, ldb


def _call(fn, M, N, K, ad, lda, bd, ldb):
    ldc = _up(N, 4)
    c = torch.full((M, ldc), -7, dtype=torch.int32, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = fn(M, N, K, ad.data_ptr(), lda, bd.data_ptr(), ldb, c.data_ptr(), ldc, stream)
    assert st == 0, tcl.STATUS.get(st, st)
    torch.cuda.synchronize()
    return c


def test_static_entry_matches_gemm_s8_on_two_calls_in_a_row(L):
    # first a larger problem, then a smaller one with different ragged edges:
    # the second call runs over what the first left in the shared array
    for (M, N, K, seed) in [(1000, 520, 1029, 1), (384, 260, 777, 2)]:
        ad, lda, bd, ldb = _operands(M, N, K, seed)
        ref = _call(L.gemm_s8, M, N, K, ad, lda, bd, ldb)
        got = _call(L.gemm_s8_static, M, N, K, ad, lda, bd, ldb)
        assert torch.equal(got, ref), f"gemm_s8_static differs from gemm_s8 at {M}x{N}x{K}"
        assert (got[:, N:] == -7).all(), "wrote outside C"
    st, code = tcl.last_device_error()
    assert st == 0, f"device status word reported code {code}"


def _sample_rows(M, n, seed):
    g = np.random.default_rng(seed)
    fixed = {0, 1, 127, 128, M // 2, M - 129, M - 128, M - 1}
    return sorted(r for r in fixed.union(g.integers(0, M, n).tolist()) if 0 <= r < M)


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 4096), (3072, 3072, 2048)])
def test_static_entry_large_problems_exact(L, oracle_mod, M, N, K):
    # Problems for which gemm_s8 itself runs on two SMs per tile: 4096³ fills the
    # 64 MiB array exactly (2·(4096·4096 + 4096·4096) bytes of bf16 copies). The
    # result is checked bit for bit against the CPU oracle on sampled rows and in
    # full against gemm_s8, on two calls in a row (the second over the first's
    # leftovers in the shared array).
    assert tcl.plan(tcl.IN_S8, 0, M, N, K)["cta_pair"] == 2
    a, b = inputs.s8_pair(M, N, K, seed=M + K)
    ad, bd = a.to(DEV), b.to(DEV)
    ref = _call(L.gemm_s8, M, N, K, ad, K, bd, N)
    for call in range(2):
        got = _call(L.gemm_s8_static, M, N, K, ad, K, bd, N)
        assert torch.equal(got, ref), f"call {call}: gemm_s8_static differs from gemm_s8 at {M}x{N}x{K}"
    host = got.cpu().numpy()
    an, bn = a.numpy(), b.numpy()
    for r in _sample_rows(M, 6, seed=K):
        want = oracle_mod.gemm_s8(an, bn, rows=(r, r + 1))
        assert np.array_equal(host[r:r + 1, :N].astype(np.int64), want), f"row {r} differs from the oracle"
    st, code = tcl.last_device_error()
    assert st == 0, f"device status word reported code {code}"


def test_static_entry_rejects_problems_beyond_its_buffer(L):
    # 8192³ needs 2·(8192·8192 + 8192·8192) bytes = 256 MiB of packed operands > 64 MiB;
    # the check happens on the host before any device work (pointers never touched)
    fake = 0x10000000
    assert L.gemm_s8_static(8192, 8192, 8192, fake, 8192, fake, 8192, fake, 8192, None) == 11
    # one row more than 4096³ no longer fits
    assert L.gemm_s8_static(4097, 4096, 4096, fake, 4096, fake, 4096, fake, 4096, None) == 11
