"""Parity of the CUDA path (through the C ABI) with the CPU oracle, on a GB300.

Small problems are compared element by element over the whole output; the
full-size workloads (4096³ and the K sweep) are compared on sampled rows that
cover several M tiles, including the first and last, across all N tiles.
Bounds: tests/bounds.py. int8 is compared bit-exactly.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import tensor_core_loop_gb300 as tcl
from tensor_core_loop_gb300 import inputs

from bounds import assert_exact, assert_within

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tcl.lib()
    yield
    st, code = tcl.last_device_error()
    assert st == 0, f"device status word reported code {code}"


def run(a, b, out_dtype=None, cfg=None, ldc=None, canary=True):
    """Run through the C ABI into a C buffer padded to `ldc` columns plus one guard row
    filled with a sentinel; check the sentinel survived; return C[:M, :N] on the host."""
    M, N = a.shape[0], b.shape[1]
    out_dtype = out_dtype or {torch.bfloat16: torch.float32, torch.float32: torch.float32,
                              torch.int8: torch.int32}[a.dtype]
    if ldc is None:   # smallest leading dimension that keeps rows 16-byte aligned
        q = 16 // torch.empty((), dtype=out_dtype).element_size()
        ldc = -(-N // q) * q
    buf = torch.empty((M + 1, ldc), dtype=out_dtype, device=DEV)
    sentinel = -12345 if out_dtype == torch.int32 else float("nan") if out_dtype == torch.float32 else -3.0
    buf.fill_(sentinel)
    c = buf[:M, :N]
    tcl.gemm_into(a, b, c, cfg=cfg)
    torch.cuda.synchronize()
    host = buf.cpu()
    if canary:
        pad = torch.cat([host[:M, N:].reshape(-1), host[M].reshape(-1)])
        if out_dtype == torch.float32:
            assert torch.isnan(pad).all(), "kernel wrote outside C"
        else:
            assert (pad == sentinel).all(), "kernel wrote outside C"
    return host[:M, :N]


def to_dev(t):
    """Copy a (possibly padded) host view to the device, keeping its leading dimension."""
    if t.is_contiguous():
        return t.to(DEV)
    rows, cols = t.shape
    ld = t.stride(0)
    full = torch.as_strided(t, (rows, ld), (ld, 1)) if rows else t
    return full.to(DEV)[:, :cols]


def up(x, q):
    return -(-x // q) * q


def to_dev_off(t, off):
    """Copy a (possibly padded) host view to the device `off` elements into a fresh buffer,
    so that its base address sits off the 16-byte grid; the bytes before it hold the view's
    own padding pattern (or zeros for a dense view)."""
    rows, cols = t.shape
    ld = t.stride(0) if rows > 1 else cols
    full = torch.as_strided(t, (rows, ld), (ld, 1))
    flat = torch.zeros(off + rows * ld, dtype=t.dtype, device=DEV)
    flat[off:] = full.reshape(-1).to(DEV)
    return torch.as_strided(flat, (rows, cols), (ld, 1), off)


def run_off(a, b, out_dtype, ldc, off):
    """Run into a C placed `off` elements into a sentinel-filled buffer with leading dimension
    ldc; check nothing outside the M×N block changed; return C on the host."""
    M, N = a.shape[0], b.shape[1]
    sentinel = -12345 if out_dtype == torch.int32 else -3.0
    flat = torch.full((off + (M + 1) * ldc,), sentinel, dtype=out_dtype, device=DEV)
    c = torch.as_strided(flat, (M, N), (ldc, 1), off)
    tcl.gemm_into(a, b, c)
    torch.cuda.synchronize()
    host = flat.cpu()
    inside = torch.zeros_like(host, dtype=torch.bool)
    torch.as_strided(inside, (M, N), (ldc, 1), off).fill_(True)
    assert (host[~inside] == sentinel).all(), "kernel wrote outside C"
    return torch.as_strided(host, (M, N), (ldc, 1), off).clone()


def bf16_case(oracle_mod, M, N, K, seed=0, out_dtype=torch.float32, cfg=None, lda=None, ldb=None, ldc=None,
              rows=None):
    a, b = inputs.bf16_pair(M, N, K, seed=seed, lda=lda or up(K, 8), ldb=ldb or up(N, 8))
    got = run(to_dev(a), to_dev(b), out_dtype=out_dtype, cfg=cfg, ldc=ldc).double().numpy()
    kind = "bf16_f32" if out_dtype == torch.float32 else "bf16_bf16"
    if rows is None:
        ref, S = oracle_mod.gemm_bf16(inputs.bf16_bits(a), inputs.bf16_bits(b))
        return assert_within(kind, got, ref, S, f"bf16 {M}x{N}x{K}")
    worst = 0.0
    for r in rows:
        ref, S = oracle_mod.gemm_bf16(inputs.bf16_bits(a), inputs.bf16_bits(b), rows=(r, r + 1))
        worst = max(worst, assert_within(kind, got[r:r + 1], ref, S, f"bf16 {M}x{N}x{K} row {r}"))
    return worst


def sample_rows(M, n=24, seed=0):
    g = np.random.default_rng(seed)
    fixed = {0, 1, 31, 32, 127, 128, M // 2, M - 129, M - 128, M - 1}
    return sorted(r for r in fixed.union(g.integers(0, M, n).tolist()) if 0 <= r < M)


# ------------------------------------------------------------- small, full compare

def test_bf16_256_cube_fp32(oracle_mod):
    bf16_case(oracle_mod, 256, 256, 256, seed=0)


def test_bf16_512_cube_fp32(oracle_mod):
    bf16_case(oracle_mod, 512, 512, 512, seed=1)


@pytest.mark.parametrize("K", [8, 16, 64, 72, 128, 200, 3 * 64, 5 * 64, 7 * 64, 1000])
def test_bf16_k_edges(oracle_mod, K):
    # one k-block, two, fewer blocks than stages, ring wrap (stages ± 1), ragged last block
    bf16_case(oracle_mod, 256, 384, K, seed=K)


@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (130, 260, 200), (129, 136, 64), (300, 520, 96), (77, 1000, 40)])
def test_bf16_ragged_shapes(oracle_mod, M, N, K):
    bf16_case(oracle_mod, M, N, K, seed=M + N)


def test_bf16_padded_leading_dims(oracle_mod):
    bf16_case(oracle_mod, 200, 264, 136, seed=5, lda=136 + 8, ldb=264 + 16, ldc=264 + 12)


@pytest.mark.parametrize("N,ldc", [(1, 4), (3, 8), (5, 12), (261, 264), (259, 268)])
def test_bf16_ragged_right_edge_fp32(oracle_mod, N, ldc):
    # a right edge off the 16-byte grid is stored element by element; the canary
    # columns between N and ldc must stay untouched
    bf16_case(oracle_mod, 140, N, 72, seed=N, ldc=ldc)


@pytest.mark.parametrize("N,ldc", [(1, 8), (7, 8), (260, 272), (300, 304)])
def test_bf16_ragged_right_edge_bf16(oracle_mod, N, ldc):
    bf16_case(oracle_mod, 140, N, 72, seed=N, out_dtype=torch.bfloat16, ldc=ldc)


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (300, 520, 200)])
def test_bf16_out_bf16(oracle_mod, M, N, K):
    bf16_case(oracle_mod, M, N, K, seed=3, out_dtype=torch.bfloat16)


@pytest.mark.parametrize("bn,stages", [(256, 1), (256, 2), (256, 3), (256, 4), (128, 1), (128, 2), (128, 4),
                                       (128, 6)])
def test_bf16_each_variant(oracle_mod, bn, stages):
    bf16_case(oracle_mod, 384, 512, 640, seed=9, cfg=tcl.Config(bn=bn, stages=stages))


@pytest.mark.parametrize("stages", [1, 2, 4])
def test_bf16_sync_producer(oracle_mod, stages):
    bf16_case(oracle_mod, 384, 512, 640, seed=9, cfg=tcl.Config(bn=256, stages=stages, producer=1))
    bf16_case(oracle_mod, 130, 261, 200, seed=10, cfg=tcl.Config(bn=256, stages=stages, producer=1), ldc=264)


@pytest.mark.parametrize("stages", [1, 2, 3, 4])
def test_bf16_cpasync_producer(oracle_mod, stages):
    cfg = tcl.Config(bn=256, stages=stages, producer=tcl.PRODUCER_CPASYNC)
    bf16_case(oracle_mod, 384, 512, 640, seed=9, cfg=cfg)
    # ragged M, N (a chunk straddling the right edge copies only its in-range columns) and K
    bf16_case(oracle_mod, 130, 261, 200, seed=10, cfg=cfg, ldc=264)
    bf16_case(oracle_mod, 1, 9, 8, seed=11, cfg=cfg)


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (512, 512, 1024), (300, 520, 200), (130, 261, 72), (1, 8, 8),
                                   (777, 1000, 1216), (1024, 768, 4096)])
def test_bf16_pair_kernel(oracle_mod, M, N, K):
    # two SMs per 256×256 tile (cta_group::2); ragged shapes leave the peer CTA's rows
    # or B columns partly or wholly outside the matrix
    ldc = -(-N // 4) * 4 if N % 4 else None
    bf16_case(oracle_mod, M, N, K, seed=M + K, cfg=tcl.Config(cta_pair=2), ldc=ldc)


@pytest.mark.parametrize("M,N,K", [(256, 224, 256), (512, 1000, 640), (300, 452, 200), (1024, 4096, 512)])
def test_bf16_pair_kernel_224(oracle_mod, M, N, K):
    # 256×224 pair tiles: each SM supplies 112 columns of B (two 64-column boxes, the
    # last 16 columns unread by the MMA)
    bf16_case(oracle_mod, M, N, K, seed=N, cfg=tcl.Config(cta_pair=2, bn=224))


@pytest.mark.parametrize("stages", [4, 6])
def test_bf16_pair_kernel_stages_and_grid(oracle_mod, stages):
    bf16_case(oracle_mod, 768, 1280, 832, seed=stages, cfg=tcl.Config(cta_pair=2, stages=stages))
    bf16_case(oracle_mod, 768, 1280, 832, seed=stages, cfg=tcl.Config(cta_pair=2, stages=stages, max_ctas=4,
                                                                         group_m=2))
    bf16_case(oracle_mod, 768, 1280, 832, seed=stages, cfg=tcl.Config(cta_pair=2, stages=stages,
                                                                         one_cta_per_tile=1))


@pytest.mark.parametrize("M,N,K", [(512, 512, 512), (300, 264, 200)])
def test_bf16_pair_kernel_bf16_out(oracle_mod, M, N, K):
    bf16_case(oracle_mod, M, N, K, seed=5, out_dtype=torch.bfloat16, cfg=tcl.Config(cta_pair=2))


@pytest.mark.parametrize("M,N,K,pieces", [
    (768, 768, 4096, 0),     # automatic (64 k-blocks): the 9th tile in 4 pieces, three fp32 partials
    (768, 768, 2048, 0),     # automatic at 32 k-blocks (the bf16 C's tail threshold): 4 pieces of 8
    (768, 768, 2048, 2),
    (768, 768, 2048, 3),
    (700, 750, 1000, 4),     # ragged M, N: the last piece rounds and stores only what lies in C
    (512, 1280, 576, 2),
    (1536, 1280, 2048, 2),   # 30 tiles on 4 pairs: two tail tiles, each with its own workspace rows
])
def test_bf16_out_stream_k(oracle_mod, M, N, K, pieces):
    # bf16 C with a stream-K tail: the pieces' fp32 sums meet in an fp32 workspace in piece
    # order and the last piece rounds once into C, so the bf16 bound holds unchanged
    cfg = tcl.Config(cta_pair=2, max_ctas=8, stream_k=pieces)
    pl = tcl.plan(tcl.IN_BF16, tcl.OUT_BF16, M, N, K, cfg)
    assert pl["sk_tiles"] > 0 and pl["workspace_bytes"] > 0
    ldc = -(-N // 8) * 8 if N % 8 else None
    bf16_case(oracle_mod, M, N, K, seed=K + pieces, out_dtype=torch.bfloat16, cfg=cfg, ldc=ldc)


@pytest.mark.parametrize("M,N,K,max_ctas,out", [
    (1280, 1280, 2048, 8, torch.float32),    # 25 tiles on 4 pairs: 5 waves, then 5 tiles in ranges of 40 k-blocks
    (1280, 1280, 2048, 8, torch.bfloat16),   # the cut tiles' fp32 partials through the per-boundary workspace
    (700, 750, 2000, 4, torch.float32),      # ragged M, N and last k-block; 9 tiles on 2 pairs
    (1536, 1280, 4096, 14, torch.float32),   # 30 tiles on 7 pairs: ranges of 64 + 3/7 k-blocks
])
def test_bf16_balanced_stream_k(oracle_mod, M, N, K, max_ctas, out):
    # balanced stream-K: equal k-block ranges per pair crossing tile boundaries; each cut
    # tile's head is stored first, its rest added after the head's flag
    cfg = tcl.Config(cta_pair=2, max_ctas=max_ctas, stream_k=5)
    pl = tcl.plan(tcl.IN_BF16, tcl.OUT_F32 if out == torch.float32 else tcl.OUT_BF16, M, N, K, cfg)
    assert pl["sk_balanced"] == 1 and pl["sk_tiles"] > 0
    ldc = up(N, 4 if out == torch.float32 else 8)
    bf16_case(oracle_mod, M, N, K, seed=K + M, out_dtype=out, cfg=cfg, ldc=ldc)
    a, b = inputs.bf16_pair(M, N, K, seed=K + M, lda=up(K, 8), ldb=up(N, 8))
    a, b = to_dev(a), to_dev(b)
    first = run(a, b, out_dtype=out, cfg=cfg, ldc=ldc, canary=False)
    for _ in range(3):
        assert torch.equal(run(a, b, out_dtype=out, cfg=cfg, ldc=ldc, canary=False), first)


def test_balanced_stream_k_int8_and_tf32(oracle_mod):
    a, b = inputs.s8_pair(1280, 1280, 2112, seed=61)
    cfg = tcl.Config(cta_pair=2, bn=256, max_ctas=8, stream_k=5)
    assert tcl.plan(tcl.IN_S8, 0, 1280, 1280, 2112, cfg)["sk_balanced"] == 1
    got = run(a.to(DEV), b.to(DEV), cfg=cfg).numpy()
    assert_exact(got, oracle_mod.gemm_s8(a.numpy(), b.numpy()), "s8 balanced stream-K")
    got2 = run(a.to(DEV), b.to(DEV), cfg=tcl.Config(cta_pair=2, bn=256, max_ctas=8, stream_k=5, s8_path=2)).numpy()
    assert (got2 == got).all()
    a, b = inputs.tf32_pair(1280, 1280, 1024, seed=62)
    cfg = tcl.Config(cta_pair=2, max_ctas=8, stream_k=5)
    assert tcl.plan(tcl.IN_TF32, 0, 1280, 1280, 1024, cfg)["sk_balanced"] == 1
    got = run(a.to(DEV), b.to(DEV), cfg=cfg).double().numpy()
    ref, S = oracle_mod.gemm_tf32(a.numpy(), b.numpy())
    assert_within("tf32", got, ref, S, "tf32 balanced stream-K")


def test_bf16_out_stream_k_rounds_once():
    # the same tile split or not: the fp32 sums differ only in summation order, and the
    # split result equals the split fp32 result rounded to bf16 (one rounding)
    a, b = inputs.bf16_pair(768, 768, 2048, seed=41)
    a, b = a.to(DEV), b.to(DEV)
    for pieces in (2, 4):
        cfg = tcl.Config(cta_pair=2, max_ctas=8, stream_k=pieces)
        c16 = run(a, b, out_dtype=torch.bfloat16, cfg=cfg)
        c32 = run(a, b, out_dtype=torch.float32, cfg=cfg)
        assert torch.equal(c16, c32.to(torch.bfloat16))
        for _ in range(5):
            assert torch.equal(run(a, b, out_dtype=torch.bfloat16, cfg=cfg, canary=False), c16)


@pytest.mark.parametrize("M,N,K,pieces", [
    (768, 768, 2048, 0),     # 9 tiles on 4 pairs: 2 full waves, the 9th tile in 4 pieces of 8 k-blocks
    (768, 768, 2048, 2),
    (768, 768, 2048, 3),     # uneven pieces: 10, 11, 11 k-blocks
    (700, 750, 1000, 4),     # ragged M, N (last chunk added element by element), K tail in the last piece
    (700, 750, 2000, 0),     # automatic: 32 k-blocks (the last one ragged) in 4 pieces
    (512, 1280, 576, 2),     # 10 tiles on 4 pairs: two tail tiles, pieces of 4 and 5 k-blocks
])
def test_bf16_pair_stream_k(oracle_mod, M, N, K, pieces):
    # four pairs of SMs (max_ctas 8); the last partial wave of tiles is cut into K ranges
    # whose results are added in range order (store, then TMA reductions)
    cfg = tcl.Config(cta_pair=2, max_ctas=8, stream_k=pieces)
    pl = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, M, N, K, cfg)
    assert pl["sk_tiles"] > 0 and pl["sk_pieces"] == (pieces or pl["sk_pieces"]) and pl["sk_pieces"] >= 2
    ldc = -(-N // 4) * 4 if N % 4 else None
    bf16_case(oracle_mod, M, N, K, seed=K + pieces, cfg=cfg, ldc=ldc)


def test_stream_k_deterministic():
    # the same plan gives the same bits every time: the pieces of a split tile are
    # added in range order whatever order the pairs finish in
    a, b = inputs.bf16_pair(768, 768, 2048, seed=29)
    a, b = a.to(DEV), b.to(DEV)
    for pieces in (2, 4):
        cfg = tcl.Config(cta_pair=2, max_ctas=8, stream_k=pieces)
        first = run(a, b, cfg=cfg)
        for _ in range(10):
            assert torch.equal(run(a, b, cfg=cfg, canary=False), first)


@pytest.mark.parametrize("M,N,K,lda,ldb,ldc,offs,out", [
    (130, 261, 203, 205, 263, 263, (1, 3, 1), torch.float32),    # K % 8 = 3, odd pitches, odd bases
    (200, 300, 1000, 1003, 304, 301, (0, 0, 1), torch.bfloat16),  # only A's pitch and C's base/pitch off-grid
    (300, 264, 512, 512, 264, 266, (0, 0, 2), torch.float32),     # only C off-grid (fp32 base 8 B off)
    (1, 9, 5, 5, 9, 9, (1, 1, 1), torch.float32),                 # one row, K = 5
])
def test_bf16_off_grid_operands(oracle_mod, M, N, K, lda, ldb, ldc, offs, out):
    # operands and outputs off the 16-byte grid the tensor copies need go through
    # aligned copies (K zero-padded) and a copy-out; the padding poison must not leak
    a, b = inputs.bf16_pair(M, N, K, seed=K, lda=lda, ldb=ldb)
    got = run_off(to_dev_off(a, offs[0]), to_dev_off(b, offs[1]), out, ldc, offs[2]).double().numpy()
    ref, S = oracle_mod.gemm_bf16(inputs.bf16_bits(a), inputs.bf16_bits(b))
    assert_within("bf16_f32" if out == torch.float32 else "bf16_bf16", got, ref, S, f"off-grid {M}x{N}x{K}")


def test_bf16_off_grid_pair_kernel(oracle_mod):
    a, b = inputs.bf16_pair(1024, 1000, 1004, seed=31, lda=1005, ldb=1001)
    da, db = to_dev_off(a, 1), to_dev_off(b, 1)
    M, N = 1024, 1000
    flat = torch.full((1 + M * 1001,), -3.0, dtype=torch.float32, device=DEV)
    c = torch.as_strided(flat, (M, N), (1001, 1), 1)
    tcl.gemm_into(da, db, c, cfg=tcl.Config(cta_pair=2))
    got = c.cpu().double().numpy()
    ref, S = oracle_mod.gemm_bf16(inputs.bf16_bits(a), inputs.bf16_bits(b))
    assert_within("bf16_f32", got, ref, S, "off-grid pair kernel")


def test_tf32_off_grid_operands(oracle_mod):
    a, b = inputs.tf32_pair(130, 100, 203, seed=3, lda=207, ldb=101)   # K % 4 = 3
    got = run_off(to_dev_off(a, 1), to_dev_off(b, 1), torch.float32, 101, 1).double().numpy()
    ref, S = oracle_mod.gemm_tf32(a.numpy(), b.numpy())
    assert_within("tf32", got, ref, S, "tf32 off-grid")


@pytest.mark.parametrize("M,N,K,cfg", [
    (512, 512, 512, dict(cta_pair=2)),
    (300, 452, 200, dict(cta_pair=2)),                       # ragged: the peer CTA's rows past M
    (1024, 1000, 1004, dict(cta_pair=2, bn=224)),            # B half of 112 columns in 4 boxes; K % 32 = 12
    (768, 768, 2048, dict(cta_pair=2, max_ctas=8, stream_k=3)),   # stream-K pieces added by TMA reductions
])
def test_tf32_pair_kernel(oracle_mod, M, N, K, cfg):
    # TF32 on two SMs per tile: kind::tf32 pair MMAs, B N-major (32-byte swizzle units), 32-deep k-blocks
    c = tcl.Config(**cfg)
    assert tcl.plan(tcl.IN_TF32, 0, M, N, K, c)["cta_pair"] == 2
    a, b = inputs.tf32_pair(M, N, K, seed=M + N)
    ldc = -(-N // 4) * 4
    got = run(a.to(DEV), b.to(DEV), cfg=c, ldc=ldc).double().numpy()
    ref, S = oracle_mod.gemm_tf32(a.numpy(), b.numpy())
    assert_within("tf32", got, ref, S, f"tf32 pair {M}x{N}x{K}")


def test_s8_off_grid_operands(oracle_mod):
    a, b = inputs.s8_pair(130, 261, 203, seed=4, lda=205, ldb=263)
    got = run_off(to_dev_off(a, 1), to_dev_off(b, 3), torch.int32, 263, 1).numpy()
    ref = oracle_mod.gemm_s8(a.numpy(), b.numpy())
    assert_exact(got, ref, "int8 off-grid")


def simt_case(oracle_mod, M, N, K, seed, lda=None, ldb=None, ldc=None, offs=(0, 0, 0), rows=None):
    a, b = inputs.tf32_pair(M, N, K, seed=seed, lda=lda, ldb=ldb)   # fp32 N(0,1) operands
    ldc = ldc or N
    got = run_off_simt(to_dev_off(a, offs[0]), to_dev_off(b, offs[1]), ldc, offs[2]).double().numpy()
    for r in (rows or [None]):
        sl = slice(None) if r is None else slice(r, r + 1)
        ref, S = oracle_mod.gemm_f32(a.numpy(), b.numpy(), rows=None if r is None else (r, r + 1))
        assert_within("f32", got[sl], ref, S, f"simt {M}x{N}x{K}", K=K)


def run_off_simt(a, b, ldc, off):
    M, N = a.shape[0], b.shape[1]
    flat = torch.full((off + (M + 1) * ldc,), -3.0, dtype=torch.float32, device=DEV)
    c = torch.as_strided(flat, (M, N), (ldc, 1), off)
    tcl.gemm_simt_into(a, b, c)
    torch.cuda.synchronize()
    host = flat.cpu()
    inside = torch.zeros_like(host, dtype=torch.bool)
    torch.as_strided(inside, (M, N), (ldc, 1), off).fill_(True)
    assert (host[~inside] == -3.0).all(), "kernel wrote outside C"
    return torch.as_strided(host, (M, N), (ldc, 1), off).clone()


@pytest.mark.parametrize("M,N,K,lda,ldb,ldc,offs", [
    (256, 256, 256, None, None, None, (0, 0, 0)),
    (1000, 1000, 1000, None, None, None, (0, 0, 0)),     # ragged 128×128 tiles, K % 16 = 8
    (130, 261, 203, 205, 263, 263, (1, 3, 1)),           # scalar path: odd pitches and bases
    (129, 130, 17, 20, 132, 132, (0, 0, 0)),             # vector path with ragged edges
    (1, 1, 1, None, None, None, (0, 0, 0)),
])
def test_simt_f32(oracle_mod, M, N, K, lda, ldb, ldc, offs):
    simt_case(oracle_mod, M, N, K, seed=M + K, lda=lda, ldb=ldb, ldc=ldc, offs=offs)


def test_simt_f32_4096_sampled(oracle_mod):
    simt_case(oracle_mod, 4096, 4096, 4096, seed=0, rows=sample_rows(4096, n=6))


def test_pair_kernel_variants_bitwise_identical():
    a, b = inputs.bf16_pair(1024, 1280, 1216, seed=19)
    a, b = a.to(DEV), b.to(DEV)
    outs = [run(a, b, cfg=tcl.Config(cta_pair=2, stages=st, max_ctas=mc, group_m=gm, one_cta_per_tile=op),
                canary=False)
            for st in (4, 6) for (mc, gm, op) in ((0, 0, 0), (6, 3, 0), (0, 0, 1))]
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


@pytest.mark.parametrize("M,N,K,splits,out", [
    (512, 512, 4096, 0, torch.float32),        # automatic: 8 ranges
    (512, 512, 8192, 0, torch.bfloat16),       # automatic: 9 ranges, bf16 written by the reduction
    (300, 261, 1000, 3, torch.float32),        # ragged M, N (edge stored element by element), last range short
    (300, 260, 1000, 7, torch.bfloat16),
    (130, 136, 72, 2, torch.float32),          # 2 k-blocks: one per range
])
def test_bf16_split_k(oracle_mod, M, N, K, splits, out):
    cfg = tcl.Config(split_k=splits)
    assert tcl.plan(tcl.IN_BF16, 0 if out == torch.float32 else 1, M, N, K, cfg)["splits"] > 1
    bf16_case(oracle_mod, M, N, K, seed=K + splits, out_dtype=out, cfg=cfg)


def test_tf32_split_k(oracle_mod):
    a, b = inputs.tf32_pair(256, 384, 2048, seed=8)
    got = run(a.to(DEV), b.to(DEV), cfg=tcl.Config(split_k=5)).double().numpy()
    ref, S = oracle_mod.gemm_tf32(a.numpy(), b.numpy())
    assert_within("tf32", got, ref, S, "tf32 split-K")


def test_split_k_deterministic():
    a, b = inputs.bf16_pair(512, 512, 8192, seed=23)
    a, b = a.to(DEV), b.to(DEV)
    first = tcl.gemm(a, b)
    for _ in range(5):
        assert torch.equal(tcl.gemm(a, b), first)
    # the same ranges through a different grid give the same bits (fixed summation order)
    assert torch.equal(tcl.gemm(a, b, cfg=tcl.Config(split_k=9, max_ctas=40)), first)


@pytest.mark.parametrize("M,N,K,cfg", [
    (1024, 1280, 2048, dict(cta_pair=2, max_ctas=4, stream_k=1)),   # 2 pairs walk 10 tiles each
    (768, 768, 2048, dict(cta_pair=2, max_ctas=8, stream_k=2)),     # with a stream-K tail
    (700, 750, 2000, dict(cta_pair=2, max_ctas=4)),                 # ragged M, N and last k-block
    (640, 768, 1216, dict(cta_pair=1, bn=128, max_ctas=3, split_k=1)),   # one SM per tile, 10 tiles per CTA
])
def test_bf16_alternating_k_order(oracle_mod, M, N, K, cfg):
    # every second tile of a CTA's walk loads K in descending order: a different fp32
    # summation order, within the same bound, and the same bits on every run
    c = tcl.Config(k_order=2, **cfg)
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, M, N, K, c)["k_serpentine"] == 1
    ldc = up(N, 4)
    bf16_case(oracle_mod, M, N, K, seed=K + M, cfg=c, ldc=ldc)
    a, b = inputs.bf16_pair(M, N, K, seed=K + M, lda=up(K, 8), ldb=up(N, 8))
    a, b = to_dev(a), to_dev(b)
    first = run(a, b, cfg=c, ldc=ldc, canary=False)
    assert torch.equal(run(a, b, cfg=c, ldc=ldc, canary=False), first)


def test_alternating_k_order_exact_and_tf32(oracle_mod):
    # int8: each accumulation unit still holds at most 1024 products, so the int32
    # result is exact and equal to the ascending order's; TF32 within its bound
    a, b = inputs.s8_pair(1024, 1024, 2112, seed=51)
    asc = run(a.to(DEV), b.to(DEV), cfg=tcl.Config(cta_pair=2, max_ctas=4, k_order=1)).numpy()
    alt = run(a.to(DEV), b.to(DEV), cfg=tcl.Config(cta_pair=2, max_ctas=4, k_order=2)).numpy()
    assert_exact(alt, oracle_mod.gemm_s8(a.numpy(), b.numpy()), "s8 alternating K order")
    assert (asc == alt).all()
    a, b = inputs.tf32_pair(768, 1024, 1504, seed=52)
    got = run(a.to(DEV), b.to(DEV), cfg=tcl.Config(cta_pair=2, max_ctas=4, k_order=2)).double().numpy()
    ref, S = oracle_mod.gemm_tf32(a.numpy(), b.numpy())
    assert_within("tf32", got, ref, S, "tf32 alternating K order")


@pytest.mark.parametrize("kind,M,N,K,cfg", [
    ("bf16", 512, 512, 1024, dict()),                          # even k-block counts
    ("bf16", 700, 768, 1088, dict(max_ctas=4)),                 # 17 k-blocks: each tile ends on half a pair
    ("bf16", 1024, 1280, 1088, dict(max_ctas=4, k_order=2)),    # descending K walks of odd length
    ("bf16", 768, 768, 2048, dict(max_ctas=8, stream_k=3)),     # stream-K pieces of 10, 11, 11 k-blocks
    ("bf16", 768, 768, 2048, dict(max_ctas=8, stream_k=5)),     # balanced: ranges across tile boundaries
    ("bf16_out", 768, 768, 1984, dict(max_ctas=8, stream_k=3)),  # bf16 C through the workspace, 31 k-blocks
    ("tf32", 768, 1024, 1504, dict(max_ctas=4, k_order=2)),     # 47 k-blocks of 32
    ("s8", 1024, 1024, 2112, dict(max_ctas=4, k_order=2)),      # 33 k-blocks in accumulation units of 16
])
def test_two_kblocks_per_copy(oracle_mod, kind, M, N, K, cfg):
    """Two-SM 256-wide tiles with one tensor copy of each operand per two k-blocks: within the
    oracle's bound, and bit-identical to one k-block per copy (only the loads change; the MMAs
    run in the same order, also where a tile walks K downwards or ends on half a pair)."""
    two = tcl.Config(cta_pair=2, bn=256, **cfg)
    one = tcl.Config(cta_pair=2, bn=256, kblocks_per_stage=1, **cfg)
    in_kind = {"bf16": tcl.IN_BF16, "bf16_out": tcl.IN_BF16, "tf32": tcl.IN_TF32, "s8": tcl.IN_S8}[kind]
    out = {"bf16": tcl.OUT_F32, "bf16_out": tcl.OUT_BF16, "tf32": tcl.OUT_F32, "s8": 0}[kind]
    assert tcl.plan(in_kind, out, M, N, K, two)["kblocks_per_stage"] == 2
    assert tcl.plan(in_kind, out, M, N, K, one)["kblocks_per_stage"] == 1
    if kind in ("bf16", "bf16_out"):
        od = torch.float32 if kind == "bf16" else torch.bfloat16
        bf16_case(oracle_mod, M, N, K, seed=K + N, out_dtype=od, cfg=two)
        a, b = inputs.bf16_pair(M, N, K, seed=K + N)
    elif kind == "tf32":
        a, b = inputs.tf32_pair(M, N, K, seed=K + N)
        got = run(a.to(DEV), b.to(DEV), cfg=two).double().numpy()
        ref, S = oracle_mod.gemm_tf32(a.numpy(), b.numpy())
        assert_within("tf32", got, ref, S, f"tf32 two k-blocks per copy {M}x{N}x{K}")
    else:
        a, b = inputs.s8_pair(M, N, K, seed=K + N)
        assert_exact(run(a.to(DEV), b.to(DEV), cfg=two).numpy(), oracle_mod.gemm_s8(a.numpy(), b.numpy()),
                     "s8 two k-blocks per copy")
    a, b = a.to(DEV), b.to(DEV)
    od = {"bf16": None, "bf16_out": torch.bfloat16, "tf32": None, "s8": None}[kind]
    x = run(a, b, out_dtype=od, cfg=two, canary=False)
    y = run(a, b, out_dtype=od, cfg=one, canary=False)
    assert torch.equal(x, y)


@pytest.mark.parametrize("kind,M,N,K,cfg", [
    ("bf16", 700, 768, 1000, dict(cta_pair=1, bn=256)),               # 4 boxes in one copy; K tail, ragged M
    ("bf16", 640, 1024, 1216, dict(cta_pair=1, bn=128, split_k=2)),   # 2 boxes; split-K ranges
    ("bf16_out", 520, 512, 960, dict(cta_pair=1, bn=256)),
    ("tf32", 384, 512, 1000, dict(cta_pair=1, bn=256)),               # 8 boxes of 32 columns in one copy
    ("tf32", 512, 768, 1504, dict(cta_pair=1, bn=128, max_ctas=4)),
    ("s8", 640, 512, 1000, dict(cta_pair=1, bn=128, max_ctas=4)),
    ("bf16", 768, 768, 1000, dict(cta_pair=2, bn=256, max_ctas=8)),   # two-SM, K not whole k-blocks
])
def test_b_boxes_in_one_copy(oracle_mod, kind, M, N, K, cfg):
    """A CTA's B boxes of a k-block in one 3-D tensor copy (the default where N is whole boxes)
    against one copy per box: within the oracle's bound and bit-identical."""
    auto, per_box = tcl.Config(**cfg), tcl.Config(b_copy=1, **cfg)
    in_kind = {"bf16": tcl.IN_BF16, "bf16_out": tcl.IN_BF16, "tf32": tcl.IN_TF32, "s8": tcl.IN_S8}[kind]
    out = {"bf16": tcl.OUT_F32, "bf16_out": tcl.OUT_BF16, "tf32": tcl.OUT_F32, "s8": 0}[kind]
    assert tcl.plan(in_kind, out, M, N, K, auto)["kblocks_per_stage"] == 1
    if kind in ("bf16", "bf16_out"):
        od = torch.float32 if kind == "bf16" else torch.bfloat16
        bf16_case(oracle_mod, M, N, K, seed=K + N + 1, out_dtype=od, cfg=auto)
        a, b = inputs.bf16_pair(M, N, K, seed=K + N + 1)
    elif kind == "tf32":
        a, b = inputs.tf32_pair(M, N, K, seed=K + N + 1)
        got = run(a.to(DEV), b.to(DEV), cfg=auto).double().numpy()
        ref, S = oracle_mod.gemm_tf32(a.numpy(), b.numpy())
        assert_within("tf32", got, ref, S, f"tf32 B boxes in one copy {M}x{N}x{K}")
    else:
        a, b = inputs.s8_pair(M, N, K, seed=K + N + 1)
        assert_exact(run(a.to(DEV), b.to(DEV), cfg=auto).numpy(), oracle_mod.gemm_s8(a.numpy(), b.numpy()),
                     "s8 B boxes in one copy")
    a, b = a.to(DEV), b.to(DEV)
    od = torch.bfloat16 if kind == "bf16_out" else None
    assert torch.equal(run(a, b, out_dtype=od, cfg=auto, canary=False),
                       run(a, b, out_dtype=od, cfg=per_box, canary=False))


def test_die_map_measured():
    # the two dies of a GB300 each hold half of its pairs of SMs
    n0, n1 = tcl.die_pairs()
    assert n0 > 0 and n1 > 0 and n0 + n1 == tcl.num_sms() // 2, (n0, n1)


@pytest.mark.parametrize("kind,M,N,K,extra", [
    ("bf16", 2304, 4096, 2048, dict()),                 # 9 × 8 tiles per die on ~38 pairs, no tail
    ("bf16", 4096, 4096, 2048, dict()),                 # a stream-K tail on each die
    ("bf16", 4000, 3968, 2040, dict()),                 # ragged M, N and last k-block
    ("bf16_out", 4096, 4096, 2048, dict()),             # bf16 C: tail pieces through the fp32 workspace
    ("tf32", 4096, 3072, 1024, dict()),
    ("s8", 4096, 4096, 2048, dict()),                   # exact integers
    ("bf16", 4096, 4096, 2048, dict(k_order=2)),        # alternating K order
    ("bf16", 4096, 4096, 8192, dict()),                 # deep: L2 eviction hints on A and B too
])
def test_die_split(oracle_mod, kind, M, N, K, extra):
    """Each die's pairs walk their own block of tile columns: within the oracle's bound on
    sampled rows (and exact for int8)."""
    cfg = tcl.Config(cta_pair=2, die_split=2, **extra)
    in_kind = {"bf16": tcl.IN_BF16, "bf16_out": tcl.IN_BF16, "tf32": tcl.IN_TF32, "s8": tcl.IN_S8}[kind]
    out = tcl.OUT_BF16 if kind == "bf16_out" else tcl.OUT_F32
    assert tcl.plan(in_kind, out, M, N, K, cfg)["die_split"] == 1
    rows = sample_rows(M, n=12, seed=M + K)
    if kind in ("bf16", "bf16_out"):
        bf16_case(oracle_mod, M, N, K, seed=K + 7, out_dtype=torch.bfloat16 if kind == "bf16_out" else torch.float32,
                  cfg=cfg, ldc=up(N, 8), rows=rows)
    elif kind == "tf32":
        a, b = inputs.tf32_pair(M, N, K, seed=K + 7)
        got = run(a.to(DEV), b.to(DEV), cfg=cfg).double().numpy()
        for r in rows:
            ref, S = oracle_mod.gemm_tf32(a.numpy(), b.numpy(), rows=(r, r + 1))
            assert_within("tf32", got[r:r + 1], ref, S, f"tf32 die split row {r}")
    else:
        a, b = inputs.s8_pair(M, N, K, seed=K + 7)
        got = run(a.to(DEV), b.to(DEV), cfg=cfg).numpy()
        for r in rows:
            assert_exact(got[r:r + 1], oracle_mod.gemm_s8(a.numpy(), b.numpy(), rows=(r, r + 1)), f"s8 row {r}")
    assert tcl.last_device_error() == (0, 0)


def test_l2_hints_change_nothing_in_the_result():
    # the eviction priorities on A's and B's loads only steer the L2: the same bits
    a, b = inputs.bf16_pair(4096, 4096, 8192, seed=41)
    a, b = a.to(DEV), b.to(DEV)
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 8192, None)["l2_hints"] == 1
    x = run(a, b, cfg=tcl.Config(l2_hints=2), canary=False)
    y = run(a, b, cfg=tcl.Config(l2_hints=1), canary=False)
    assert torch.equal(x, y)
    assert tcl.last_device_error() == (0, 0)


@pytest.mark.parametrize("N", [4096, 3840])
def test_die_split_whole_tiles_bitwise_and_replays(N):
    """Whole tiles in ascending K: the die split changes which pair computes a tile, not
    how, so the bits are those of the plain walk (every tile computed once: with 15 tile
    columns the dies' blocks meet inside a column whatever their pairs); and the rank
    counters are zero again after every launch (CUDA graph replays and back-to-back calls
    stay exact)."""
    a, b = inputs.bf16_pair(4096, N, 1024, seed=31)
    a, b = a.to(DEV), b.to(DEV)
    base = dict(cta_pair=2, stream_k=1, k_order=1)
    plain = run(a, b, cfg=tcl.Config(die_split=1, **base), canary=False)
    split_cfg = tcl.Config(die_split=2, **base)
    pl = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, N, 1024, split_cfg)
    assert pl["die_split"] == 1 and 0 < pl["die_tiles0"] < pl["num_tiles"]
    for _ in range(3):
        assert torch.equal(run(a, b, cfg=split_cfg, canary=False), plain)
    c = torch.empty((4096, N), dtype=torch.float32, device=DEV)
    tcl.gemm_into(a, b, c, cfg=split_cfg)   # scratch in place before capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=side):
        for _ in range(3):
            tcl.gemm_into(a, b, c, cfg=split_cfg)
    for _ in range(4):
        c.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(c.cpu(), plain)
    assert tcl.last_device_error() == (0, 0)


def test_variants_bitwise_identical():
    """Pipelining only reorders loads: every ring depth, persistent or one CTA per
    tile, gives the same bits (the MMA order inside a tile does not change)."""
    a, b = inputs.bf16_pair(640, 768, 1216, seed=13)
    a, b = a.to(DEV), b.to(DEV)
    for bn, stages_list in ((256, (1, 2, 3, 4)), (128, (1, 2, 4, 6))):
        outs = []
        for st in stages_list:
            for one_per_tile in (0, 1):
                for max_ctas in (0, 3):
                    cfg = tcl.Config(bn=bn, stages=st, one_cta_per_tile=one_per_tile, max_ctas=max_ctas,
                                     group_m=3 if max_ctas else 0, split_k=1)
                    outs.append(run(a, b, cfg=cfg, canary=False))
        if bn == 256:   # the synchronous and cp.async producers feed the same MMA sequence
            for st in (1, 2, 4):
                outs.append(run(a, b, cfg=tcl.Config(bn=256, stages=st, producer=1, split_k=1), canary=False))
            for st in (1, 2, 3, 4):
                outs.append(run(a, b, cfg=tcl.Config(bn=256, stages=st, producer=tcl.PRODUCER_CPASYNC, split_k=1),
                                canary=False))
        for o in outs[1:]:
            assert torch.equal(o, outs[0])


@pytest.mark.parametrize("M,N,K,lda,ldb,ldc,out", [
    (4096, 4096, 4096, 4096, 4096, 4096, torch.float32),    # eight row chunks, sampled rows
    (1536, 2100, 520, 520, 2104, 2100, torch.float32),      # three chunks of 512 rows, unpadded host C
    (1100, 2304, 96, 96, 2304, 2312, torch.bfloat16),       # chunks of 768 and 332 rows, bf16 C
    (1000, 777, 203, 205, 779, 780, torch.float32),         # K % 8 = 3 (zero-padded on the device), ragged
    (1000, 520, 640, 640, 520, 528, torch.bfloat16),        # two chunks, bf16 C
    (100, 64, 64, 64, 64, 64, torch.float32),               # one chunk
])
def test_host_buffer_entry_point(oracle_mod, M, N, K, lda, ldb, ldc, out):
    # A, B, C in page-locked host memory; uploads, GEMMs and downloads pipelined
    a, b = inputs.bf16_pair(M, N, K, seed=M + K, lda=lda, ldb=ldb)
    ah = torch.as_strided(a, (M, lda), (lda, 1)).pin_memory()[:, :K] if lda != K else a.pin_memory()
    bh = torch.as_strided(b, (K, ldb), (ldb, 1)).pin_memory()[:, :N] if ldb != N else b.pin_memory()
    sentinel = -3.0
    full = torch.full((M + 1, ldc), sentinel, dtype=out).pin_memory()
    c = full[:M, :N]
    side = torch.cuda.Stream()
    tcl.gemm_host_into(ah, bh, c, stream=side)
    side.synchronize()
    assert (full[:M, N:] == sentinel).all() and (full[M] == sentinel).all(), "wrote outside C"
    got = c.double().numpy()
    kind = "bf16_f32" if out == torch.float32 else "bf16_bf16"
    rows = sample_rows(M, n=8) if M >= 4096 else None
    if rows is None:
        ref, S = oracle_mod.gemm_bf16(inputs.bf16_bits(a), inputs.bf16_bits(b))
        assert_within(kind, got, ref, S, f"host {M}x{N}x{K}")
    else:
        for r in rows:
            ref, S = oracle_mod.gemm_bf16(inputs.bf16_bits(a), inputs.bf16_bits(b), rows=(r, r + 1))
            assert_within(kind, got[r:r + 1], ref, S, f"host {M}x{N}x{K} row {r}")


def test_repeat_runs_bitwise_identical():
    a, b = inputs.bf16_pair(1024, 1024, 2048, seed=17)
    a, b = a.to(DEV), b.to(DEV)
    first = tcl.gemm(a, b)
    for _ in range(10):
        assert torch.equal(tcl.gemm(a, b), first)


# ------------------------------------------------------------- tf32 and int8, small

@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (130, 260, 200), (64, 40, 36)])
def test_tf32_small(oracle_mod, M, N, K):
    a, b = inputs.tf32_pair(M, N, K, seed=M, lda=up(K, 4), ldb=up(N, 4))
    got = run(to_dev(a), to_dev(b)).double().numpy()
    ref, S = oracle_mod.gemm_tf32(a.numpy(), b.numpy())
    assert_within("tf32", got, ref, S, f"tf32 {M}x{N}x{K}")


@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("M,N,K,split", [(512, 512, 256, 1), (512, 512, 1024, 1), (300, 200, 520, 1),
                                         (512, 512, 2048, 4), (130, 72, 64, 1)])
def test_bf16_64_wide_tiles(oracle_mod, out, M, N, K, split):
    # 64-wide one-SM tiles (one B box per stage, 8 stages), with and without split-K;
    # ragged right edges inside the single 64-column box
    cfg = tcl.Config(bn=64, split_k=split, cluster_k=1)
    pl = tcl.plan(tcl.IN_BF16, tcl.OUT_F32 if out == torch.float32 else tcl.OUT_BF16, M, N, K, cfg)
    assert pl["bn"] == 64 and pl["cta_pair"] == 1 and pl["splits"] == split and pl["cluster_k"] == 1
    ldc = up(N, 4 if out == torch.float32 else 8)
    bf16_case(oracle_mod, M, N, K, seed=M + N + K, out_dtype=out, cfg=cfg, ldc=ldc)


@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("M,N,K", [(64, 64, 64), (512, 512, 256), (300, 200, 520), (130, 72, 64),
                                   (1000, 130, 1000), (768, 768, 1024), (200, 136, 2064), (200, 136, 192)])
def test_bf16_64_row_tiles(oracle_mod, out, M, N, K):
    # 64×64 tiles (tcgen05.mma with M = 64: the accumulator in lanes 0-15 of each TMEM lane
    # quarter), C stored from registers: ragged M, N (a partial last column tile stored
    # element by element) and K; K a multiple of 64 takes two k-blocks per stage (a 3-D map
    # of A), an odd count of them leaving the last stage's second k-block to zero fill;
    # the canaries around C catch any store outside it
    cfg = tcl.Config(tile_m=64)
    pl = tcl.plan(tcl.IN_BF16, tcl.OUT_F32 if out == torch.float32 else tcl.OUT_BF16, M, N, K, cfg)
    assert (pl["tile_m"], pl["bn"], pl["splits"], pl["cta_pair"]) == (64, 64, 1, 1)
    assert pl["grid"] == pl["num_tiles"] == ((M + 63) // 64) * ((N + 63) // 64)
    ldc = up(N, 4 if out == torch.float32 else 8)
    bf16_case(oracle_mod, M, N, K, seed=M + N + K + 64, out_dtype=out, cfg=cfg, ldc=ldc)


def test_bf16_64_row_tiles_chosen_and_exact_match():
    # the planner's choice for a small shallow grid; the same sums as 128×64 tiles (each
    # output element's K order is the same MMA sequence), so the results agree closely
    a, b = inputs.bf16_pair(512, 512, 512, seed=9)
    a, b = a.to(DEV), b.to(DEV)
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 512, 512, 512)["tile_m"] == 64
    x = tcl.gemm(a, b)
    y = tcl.gemm(a, b, cfg=tcl.Config(tile_m=128))
    assert torch.allclose(x, y, rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("cl", [2, 4])
@pytest.mark.parametrize("M,N,K", [(512, 512, 256), (512, 512, 1024), (300, 200, 520), (130, 72, 64),
                                   (256, 136, 2000), (1000, 130, 1000)])
def test_bf16_cluster_k(oracle_mod, out, cl, M, N, K):
    # each 128×64 tile on a cluster of `cl` CTAs, one K range each, summed through
    # distributed shared memory in rank order; ragged M, N and K, and at K = 64 (one
    # k-block) the ranges of all but one CTA are empty
    cfg = tcl.Config(cluster_k=cl)
    pl = tcl.plan(tcl.IN_BF16, tcl.OUT_F32 if out == torch.float32 else tcl.OUT_BF16, M, N, K, cfg)
    assert (pl["cluster_k"], pl["bn"], pl["splits"]) == (cl, 64, 1)
    assert pl["grid"] == cl * pl["num_tiles"]
    ldc = up(N, 4 if out == torch.float32 else 8)
    bf16_case(oracle_mod, M, N, K, seed=M + N + K + cl, out_dtype=out, cfg=cfg, ldc=ldc)


def test_bf16_cluster_k_deterministic():
    # the partials are added in a fixed order, so every run gives the same bits
    a, b = inputs.bf16_pair(512, 512, 512, seed=5)
    a, b = a.to(DEV), b.to(DEV)
    cfg = tcl.Config(cluster_k=4)
    first = tcl.gemm(a, b, cfg=cfg)
    for _ in range(20):
        assert torch.equal(tcl.gemm(a, b, cfg=cfg), first)
    one = tcl.gemm(a, b)   # one CTA per tile: another summation order
    assert torch.allclose(one, first, rtol=1e-5, atol=1e-3)


@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("M,N,K", [(256, 512, 1004), (200, 300, 96), (384, 264, 32)])
def test_tf32_one_sm_kernel(oracle_mod, bn, M, N, K):
    # TF32 on one SM per tile with B read N-major in place: boxes of 32 columns, the last
    # one ragged (N % 32 != 0) or past N, K ragged within the last 32-deep k-block
    a, b = inputs.tf32_pair(M, N, K, seed=M + K + bn)
    cfg = tcl.Config(cta_pair=1, bn=bn, split_k=1)
    assert tcl.plan(tcl.IN_TF32, 0, M, N, K, cfg)["cta_pair"] == 1
    got = run(a.to(DEV), b.to(DEV), cfg=cfg, ldc=up(N, 4)).double().numpy()
    ref, S = oracle_mod.gemm_tf32(a.numpy(), b.numpy())
    assert_within("tf32", got, ref, S, f"tf32 one SM bn {bn} {M}x{N}x{K}")


def test_tf32_padded(oracle_mod):
    a, b = inputs.tf32_pair(100, 96, 52, seed=4, lda=56, ldb=100)
    got = run(to_dev(a), to_dev(b), ldc=100).double().numpy()
    ref, S = oracle_mod.gemm_tf32(a.numpy(), b.numpy())
    assert_within("tf32", got, ref, S, "tf32 padded")


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (130, 260, 208), (64, 40, 1040), (200, 136, 2064)])
def test_s8_small_exact(oracle_mod, M, N, K):
    a, b = inputs.s8_pair(M, N, K, seed=M, lda=up(K, 16), ldb=up(N, 16))
    got = run(to_dev(a), to_dev(b)).numpy()
    assert_exact(got, oracle_mod.gemm_s8(a.numpy(), b.numpy()), f"s8 {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(33, 45, 37), (128, 130, 1029), (5, 3, 1)])
def test_s8_ragged_k_exact(oracle_mod, M, N, K):
    # int8 K need not keep the 16-byte grid: the operands are repacked with zero padding
    a, b = inputs.s8_pair(M, N, K, seed=K, lda=up(K, 16), ldb=up(N, 16))
    got = run(to_dev(a), to_dev(b)).numpy()
    assert_exact(got, oracle_mod.gemm_s8(a.numpy(), b.numpy()), f"s8 {M}x{N}x{K}")


def test_s8_padded(oracle_mod):
    a, b = inputs.s8_pair(100, 90, 70, seed=8, lda=80, ldb=96)
    got = run(to_dev(a), to_dev(b), ldc=92).numpy()
    assert_exact(got, oracle_mod.gemm_s8(a.numpy(), b.numpy()), "s8 padded")


@pytest.mark.parametrize("pair,bn,sk", [(1, 0, 1), (2, 128, 1), (2, 256, 1), (2, 256, 3)])
@pytest.mark.parametrize("va,vb", [(127, 127), (-128, -128), (127, -128)])
def test_s8_extremes_closed_form(va, vb, pair, bn, sk):
    # |sum| = 2^26 at K = 4096: four fp32 units of 1024 products each (exactly 2^24 apiece
    # for (-128)·(-128)), added as int32
    # (sk = 3: 1280 columns of 256 on four pairs, the 5th tile in three K pieces)
    K = 4096
    a = torch.full((256, K), va, dtype=torch.int8, device=DEV)
    b = torch.full((K, 1280 if sk > 1 else 512), vb, dtype=torch.int8, device=DEV)
    cfg = tcl.Config(cta_pair=pair, bn=bn, stream_k=sk, max_ctas=8 if sk > 1 else 0)
    c = tcl.gemm(a, b, cfg=cfg)
    assert (c == va * vb * K).all()


@pytest.mark.parametrize("pair,bn", [(1, 0), (2, 256)])
@pytest.mark.parametrize("K", [1024, 4096, 3000])
def test_s8_odd_sums_near_2_24(K, pair, bn):
    # rows and columns of -128 that end in 127: every 1024-deep unit but the last sums to
    # exactly 2^24, the last to (n-1)·2^14 + 127² — odd, just below 2^24 when n = 1024
    a = torch.full((256, K), -128, dtype=torch.int8, device=DEV)
    b = torch.full((K, 256), -128, dtype=torch.int8, device=DEV)
    a[:, K - 1] = 127
    b[K - 1, :] = 127
    c = tcl.gemm(a, b, cfg=tcl.Config(cta_pair=pair, bn=bn))
    assert (c == (K - 1) * 16384 + 127 * 127).all()


@pytest.mark.parametrize("va,vb", [(-128, -128), (127, -128)])
def test_s8_largest_k_closed_form(va, vb):
    # K = 131071, the largest the int32 result guarantees: |sum| up to 2^14·131071 < 2^31;
    # 128 accumulation units of 1024 K values, all added in int32 registers
    K = 131071
    a = torch.full((130, K), va, dtype=torch.int8, device=DEV)
    b = torch.full((K, 72), vb, dtype=torch.int8, device=DEV)
    c = tcl.gemm(a, b)
    assert (c == va * vb * K).all()
    with pytest.raises(tcl.TclError):
        tcl.gemm(torch.ones((8, K + 1), dtype=torch.int8, device=DEV), torch.ones((K + 1, 8), dtype=torch.int8, device=DEV))


@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("M,N,K", [(256, 128, 64), (512, 384, 4096), (300, 200, 1100), (520, 390, 2064),
                                   (1000, 700, 520)])
def test_s8_pair_kernel_exact(oracle_mod, M, N, K, bn):
    # two SMs per 256×bn tile (bn = 256: eight epilogue warps, two per TMEM lane quarter);
    # K ranges that end inside a 512-deep unit and ragged M, N edges
    a, b = inputs.s8_pair(M, N, K, seed=M + N, lda=up(K, 16), ldb=up(N, 16))
    got = run(to_dev(a), to_dev(b), cfg=tcl.Config(cta_pair=2, bn=bn)).numpy()
    assert_exact(got, oracle_mod.gemm_s8(a.numpy(), b.numpy()), f"s8 pair {M}x{N}x{K} bn {bn}")


@pytest.mark.parametrize("bn,M,N,K,pieces", [
    (256, 768, 768, 2048, 0),    # 9 tiles on 4 pairs: the 9th in 4 pieces of 8 k-blocks (one unit each)
    (256, 768, 768, 2048, 3),    # pieces of 10, 11, 11 k-blocks: units end inside a piece
    (256, 700, 750, 1000, 4),    # ragged M, N (the last chunk added element by element), K tail in the last piece
    (256, 512, 1280, 4160, 2),   # pieces of 32 and 33 k-blocks, units of 8 and a ragged last one
    (128, 768, 768, 2048, 0),    # 18 tiles on 4 pairs: two tail tiles in 2 pieces each
    (128, 700, 750, 1000, 2),
    (128, 512, 1152, 4160, 2),
])
def test_s8_pair_stream_k_exact(oracle_mod, M, N, K, pieces, bn):
    # the last partial wave of tiles in K pieces; later pieces add their int32 sums into C
    cfg = tcl.Config(cta_pair=2, bn=bn, max_ctas=8, stream_k=pieces)
    pl = tcl.plan(tcl.IN_S8, 0, M, N, K, cfg)
    assert pl["sk_tiles"] > 0 and pl["sk_pieces"] >= 2
    a, b = inputs.s8_pair(M, N, K, seed=K + pieces, lda=up(K, 16), ldb=up(N, 16))
    got = run(to_dev(a), to_dev(b), cfg=cfg).numpy()
    assert_exact(got, oracle_mod.gemm_s8(a.numpy(), b.numpy()), f"s8 stream-K {M}x{N}x{K} bn {bn}")


@pytest.mark.parametrize("M,N,K,extra", [
    (512, 384, 4096, {}),
    (300, 200, 1100, {}),                            # K % 16 = 12 and N % 16 = 8: chunks cut by the row ends
    (1000, 700, 520, {}),                            # 520 = 8 k-blocks + 8: a ragged last k-block
    (700, 750, 1000, dict(max_ctas=8, stream_k=4)),  # stream-K pieces, ragged M and N
    (768, 1024, 1536, dict(max_ctas=8)),             # 4 pairs walk 3 tiles each
    (1024, 1024, 2112, dict(max_ctas=4, k_order=2)), # alternating K order
])
def test_s8_in_kernel_widening_exact(oracle_mod, M, N, K, extra):
    # the two-SM kernel that widens int8 to fp16 itself (converter warps, no scratch) against
    # the oracle and against the widening pass (bf16 copies in scratch), bit for bit
    a, b = inputs.s8_pair(M, N, K, seed=M + K, lda=up(K, 16), ldb=up(N, 16))
    ref = oracle_mod.gemm_s8(a.numpy(), b.numpy())
    outs = {}
    for path in (2, 1):
        cfg = tcl.Config(cta_pair=2, bn=256, s8_path=path, **extra)
        assert tcl.plan(tcl.IN_S8, 0, M, N, K, cfg)["s8_in_kernel"] == (1 if path == 2 else 0)
        outs[path] = run(to_dev(a), to_dev(b), cfg=cfg).numpy()
        assert_exact(outs[path], ref, f"s8 {M}x{N}x{K} path {path}")
    assert (outs[1] == outs[2]).all()


def test_s8_in_kernel_needs_aligned_rows(oracle_mod):
    # rows of A off the 16-byte grid: the in-kernel widening (its tensor copies need 16-byte
    # rows) is refused, the automatic path (the widening pass) is exact
    a, b = inputs.s8_pair(600, 520, 1000, seed=3, lda=1001, ldb=528)
    ad, bd = to_dev(a), to_dev(b)
    got = run(ad, bd, cfg=tcl.Config(cta_pair=2, bn=256)).numpy()
    assert_exact(got, oracle_mod.gemm_s8(a.numpy(), b.numpy()), "s8 unaligned rows, automatic path")
    c = torch.empty((600, 520), dtype=torch.int32, device=DEV)
    with pytest.raises(tcl.TclError):
        tcl.gemm_into(ad, bd, c, cfg=tcl.Config(cta_pair=2, bn=256, s8_path=2))


@pytest.mark.parametrize("bn", [128, 256])
def test_s8_pair_kernel_grid_smaller_than_tiles(oracle_mod, bn):
    # 4 pairs walk more tiles than they are: each pair's accumulator units cycle through both
    # TMEM buffers and its epilogue stores several tiles
    a, b = inputs.s8_pair(768, 1024, 1536, seed=11, lda=1536, ldb=1024)
    got = run(to_dev(a), to_dev(b), cfg=tcl.Config(cta_pair=2, bn=bn, max_ctas=8)).numpy()
    assert_exact(got, oracle_mod.gemm_s8(a.numpy(), b.numpy()), f"s8 pair bn {bn}, 4 pairs")


# ------------------------------------------------------------- full-size workloads, sampled

def test_bf16_4096_cube_fp32_sampled(oracle_mod):
    bf16_case(oracle_mod, 4096, 4096, 4096, seed=0, rows=sample_rows(4096))


def test_bf16_large_grid_sampled(oracle_mod):
    # 16384×16384×4096: 4096 pair tiles, 54 waves on 76 pairs (the last one 68 tiles); a 1 GB
    # fp32 C compared on sampled rows that cross every column of tiles
    M = N = 16384
    pl = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, M, N, 4096)
    assert pl["cta_pair"] == 2 and pl["num_tiles"] == 64 * 64
    bf16_case(oracle_mod, M, N, 4096, seed=7, rows=sample_rows(M, n=8, seed=7))


def test_bf16_4096_cube_bf16_sampled(oracle_mod):
    bf16_case(oracle_mod, 4096, 4096, 4096, seed=0, out_dtype=torch.bfloat16, rows=sample_rows(4096, n=8))


@pytest.mark.parametrize("MN", [512, 4096])
@pytest.mark.parametrize("K", [256, 512, 1024, 4096, 8192])
def test_bf16_k_sweep_sampled(oracle_mod, MN, K):
    rows = list(range(MN)) if MN == 512 and K <= 1024 else sample_rows(MN, n=6, seed=K)
    bf16_case(oracle_mod, MN, MN, K, seed=0, rows=rows)


def test_s8_4096_cube_sampled_exact(oracle_mod):
    a, b = inputs.s8_pair(4096, 4096, 4096, seed=0)
    got = run(a.to(DEV), b.to(DEV)).numpy()
    rows = sample_rows(4096, n=10)
    for r in rows:
        assert_exact(got[r:r + 1], oracle_mod.gemm_s8(a.numpy(), b.numpy(), rows=(r, r + 1)), f"s8 row {r}")


def test_tf32_4096_cube_sampled(oracle_mod):
    a, b = inputs.tf32_pair(4096, 4096, 4096, seed=0)
    got = run(a.to(DEV), b.to(DEV)).double().numpy()
    for r in sample_rows(4096, n=8):
        ref, S = oracle_mod.gemm_tf32(a.numpy(), b.numpy(), rows=(r, r + 1))
        assert_within("tf32", got[r:r + 1], ref, S, f"tf32 row {r}")
