"""Failure detection on the GPU without a fault: every wait in the kernels is
bounded. Test hooks make CTA 0's producer skip one k-block (the MMA warp waits
for data that never arrives) or hold back a stream-K piece's hand-over (the
next piece waits for a flag that nothing sets); the wait must run out, record
the code in the device status word, let the kernel return, and leave the
context usable for the next call."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import tensor_core_loop_gb300 as tcl
from tensor_core_loop_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tcl.lib()
    tcl.last_device_error()   # start from a clear status word


def test_bounded_wait_runs_out_and_context_survives():
    a, b = inputs.bf16_pair(1024, 1024, 1024, seed=3)
    a, b = a.to(DEV), b.to(DEV)
    c = torch.zeros((1024, 1024), dtype=torch.float32, device=DEV)
    cfg = tcl.Config(timeout_ns=50_000_000, debug_skip_kblock=3)
    tcl.gemm_into(a, b, c, cfg=cfg)              # the launch itself succeeds
    st, code = tcl.last_device_error()
    assert st == 7, f"expected TCL_ERR_DEVICE_TIMEOUT, got {tcl.STATUS.get(st, st)}"
    assert code in (1, 2, 3, 4)                  # which role gave up first
    assert tcl.last_device_error() == (0, 0)     # reading clears the word
    # the context is still usable and the next call is correct
    ref = tcl.gemm(a, b)
    again = tcl.gemm(a, b)
    torch.cuda.synchronize()
    assert torch.equal(ref, again)
    assert tcl.last_device_error() == (0, 0)


@pytest.mark.parametrize("kps,skip", [(1, 2), (2, 2), (2, 3)])
def test_two_sm_kernel_bounded_wait_runs_out(kps, skip):
    # CTA 0 of the first pair announces a stage's bytes but never loads its share (with two
    # k-blocks per copy: the pair of ring slots holding that k-block): the leader's MMA wait
    # runs out; both CTAs of the pair abort and return
    a, b = inputs.bf16_pair(1024, 1024, 1024, seed=5)
    a, b = a.to(DEV), b.to(DEV)
    c = torch.zeros((1024, 1024), dtype=torch.float32, device=DEV)
    cfg = tcl.Config(cta_pair=2, bn=256, kblocks_per_stage=kps, timeout_ns=50_000_000, debug_skip_kblock=skip)
    tcl.gemm_into(a, b, c, cfg=cfg)
    st, code = tcl.last_device_error()
    assert st == 7 and code in (1, 2, 3, 4), (st, code)
    ref = tcl.gemm(a, b, cfg=tcl.Config(cta_pair=2))
    again = tcl.gemm(a, b)
    torch.cuda.synchronize()
    assert torch.allclose(ref, again, rtol=0, atol=1e-2)   # both correct (different plans)
    assert tcl.last_device_error() == (0, 0)


def test_die_split_bounded_wait_runs_out_and_counters_reset():
    # under the die split CTA 0 skips a k-block: the wait runs out, every pair still reaches
    # the end (the last one zeroes the rank counters), and the next calls are exact
    a, b = inputs.bf16_pair(4096, 4096, 2048, seed=12)
    a, b = a.to(DEV), b.to(DEV)
    c = torch.zeros((4096, 4096), dtype=torch.float32, device=DEV)
    base = dict(cta_pair=2, die_split=2, stream_k=1, k_order=1)
    tcl.gemm_into(a, b, c, cfg=tcl.Config(timeout_ns=50_000_000, debug_skip_kblock=3, **base))
    st, code = tcl.last_device_error()
    assert st == 7 and code in (1, 2, 3, 4), (st, code)
    x = tcl.gemm(a, b, cfg=tcl.Config(**base))
    y = tcl.gemm(a, b, cfg=tcl.Config(cta_pair=2, die_split=1, stream_k=1, k_order=1))
    torch.cuda.synchronize()
    assert torch.equal(x, y)
    assert tcl.last_device_error() == (0, 0)


@pytest.mark.parametrize("sk,split", [(2, 1), (5, 3)])
def test_stream_k_order_wait_runs_out(sk, split):
    # the first piece of split tile 0 (balanced: of the tile cut by the first range boundary)
    # never hands over: the last piece's wait for it (the last unit of its pair, so nothing
    # else is waiting) runs out with code 5
    a, b = inputs.bf16_pair(768, 768, 2048, seed=6)
    a, b = a.to(DEV), b.to(DEV)
    c = torch.zeros((768, 768), dtype=torch.float32, device=DEV)
    base = dict(cta_pair=2, max_ctas=8, stream_k=sk)
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 768, 768, 2048, tcl.Config(**base))["sk_tiles"] == split
    tcl.gemm_into(a, b, c, cfg=tcl.Config(timeout_ns=50_000_000, debug_stream_k_stall=1, **base))
    st, code = tcl.last_device_error()
    assert (st, code) == (7, 5), (st, code)
    # the next stream-K call (a new flag generation) is correct
    x = tcl.gemm(a, b, cfg=tcl.Config(**base))
    y = tcl.gemm(a, b, cfg=tcl.Config(**base))
    torch.cuda.synchronize()
    assert torch.equal(x, y)
    assert tcl.last_device_error() == (0, 0)


def test_stream_k_order_wait_runs_out_int8():
    # the same hold in the exact-integer epilogue (eight warps per CTA, int32 pieces)
    a = torch.randint(-128, 128, (768, 2048), dtype=torch.int8, generator=torch.Generator().manual_seed(8)).to(DEV)
    b = torch.randint(-128, 128, (2048, 768), dtype=torch.int8, generator=torch.Generator().manual_seed(9)).to(DEV)
    c = torch.zeros((768, 768), dtype=torch.int32, device=DEV)
    base = dict(cta_pair=2, bn=256, max_ctas=8, stream_k=2)
    assert tcl.plan(tcl.IN_S8, 0, 768, 768, 2048, tcl.Config(**base))["sk_tiles"] == 1
    tcl.gemm_into(a, b, c, cfg=tcl.Config(timeout_ns=50_000_000, debug_stream_k_stall=1, **base))
    st, code = tcl.last_device_error()
    assert (st, code) == (7, 5), (st, code)
    x = tcl.gemm(a, b, cfg=tcl.Config(**base))
    y = tcl.gemm(a, b, cfg=tcl.Config(cta_pair=1))
    torch.cuda.synchronize()
    assert torch.equal(x, y)
    assert tcl.last_device_error() == (0, 0)


@pytest.mark.parametrize("pair", [1, 2])
def test_trace_shows_loads_ahead_of_mma(pair):
    """The per-k-block timeline of CTA 0: each block's load is issued before its
    data lands, the MMAs are issued after, and the loads of later blocks are in
    flight while earlier blocks' MMAs run (the software pipeline)."""
    M, N, K = 128 * pair, 256, 64 * 48
    a, b = inputs.bf16_pair(M, N, K, seed=4)
    a, b = a.to(DEV), b.to(DEV)
    cap = 48
    trace = torch.zeros(4 * cap + 4, dtype=torch.int64, device=DEV)
    cfg = tcl.Config(bn=256, stages=4, cta_pair=pair, split_k=1, trace=trace.data_ptr(), trace_cap=cap)
    c = tcl.gemm(a, b, cfg=cfg)
    torch.cuda.synchronize()
    t = trace[:4 * cap].view(cap, 4).cpu().numpy().astype(np.int64)
    issued, landed, mma, done = t[:, 0], t[:, 1], t[:, 2], t[:, 3]
    assert (issued > 0).all() and (landed > 0).all() and (mma > 0).all()
    assert (landed >= issued).all() and (mma >= landed).all()
    n = cap - 4   # the last ring's worth of blocks has no later reuse to stamp "done"
    assert (done[:n] >= mma[:n]).all()
    # load of block k+1 issued before MMA of block k completed: overlap
    overlap = (issued[1:n + 1] < done[:n]).mean()
    assert overlap > 0.9, overlap
    # tracing changes nothing in the result
    ref = tcl.gemm(a, b, cfg=tcl.Config(bn=256, stages=4, cta_pair=pair, split_k=1))
    assert torch.equal(c, ref)


def test_cluster_k_bounded_wait_runs_out():
    # CTA 0 of the first cluster never loads one of its k-blocks: its MMA warp's bounded
    # wait runs out, every CTA still reaches both cluster barriers and returns, and the
    # next call on the device is correct
    a, b = inputs.bf16_pair(512, 512, 1024, seed=7)
    a, b = a.to(DEV), b.to(DEV)
    c = torch.zeros((512, 512), dtype=torch.float32, device=DEV)
    tcl.gemm_into(a, b, c, cfg=tcl.Config(cluster_k=4, timeout_ns=50_000_000, debug_skip_kblock=2))
    st, code = tcl.last_device_error()
    assert st == 7 and code in (1, 2, 4), (st, code)
    x = tcl.gemm(a, b, cfg=tcl.Config(cluster_k=4))
    y = tcl.gemm(a, b, cfg=tcl.Config(cluster_k=1))
    torch.cuda.synchronize()
    assert torch.allclose(x, y, rtol=1e-5, atol=1e-3)
    assert tcl.last_device_error() == (0, 0)


def test_64_row_tiles_bounded_wait_runs_out():
    # the 64×64-tile kernel: CTA 0 never loads one k-block, its MMA warp's wait runs out
    a, b = inputs.bf16_pair(512, 512, 512, seed=8)
    a, b = a.to(DEV), b.to(DEV)
    c = torch.zeros((512, 512), dtype=torch.float32, device=DEV)
    tcl.gemm_into(a, b, c, cfg=tcl.Config(tile_m=64, timeout_ns=50_000_000, debug_skip_kblock=2))
    st, code = tcl.last_device_error()
    assert st == 7 and code in (1, 2, 4), (st, code)
    x = tcl.gemm(a, b, cfg=tcl.Config(tile_m=64))
    y = tcl.gemm(a, b, cfg=tcl.Config(tile_m=128))
    torch.cuda.synchronize()
    assert torch.allclose(x, y, rtol=1e-5, atol=1e-4)
    assert tcl.last_device_error() == (0, 0)


def test_s8_in_kernel_bounded_wait_runs_out():
    # CTA 0's converter warps never hand one k-block over: the leader's MMA warp's bounded
    # wait for the stage runs out, both CTAs of the pair abort and return, and the next
    # call on the same device is exact
    a = torch.randint(-128, 128, (1024, 1024), dtype=torch.int8, generator=torch.Generator().manual_seed(3)).to(DEV)
    b = torch.randint(-128, 128, (1024, 1024), dtype=torch.int8, generator=torch.Generator().manual_seed(4)).to(DEV)
    c = torch.zeros((1024, 1024), dtype=torch.int32, device=DEV)
    cfg = tcl.Config(cta_pair=2, bn=256, s8_path=2, timeout_ns=50_000_000, debug_skip_kblock=3)
    tcl.gemm_into(a, b, c, cfg=cfg)
    st, code = tcl.last_device_error()
    assert st == 7 and code in (1, 2, 3, 4), (st, code)
    x = tcl.gemm(a, b, cfg=tcl.Config(cta_pair=2, bn=256, s8_path=2))
    y = tcl.gemm(a, b, cfg=tcl.Config(cta_pair=1))
    torch.cuda.synchronize()
    assert torch.equal(x, y)
    assert tcl.last_device_error() == (0, 0)
