"""The device-pointer entry points captured into CUDA graphs and replayed.

A replay re-runs the captured launches with the values they were captured with:
the same TMA descriptors, scratch addresses and stream-K flag generation. The
kernels leave the flags as they found them, so every replay orders the pieces
of a split tile again; results are compared bit for bit with direct calls.
"""
from __future__ import annotations

import subprocess
import sys
import os

import pytest
import torch

import tensor_core_loop_gb300 as tcl
from tensor_core_loop_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tcl.lib()
    yield
    assert tcl.last_device_error() == (0, 0)


def replay_matches(a, b, c, cfg, replays=25, calls=3):
    """Direct result, then a graph of `calls` captured calls replayed `replays` times,
    C cleared before each replay; every replay must reproduce the direct result."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        tcl.gemm_into(a, b, c, cfg=cfg)   # outside capture: plans, descriptors and scratch exist
        ref = c.clone()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(calls):
            tcl.gemm_into(a, b, c, cfg=cfg)
    with torch.cuda.stream(s):
        for _ in range(replays):
            c.zero_()
            g.replay()
            s.synchronize()
            assert torch.equal(c, ref)
    torch.cuda.synchronize()
    return ref


@pytest.mark.parametrize("pieces", [2, 4])
def test_stream_k_bf16_replays(pieces):
    a, b = inputs.bf16_pair(768, 768, 2048, seed=31)
    a, b = a.to(DEV), b.to(DEV)
    cfg = tcl.Config(cta_pair=2, max_ctas=8, stream_k=pieces)
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 768, 768, 2048, cfg)["sk_pieces"] == pieces
    c = torch.empty((768, 768), dtype=torch.float32, device=DEV)
    ref = replay_matches(a, b, c, cfg)
    direct = tcl.gemm(a, b, cfg=cfg)
    assert torch.equal(ref, direct)


def test_stream_k_bf16_out_replays():
    # bf16 C: the pieces meet in the fp32 workspace (library scratch) before one rounding
    a, b = inputs.bf16_pair(768, 768, 2048, seed=36)
    a, b = a.to(DEV), b.to(DEV)
    cfg = tcl.Config(cta_pair=2, max_ctas=8, stream_k=3)
    c = torch.empty((768, 768), dtype=torch.bfloat16, device=DEV)
    replay_matches(a, b, c, cfg)


def test_stream_k_int8_replays():
    a, b = inputs.s8_pair(768, 768, 2048, seed=32)
    a, b = a.to(DEV), b.to(DEV)
    cfg = tcl.Config(cta_pair=2, bn=256, max_ctas=8, stream_k=2)
    c = torch.empty((768, 768), dtype=torch.int32, device=DEV)
    ref = replay_matches(a, b, c, cfg)
    assert torch.equal(ref, (a.double() @ b.double()).to(torch.int32))


def test_headline_plan_replays():
    # the default 4096³ plan: two SMs per tile with a stream-K tail of 28 tiles × 2 pieces
    a, b = inputs.bf16_pair(4096, 4096, 4096, seed=33)
    a, b = a.to(DEV), b.to(DEV)
    pl = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 4096)
    assert pl["sk_tiles"] > 0
    c = torch.empty((4096, 4096), dtype=torch.float32, device=DEV)
    replay_matches(a, b, c, None, replays=8, calls=2)


def test_split_k_and_tf32_replay():
    # split-K partial tiles (and off-grid copies) live in library scratch
    a, b = inputs.bf16_pair(512, 512, 4096, seed=34)
    a, b = a.to(DEV), b.to(DEV)
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 512, 512, 4096)["splits"] > 1
    replay_matches(a, b, torch.empty((512, 512), dtype=torch.float32, device=DEV), None)
    at, bt = inputs.tf32_pair(384, 640, 512, seed=35)
    replay_matches(at.to(DEV), bt.to(DEV), torch.empty((384, 640), dtype=torch.float32, device=DEV), None)


def test_capture_refuses_to_grow_scratch():
    # in a fresh process: the first int8 call needs scratch, and the stream is capturing
    code = r"""
import torch, tensor_core_loop_gb300 as tcl
dev = torch.device("cuda:0")
x = torch.ones((256, 256), dtype=torch.bfloat16, device=dev)
tcl.gemm(x, x)                       # device set up outside capture (no scratch needed)
torch.cuda.synchronize()
a = torch.ones((256, 512), dtype=torch.int8, device=dev)
b = torch.ones((512, 256), dtype=torch.int8, device=dev)
c = torch.empty((256, 256), dtype=torch.int32, device=dev)
s = torch.cuda.Stream()
g = torch.cuda.CUDAGraph()
status = None
try:
    with torch.cuda.graph(g, stream=s):
        try:
            tcl.gemm_into(a, b, c)
        except tcl.TclError as e:
            status = e.status
except Exception:
    pass
print("STATUS", status)
tcl.gemm_into(a, b, c)               # outside capture the scratch grows and the call runs
torch.cuda.synchronize()
print("OK", bool((c == 512).all()))
"""
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert "STATUS 12" in r.stdout, r.stdout + r.stderr
    assert "OK True" in r.stdout, r.stdout + r.stderr
