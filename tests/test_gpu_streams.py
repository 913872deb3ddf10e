"""Calls on several streams at once.

Each stream has its own library scratch (widened int8 operands, repacked
operands, split-K partial tiles) and its own stream-K progress flags, so calls
enqueued on two streams without any ordering between them may run on the GPU
at the same time. Every result is compared bit for bit with the same call run
alone on the default stream (each plan's arithmetic order is fixed, so a call
gives the same bits wherever it runs).
"""
from __future__ import annotations

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
    yield
    assert tcl.last_device_error() == (0, 0)


def _jobs():
    """(a, b, out dtype, cfg): calls that each need scratch, stream-K flags or both."""
    jobs = []
    a, b = inputs.bf16_pair(4096, 4096, 4096, seed=11)       # two-SM tiles, stream-K tail: flags
    jobs.append((a.to(DEV), b.to(DEV), torch.float32, None))
    a, b = inputs.bf16_pair(4096, 4096, 4096, seed=12)       # bf16 C: stream-K workspace in scratch
    jobs.append((a.to(DEV), b.to(DEV), torch.bfloat16, None))
    a, b = inputs.s8_pair(2048, 2048, 3072, seed=13)         # int8: widened copies in scratch
    jobs.append((a.to(DEV), b.to(DEV), torch.int32, None))
    a, b = inputs.bf16_pair(512, 512, 4096, seed=14)         # small grid: split-K partial tiles
    jobs.append((a.to(DEV), b.to(DEV), torch.float32, None))
    a, b = inputs.tf32_pair(1000, 776, 1030, seed=15)        # K off the 16-byte grid: repacked operands
    jobs.append((a.to(DEV), b.to(DEV), torch.float32, None))
    return jobs


def test_concurrent_streams_match_serial():
    jobs = _jobs()
    ref = [tcl.gemm(a, b, out_dtype=o, cfg=c) for a, b, o, c in jobs]
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = {1: [], 2: []}
    for s in (s1, s2):
        s.wait_stream(torch.cuda.current_stream())
    # every job on both streams, in opposite orders, several rounds, no ordering between the streams
    for rnd in range(4):
        for k in range(len(jobs)):
            for sid, s, j in ((1, s1, k), (2, s2, len(jobs) - 1 - k)):
                a, b, o, c = jobs[j]
                with torch.cuda.stream(s):
                    outs[sid].append((j, tcl.gemm(a, b, out_dtype=o, cfg=c, stream=s)))
    torch.cuda.synchronize()
    assert tcl.last_device_error() == (0, 0)
    for sid in (1, 2):
        for j, x in outs[sid]:
            assert torch.equal(x, ref[j]), (sid, j)
    tcl.stream_release(s1)
    tcl.stream_release(s2)


def test_released_stream_works_again():
    a, b = inputs.s8_pair(1024, 768, 2048, seed=21)
    a, b = a.to(DEV), b.to(DEV)
    ref = tcl.gemm(a, b)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    x = tcl.gemm(a, b, stream=s)
    tcl.stream_release(s)       # synchronises the stream, frees its scratch and flags
    assert torch.equal(x, ref)
    y = tcl.gemm(a, b, stream=s)   # a new set for the same stream
    s.synchronize()
    assert torch.equal(y, ref)
    tcl.stream_release(s)
    tcl.stream_release(torch.cuda.current_stream())   # the default stream: a no-op
