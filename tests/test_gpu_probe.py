"""The tensor-pipe probe on the GPU: tcgen05.mma reaches its per-SM rate, and the
warp-level mma.sync forms (int8 m16n8k32, bf16 m16n8k16) run and report a rate
far below it (the reason the int8 path widens to bf16 for tcgen05)."""
from __future__ import annotations

import pytest
import torch

import tensor_core_loop_gb300 as tcl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tcl.lib()
    tcl.last_device_error()


def test_tcgen05_rate_per_sm():
    cyc, rate, _ = tcl.mma_peak(tcl.IN_BF16, 256, 1, iters=1024, flags=2)
    assert min(cyc) > 0
    assert 7000 < rate <= 8192 * 1.01          # 8192 bf16 flop/clk/SM at N = 256
    assert tcl.last_device_error() == (0, 0)


@pytest.mark.parametrize("kind,flags", [(tcl.IN_S8, 0), (tcl.IN_BF16, 128)])
def test_warp_mma_forms_run(kind, flags):
    cyc, rate, _ = tcl.mma_peak(kind, 128, 0, iters=256, flags=flags)
    assert min(cyc) > 0 and len(cyc) == tcl.num_sms()
    _, tc_rate, _ = tcl.mma_peak(tcl.IN_BF16, 256, 1, iters=1024, flags=2)
    assert 0 < rate < tc_rate                  # the legacy path is slower than tcgen05 per SM
    assert tcl.last_device_error() == (0, 0)
