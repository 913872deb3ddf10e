"""Host-side tiling arithmetic against the worked examples the pages print
(tests/golden/pages_worked_examples.json, each entry with its citation)."""
from __future__ import annotations

import json
import os

import pytest

import bench

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "pages_worked_examples.json")
with open(GOLDEN, encoding="utf-8") as f:
    G = json.load(f)


@pytest.mark.parametrize("case", G["compute_load_ratio"], ids=lambda c: f"{c['bm']}x{c['bn']}x{c['bk']}")
def test_compute_load_ratio(case):
    assert bench.compute_load_ratio(case["bm"], case["bn"], case["bk"], case["esize"]) == pytest.approx(case["value"])


@pytest.mark.parametrize("case", G["stage_bytes"], ids=lambda c: f"{c['bm']}x{c['bn']}x{c['bk']}")
def test_stage_bytes(case):
    assert bench.stage_bytes(case["bm"], case["bn"], case["bk"], case["esize"]) == (case["a"], case["b"], case["stage"])


@pytest.mark.parametrize("case", G["wave_blocks"], ids=lambda c: f"{c['sms']}x{c['blocks_per_sm']}")
def test_wave_blocks(case):
    assert bench.wave_blocks(case["sms"], case["blocks_per_sm"]) == case["value"]


def test_this_build_figures():
    # the same arithmetic for this build's tiles: one SM, 128×256×64 bf16 (the ablation);
    # the 4096³ plan's 256 two-SM tiles on 152 SMs
    assert bench.compute_load_ratio(128, 256, 64, 2) == pytest.approx(2 * 128 * 256 * 64 / ((128 * 64 + 64 * 256) * 2))
    assert bench.stage_bytes(128, 256, 64, 2)[2] == 48 * 1024
    assert bench.tile_waves({"num_tiles": 256, "cta_pair": 2}, 152) == pytest.approx(3.37, abs=0.01)
