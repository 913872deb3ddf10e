"""The C ABI on the host (no GPU): the library loads, exports every entry point
include/tcl_gemm.h declares, rejects bad arguments with the documented status
before touching the device, and plans launches as documented."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import tensor_core_loop_gb300 as tcl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from tensor_core_loop_gb300 import _build
    _build.build()
    return tcl.lib()


def header_symbols():
    text = open(os.path.join(ROOT, "include", "tcl_gemm.h")).read()
    return sorted(set(re.findall(r"TCL_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)))


def test_header_declares_expected_api():
    syms = header_symbols()
    assert set(syms) == set(tcl.EXPORTED_SYMBOLS), syms


@pytest.mark.parametrize("struct,mirror", [("tcl_config_t", tcl.Config), ("tcl_plan_t", tcl.PlanInfo)])
def test_struct_mirrors_match_the_header(struct, mirror, tmp_path):
    """The ctypes mirrors have the C structs' size and every field at the C offset (a C
    program compiled against the header prints them)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    cuda_inc = next((d for d in ("/usr/local/cuda/include", os.path.join(os.environ.get("CUDA_HOME", ""), "include"))
                     if os.path.exists(os.path.join(d, "cuda_runtime_api.h"))), None)
    if not cc or not cuda_inc:
        pytest.skip("no C compiler or CUDA headers")
    names = [n for n, _ in mirror._fields_]
    body = "".join(f'printf("%zu\\n", offsetof({struct}, {n}));' for n in names)
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "tcl_gemm.h"\n'
                   f'int main(void) {{ printf("%zu\\n", sizeof({struct})); {body} return 0; }}\n')
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()]
    assert len(got) == len(names) + 1
    assert got[0] == ctypes.sizeof(mirror), (struct, got[0], ctypes.sizeof(mirror))
    for n, off in zip(names, got[1:]):
        assert getattr(mirror, n).offset == off, (struct, n, off, getattr(mirror, n).offset)


def test_library_exports_every_declared_symbol(L):
    for name in header_symbols():
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def test_version_and_status_strings(L):
    assert "sm_103a" in tcl.version()
    for code in range(11):
        s = L.tcl_status_string(code).decode()
        assert s and s != "unknown status"
    assert L.tcl_status_string(99).decode() == "unknown status"


# Fake but well-formed device addresses: validation must reject before any CUDA call.
P = 0x10000000
PO = 0x10000001  # odd: not aligned to any element size
P2 = 0x10000002  # 2-byte aligned only
# (Only calls that the host-side checks reject get these fake pointers: a call
# that passed them would launch kernels on addresses that do not exist.)


@pytest.mark.parametrize("args,status", [
    ((64, 64, 64, 0, 64, P, 64, P, 64, 0), 1),            # A null
    ((64, 64, 64, P, 64, P, 64, 0, 64, 0), 1),            # C null
    ((0, 64, 64, P, 64, P, 64, P, 64, 0), 2),             # M = 0
    ((64, 64, -1, P, 64, P, 64, P, 64, 0), 2),            # K < 0
    ((64, 64, 64, P, 32, P, 64, P, 64, 0), 3),            # lda < K
    ((64, 64, 64, P, 64, P, 32, P, 64, 0), 3),            # ldb < N
    ((64, 64, 64, P, 64, P, 64, P, 32, 0), 3),            # ldc < N
    ((64, 64, 64, PO, 64, P, 64, P, 64, 0), 4),           # A not on a 2-byte boundary
    ((64, 64, 64, P, 64, PO, 64, P, 64, 0), 4),           # B not on a 2-byte boundary
    ((64, 64, 64, P, 64, P, 64, P2, 64, 0), 4),           # fp32 C not on a 4-byte boundary
    ((64, 64, 64, P, 64, P, 64, PO, 64, 1), 4),           # bf16 C not on a 2-byte boundary
    ((64, 64, 64, P, 64, P, 64, P, 64, 7), 8),            # unknown output type
])
def test_gemm_bf16_rejects(L, args, status):
    assert L.gemm_bf16(*args, None) == status


def test_gemm_tf32_and_s8_reject(L):
    assert L.gemm_tf32(64, 64, 64, P2, 64, P, 64, P, 64, None) == 4       # fp32 A not on a 4-byte boundary
    assert L.gemm_tf32(64, 64, 64, P, 64, P, 64, P2, 64, None) == 4
    assert L.gemm_tf32(64, 64, 64, 0, 64, P, 64, P, 64, None) == 1
    assert L.gemm_s8(64, 64, 131072, P, 131072, P, 64, P, 64, None) == 5  # K beyond the exact int32 range
    assert L.gemm_s8(64, 64, 64, P, 64, P, 64, P2, 64, None) == 4         # int32 C not on a 4-byte boundary
    assert L.gemm_bf16_host(64, 64, 64, 0, 64, P, 64, P, 64, 0, None) == 1
    assert L.gemm_bf16_host(64, 64, 64, P, 32, P, 64, P, 64, 0, None) == 3
    assert L.gemm_bf16_host(64, 64, 64, PO, 64, P, 64, P, 64, 0, None) == 4
    assert L.gemm_bf16_host(64, 64, 64, P, 64, P, 64, P, 64, 5, None) == 8
    assert L.gemm_f32_simt(64, 64, 64, P2, 64, P, 64, P, 64, None) == 4   # fp32 A not on a 4-byte boundary
    assert L.gemm_f32_simt(64, 64, 64, P, 64, P, 64, 0, 64, None) == 1
    assert L.gemm_f32_simt(64, 64, 64, P, 64, P, 32, P, 64, None) == 3
    # the allocation-free form keeps the tensor-copy rule (it has no scratch to repack into)
    assert L.gemm_s8_static(64, 64, 64, P, 72, P, 64, P, 64, None) == 4
    assert L.gemm_s8_static(64, 64, 64, P, 64, P, 64, P + 4, 64, None) == 4


def test_mma_peak_rejects(L):
    # (a real host buffer: every call here must return before any launch)
    buf = (ctypes.c_ulonglong * 4)()
    cyc = ctypes.addressof(buf)
    assert L.tcl_mma_peak(0, 256, 0, 0, 4096, 1, None, None) == 1          # no cycles buffer
    assert L.tcl_mma_peak(3, 256, 0, 0, 4096, 1, cyc, None) == 2           # unknown kind
    assert L.tcl_mma_peak(2, 256, 1, 0, 4096, 1, cyc, None) == 2           # int8 warp MMA: no B major-ness
    assert L.tcl_mma_peak(1, 256, 1, 0, 4096, 1, cyc, None) == 2           # TF32: K-major B only
    assert L.tcl_mma_peak(0, 100, 0, 0, 4096, 1, cyc, None) == 2           # N not built
    assert L.tcl_mma_peak(2, 128, 0, 1, 4096, 1, cyc, None) == 8           # warp MMA takes no other flag
    assert L.tcl_mma_peak(0, 128, 0, 129, 4096, 1, cyc, None) == 8
    assert L.tcl_mma_peak(1, 128, 0, 128, 4096, 1, cyc, None) == 8         # no TF32 warp MMA
    assert L.tcl_mma_peak(0, 128, 0, 256, 4096, 1, cyc, None) == 8         # unknown flag bit


def test_plan_without_device(L):
    cfg = tcl.Config(max_ctas=152)
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 4096, tcl.Config(max_ctas=152, stream_k=1))
    # enough 256-row tiles for every pair of SMs: two SMs per tile; even without a stream-K
    # tail 256 columns (16 × 16 tiles, a partial last wave) beat the 224 columns that give
    # exactly 4 tiles per pair (two k-blocks per copy: 89.0 against 98.7 µs on GB300)
    assert p["cta_pair"] == 2 and p["bn"] == 256 and p["num_tiles"] == 16 * 16 and p["grid"] == 152
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_BF16, 4096, 4096, 4096, cfg)
    assert p["cta_pair"] == 2 and p["bn"] == 256 and p["num_tiles"] == 16 * 16
    assert p["smem_bytes"] <= 232448
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 4096, tcl.Config(max_ctas=152, cta_pair=1))
    assert p["cta_pair"] == 1 and p["bn"] == 256 and p["num_tiles"] == 32 * 16 and p["grid"] == 152
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 300, 520, 64, tcl.Config(max_ctas=152, cta_pair=2))
    assert p["cta_pair"] == 2 and p["num_tiles"] == 2 * 3 and p["grid"] == 12
    # exact integers on two SMs: 256×128 tiles (a row's 128 int32 sums live in registers)
    for c in (cfg, tcl.Config(max_ctas=152, cta_pair=2)):
        p = tcl.plan(tcl.IN_S8, 0, 4096, 4096, 4096, c)
        assert p["cta_pair"] == 2 and p["bn"] == 256 and p["num_tiles"] == 16 * 16 and p["grid"] == 152
        assert (p["sk_tiles"], p["sk_pieces"], p["splits"]) == (28, 2, 1)   # int32 pieces add exactly
    p = tcl.plan(tcl.IN_S8, 0, 4096, 4096, 4096, tcl.Config(max_ctas=152, cta_pair=2, bn=128))
    assert p["cta_pair"] == 2 and p["bn"] == 128 and p["num_tiles"] == 16 * 32
    for bad in (tcl.Config(max_ctas=152, cta_pair=2, bn=224), tcl.Config(max_ctas=152, cta_pair=3),
                tcl.Config(max_ctas=152, cta_pair=1, stream_k=2)):
        with pytest.raises(tcl.TclError):
            tcl.plan(tcl.IN_S8, 0, 4096, 4096, 4096, bad)
    p = tcl.plan(tcl.IN_S8, 0, 4096, 4096, 4096, tcl.Config(max_ctas=152, cta_pair=1))
    assert p["cta_pair"] == 1 and p["bn"] == 128 and p["num_tiles"] == 32 * 32
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 512, 512, 4096, cfg)
    # 16 narrow tiles for 152 SMs: K is cut into 8 ranges of 8 k-blocks (split-K)
    assert p["cta_pair"] == 1 and p["bn"] == 128 and p["num_tiles"] == 16
    assert p["splits"] == 8 and p["grid"] == 128 and p["workspace_bytes"] == 8 * 512 * 512 * 4
    # 4 k-blocks on many tiles: narrow tiles for an fp32 C, wide ones for a bf16 C
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 256, cfg)["bn"] == 128
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_BF16, 4096, 4096, 256, cfg)["bn"] == 256
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 512, 512, 256, cfg)     # 4 k-blocks: too short to split
    # ... and 16 tiles of 128×128 fill a tenth of the SMs: 64×64 tiles, 64 CTAs
    assert p["splits"] == 1 and p["bn"] == 64 and p["workspace_bytes"] == 0
    assert (p["tile_m"], p["grid"], p["num_tiles"], p["stages"], p["cluster_k"]) == (64, 64, 64, 6, 1)
    # (two k-blocks per 32 KB stage when K is whole 64-wide blocks, else one per 16 KB stage)
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 512, 512, 520, cfg)["stages"] == 8
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 512, 512, 256, tcl.Config(max_ctas=152, tile_m=128))
    assert (p["tile_m"], p["bn"], p["grid"]) == (128, 64, 32)                       # 128×64 tiles
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_BF16, 768, 768, 1024, cfg)["tile_m"] == 64  # 144 CTAs
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 512, 512, 2048, cfg)["tile_m"] == 128  # split-K instead
    for bad in (tcl.Config(max_ctas=152, tile_m=32), tcl.Config(max_ctas=152, tile_m=64, bn=128),
                tcl.Config(max_ctas=152, tile_m=64, cta_pair=2), tcl.Config(max_ctas=152, tile_m=64, split_k=2),
                tcl.Config(max_ctas=152, tile_m=64, stages=4), tcl.Config(max_ctas=152, tile_m=64, cluster_k=2)):
        with pytest.raises(tcl.TclError):
            tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 512, 512, 512, bad)
    for in_kind, out in ((tcl.IN_TF32, tcl.OUT_F32), (tcl.IN_S8, 0)):   # bf16 operands only
        with pytest.raises(tcl.TclError):
            tcl.plan(in_kind, out, 512, 512, 512, tcl.Config(max_ctas=152, tile_m=64))
        assert tcl.plan(in_kind, out, 512, 512, 256, cfg)["tile_m"] == 128
    # K ranges of a tile summed in a cluster of 2 or 4 CTAs, on request
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 512, 512, 256, tcl.Config(max_ctas=152, cluster_k=4))
    assert (p["bn"], p["cluster_k"], p["grid"], p["num_tiles"], p["stages"]) == (64, 4, 128, 32, 4)
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_BF16, 1024, 512, 1024, tcl.Config(max_ctas=152, cluster_k=2))
    assert (p["cluster_k"], p["grid"], p["splits"]) == (2, 128, 1)
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 300, 200, 64, tcl.Config(max_ctas=152, cluster_k=4))
    assert (p["cluster_k"], p["bn"], p["grid"]) == (4, 64, 4 * 3 * 4)   # ranges may be empty
    for bad in (tcl.Config(max_ctas=152, cluster_k=3), tcl.Config(max_ctas=152, cluster_k=8),
                tcl.Config(max_ctas=152, cluster_k=2, split_k=2), tcl.Config(max_ctas=152, cluster_k=2, bn=128),
                tcl.Config(max_ctas=152, cluster_k=2, cta_pair=2), tcl.Config(max_ctas=152, cluster_k=2, stages=4),
                tcl.Config(max_ctas=152, cluster_k=2, one_cta_per_tile=1), tcl.Config(max_ctas=152, cluster_k=-1)):
        with pytest.raises(tcl.TclError):
            tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 512, 512, 512, bad)
    for in_kind, out in ((tcl.IN_TF32, tcl.OUT_F32), (tcl.IN_S8, 0)):   # bf16 operands only
        with pytest.raises(tcl.TclError):
            tcl.plan(in_kind, out, 512, 512, 512, tcl.Config(max_ctas=152, cluster_k=2))
    # split-K shapes keep 128-wide tiles
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 512, 512, 2048, cfg)["bn"] == 128
    # mid-size outputs by the cost model (waves × k-blocks × per-k-block cycles + fixed
    # cycles per launch): the measured fastest shape at each of these (GB300, CUDA graphs:
    # 1024×4096×4096 28.98 µs on one SM against 30.03 on 224-wide pairs, 2048²×4096 27.63
    # against 28.21 on 256-wide pairs)
    for (m, n, k), want in {(1024, 4096, 4096): (1, 256), (2048, 2048, 4096): (1, 256),
                            (1024, 4096, 1024): (1, 256), (2048, 2048, 1024): (1, 256),
                            (1536, 3072, 2048): (1, 256), (3072, 3072, 1024): (1, 256),
                            (512, 4096, 4096): (1, 128)}.items():
        p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, m, n, k, cfg)
        assert (p["cta_pair"], p["bn"]) == want, ((m, n, k), p)
    for in_kind, (m, n, k), want in ((tcl.IN_TF32, (1024, 4096, 4096), (2, 256)),   # 48.1 against 57.8 µs
                                     (tcl.IN_TF32, (1024, 4096, 1024), (1, 256)),
                                     (tcl.IN_S8, (1024, 4096, 4096), (2, 256)),
                                     (tcl.IN_S8, (1024, 4096, 1024), (2, 256))):
        p = tcl.plan(in_kind, 0, m, n, k, cfg)
        assert (p["cta_pair"], p["bn"]) == want, ((m, n, k), p)
    # deep two-SM tiles (rows of A of 16 KB and more): a row of tiles at a time, K walked
    # in alternating directions; shorter rows keep groups of 8 and ascending K
    for in_kind, k in ((tcl.IN_BF16, 8192), (tcl.IN_TF32, 4096)):
        p = tcl.plan(in_kind, tcl.OUT_F32, 4096, 4096, k, cfg)
        assert (p["cta_pair"], p["group_m"], p["k_serpentine"]) == (2, 1, 1)
    for k in (2048, 3072, 4096):   # (the whole grid: automatically, from 48 k-blocks on, the die split, row by row)
        p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, k, tcl.Config(max_ctas=152, die_split=1))
        assert (p["group_m"], p["k_serpentine"]) == (8, 0)
        p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, k, cfg)
        assert (p["die_split"], p["group_m"], p["k_serpentine"]) == ((1, 1, 0) if k >= 3072 else (0, 8, 0))
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 4096, tcl.Config(max_ctas=152, group_m=4, k_order=1))
    assert (p["group_m"], p["k_serpentine"]) == (4, 0)
    # int8 on 256-wide pair tiles widens inside the kernel on request (s8_path 2) only
    p = tcl.plan(tcl.IN_S8, 0, 4096, 4096, 4096, cfg)
    assert (p["cta_pair"], p["bn"], p["s8_in_kernel"]) == (2, 256, 0)
    p = tcl.plan(tcl.IN_S8, 0, 4096, 4096, 4096, tcl.Config(max_ctas=152, s8_path=2))
    assert (p["s8_in_kernel"], p["stages"]) == (1, 4)
    assert tcl.plan(tcl.IN_S8, 0, 4096, 4096, 4096, tcl.Config(max_ctas=152, s8_path=1))["s8_in_kernel"] == 0
    assert tcl.plan(tcl.IN_S8, 0, 4096, 4096, 4096, tcl.Config(max_ctas=152, cta_pair=1))["s8_in_kernel"] == 0
    for bad in (tcl.Config(max_ctas=152, cta_pair=1, s8_path=2), tcl.Config(max_ctas=152, s8_path=3)):
        with pytest.raises(tcl.TclError):
            tcl.plan(tcl.IN_S8, 0, 4096, 4096, 4096, bad)
    with pytest.raises(tcl.TclError):
        tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 4096, tcl.Config(max_ctas=152, s8_path=2))
    for bad in (tcl.Config(max_ctas=152, k_order=3), tcl.Config(max_ctas=152, k_order=2, producer=1)):
        with pytest.raises(tcl.TclError):
            tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 1024, 1024, 1024, bad)
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 512, 512, 8192, cfg)
    assert p["splits"] == 9 and p["grid"] == 144
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 512, 512, 8192, tcl.Config(max_ctas=152, split_k=1))
    assert p["splits"] == 1
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_BF16, 300, 261, 1000, tcl.Config(max_ctas=152, split_k=3))
    assert p["splits"] == 3 and p["workspace_bytes"] == 3 * 384 * 264 * 4
    for bad in (tcl.Config(max_ctas=152, split_k=2, cta_pair=2),):
        with pytest.raises(tcl.TclError):
            tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 512, 512, 4096, bad)
    with pytest.raises(tcl.TclError):
        tcl.plan(tcl.IN_S8, 0, 512, 512, 4096, tcl.Config(max_ctas=152, split_k=2))
    assert tcl.plan(tcl.IN_S8, 0, 512, 512, 4096, cfg)["splits"] == 1   # exact integers: never split
    p = tcl.plan(tcl.IN_S8, 0, 512, 512, 4096, cfg)   # too few 256-row tiles for the pair kernel
    assert p["bn"] == 128 and p["cta_pair"] == 1
    p = tcl.plan(tcl.IN_TF32, 0, 300, 70, 9, cfg)
    assert p["num_tiles"] == 3 * 1
    cfg2 = tcl.Config(max_ctas=152, bn=256, stages=2, one_cta_per_tile=1)
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 4096, cfg2)
    assert p["stages"] == 2 and p["grid"] == 512
    with pytest.raises(tcl.TclError):
        tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 4096, tcl.Config(max_ctas=152, bn=192))
    with pytest.raises(tcl.TclError):
        tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 4096, tcl.Config(max_ctas=152, stages=5))


def test_planner_stream_k(L):
    cfg = tcl.Config(max_ctas=152)
    # 4096³ on 76 pairs: 256 tiles of 256×256 = 3 full waves + 28 tiles, each cut in two K
    # ranges, beats 304 tiles of 256×224 (4 waves at the 224-wide k-block rate)
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 4096, cfg)
    assert (p["cta_pair"], p["bn"], p["num_tiles"], p["sk_tiles"], p["sk_pieces"], p["sk_balanced"]) == \
        (2, 256, 256, 28, 2, 0)
    assert p["workspace_bytes"] == 0   # fp32 C: pieces add into C itself
    # balanced stream-K on request: two waves of whole tiles, then the 104·64 k-blocks of the
    # last 104 tiles in 76 ranges of 87-88 k-blocks, 72 tiles cut by a range boundary
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 4096, tcl.Config(max_ctas=152, stream_k=5))
    assert (p["sk_balanced"], p["sk_tiles"], p["sk_pieces"]) == (1, 72, 2)
    # equal pieces on request: 3 full waves + 28 tiles, each cut in two K ranges (224 k-blocks)
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 4096, tcl.Config(max_ctas=152, stream_k=2))
    assert (p["bn"], p["sk_balanced"], p["sk_tiles"], p["sk_pieces"]) == (256, 0, 28, 2)
    # without stream-K the 256-wide tiles still win (one copy brings two k-blocks)
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 4096, tcl.Config(max_ctas=152, stream_k=1))
    assert (p["bn"], p["sk_tiles"], p["sk_balanced"]) == (256, 0, 0)
    # whole waves: nothing to split
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4864, 4096, 4096, cfg)
    assert (p["bn"], p["num_tiles"], p["sk_tiles"], p["sk_balanced"]) == (256, 304, 0, 0)
    # 9 tiles on 4 pairs: 4 equal pieces of the 9th tile tie with balanced ranges (72 k-blocks)
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 768, 768, 2048, tcl.Config(max_ctas=8, cta_pair=2))
    assert (p["num_tiles"], p["sk_tiles"], p["sk_pieces"], p["sk_balanced"]) == (9, 1, 4, 0)
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 768, 768, 2048, tcl.Config(max_ctas=8, cta_pair=2, stream_k=5))
    assert (p["sk_balanced"], p["sk_pieces"]) == (1, 2) and p["sk_tiles"] == 3   # 5 tiles, ranges of 40
    # short tiles (16 k-blocks): the extra piece's epilogue costs more than the tail saves
    # (automatically this shape runs on one SM per tile: 32.8 µs against 32.9 on 224-wide
    # and 33.6 on 256-wide pairs)
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 1024, cfg)["cta_pair"] == 1
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 1024, tcl.Config(max_ctas=152, cta_pair=2))
    assert (p["bn"], p["sk_tiles"], p["sk_balanced"]) == (256, 0, 0)
    for k in (2048, 8192):
        assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, k, cfg)["sk_tiles"] == 28
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_BF16, 4096, 4096, 1024, cfg)["sk_tiles"] == 0
    for bad in (tcl.Config(max_ctas=8, cta_pair=2, stream_k=6),       # no such mode
                tcl.Config(max_ctas=8, cta_pair=1, stream_k=2),       # one-SM kernel
                tcl.Config(max_ctas=4, cta_pair=2, stream_k=3),       # 1 tail tile × 3 pieces > 2 pairs
                tcl.Config(max_ctas=8, cta_pair=2, stream_k=-1)):
        with pytest.raises(tcl.TclError):
            tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 768, 768, 2048, bad)
    # as many pairs as tiles (the grid never exceeds the tiles): one whole tile per range
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 512, 512, 2048, tcl.Config(max_ctas=16, cta_pair=2, stream_k=5))
    assert (p["grid"], p["sk_balanced"], p["sk_tiles"]) == (8, 1, 0)
    # a bf16 C takes a stream-K tail through an fp32 workspace: split tiles × 256 rows × bn
    # columns, or one block per range boundary (per pair) when balanced
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_BF16, 768, 768, 2048, tcl.Config(max_ctas=8, cta_pair=2, stream_k=2))
    assert (p["sk_tiles"], p["sk_pieces"]) == (1, 2) and p["workspace_bytes"] == 1 * 256 * 256 * 4
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_BF16, 4096, 4096, 4096, tcl.Config(max_ctas=152, stream_k=2))
    assert (p["bn"], p["sk_tiles"], p["sk_pieces"]) == (256, 28, 2) and p["workspace_bytes"] == 28 * 256 * 256 * 4
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_BF16, 4096, 4096, 4096, tcl.Config(max_ctas=152, stream_k=5))
    assert p["sk_balanced"] == 1 and p["workspace_bytes"] == 76 * 256 * 256 * 4


def test_planner_kblocks_per_copy(L):
    # two-SM 256-wide tiles bring two k-blocks per tensor copy of each operand where K is whole
    # k-blocks, N whole B boxes (64 bf16 / 32 TF32 columns) and the ring depth even
    cfg = tcl.Config(max_ctas=152)
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 4096, cfg)
    assert (p["cta_pair"], p["bn"], p["stages"], p["kblocks_per_stage"]) == (2, 256, 6, 2)
    assert tcl.plan(tcl.IN_TF32, tcl.OUT_F32, 4096, 4096, 4096, cfg)["kblocks_per_stage"] == 2
    assert tcl.plan(tcl.IN_S8, 0, 4096, 4096, 4096, cfg)["kblocks_per_stage"] == 2
    assert tcl.plan(tcl.IN_TF32, tcl.OUT_F32, 4096, 4064, 4096, cfg)["kblocks_per_stage"] == 2   # 32-column boxes
    for M, N, K in ((4096, 4064, 4096), (4096, 4096, 4000)):   # N or K not whole blocks
        p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, M, N, K, cfg)
        assert p["cta_pair"] == 2 and p["kblocks_per_stage"] == 1
        with pytest.raises(tcl.TclError):
            tcl.plan(tcl.IN_BF16, tcl.OUT_F32, M, N, K, tcl.Config(max_ctas=152, kblocks_per_stage=2))
    off = tcl.Config(max_ctas=152, kblocks_per_stage=1)
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 4096, off)["kblocks_per_stage"] == 1
    for bad in (tcl.Config(max_ctas=152, cta_pair=2, stages=5, kblocks_per_stage=2),   # odd ring
                tcl.Config(max_ctas=152, cta_pair=2, bn=224, kblocks_per_stage=2),
                tcl.Config(max_ctas=152, cta_pair=1, kblocks_per_stage=2),
                tcl.Config(max_ctas=152, kblocks_per_stage=3)):
        with pytest.raises(tcl.TclError):
            tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 4096, bad)
    with pytest.raises(tcl.TclError):   # the kernel that widens int8 itself has its own ring
        tcl.plan(tcl.IN_S8, 0, 4096, 4096, 4096, tcl.Config(max_ctas=152, s8_path=2, kblocks_per_stage=2))
    for bad in (-1, 2):
        with pytest.raises(tcl.TclError):
            tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 4096, tcl.Config(max_ctas=152, b_copy=bad))
    # one SM per tile: 64×64 tiles report their two k-blocks per 32 KB stage
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 512, 512, 256, cfg)["kblocks_per_stage"] == 2
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 512, 512, 520, cfg)["kblocks_per_stage"] == 1


def test_planner_die_split(L):
    # two-SM grids of at most 16 tile columns: the tiles in one block of columns per die,
    # each with its own stream-K tail (offline, half of the max_ctas / 2 pairs on each die)
    cfg = tcl.Config(max_ctas=152)
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 8192, cfg)
    assert (p["cta_pair"], p["die_split"], p["die_tiles0"], p["group_m"]) == (2, 1, 128, 1)
    # 16 × 8 tiles per die on 38 pairs: 3 waves and 14 tiles in 2 pieces, on each die
    assert (p["sk_tiles"], p["sk_pieces"], p["grid"]) == (28, 2, 152)
    assert tcl.plan(tcl.IN_TF32, tcl.OUT_F32, 4096, 4096, 4096, cfg)["die_split"] == 1   # 16 KB rows
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_BF16, 4096, 4096, 8192, cfg)["die_split"] == 1
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 4096, cfg)["die_split"] == 1
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 8192, 8192, 8192, cfg)["die_split"] == 0   # 32 columns
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 4096, tcl.Config(max_ctas=152, group_m=4))["die_split"] == 0
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 4096, tcl.Config(max_ctas=8))["die_split"] == 0   # 4 pairs
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 3072, 3072, 4096, cfg)["die_split"] == 0   # 144 tiles: < 3 waves
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 6144, 4096, 4096, cfg)["die_split"] == 1
    # and from 48 k-blocks (6 KB of K per operand row) on
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 3072, cfg)["die_split"] == 1
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 2560, cfg)["die_split"] == 0
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 2048, cfg)["die_split"] == 0
    assert tcl.plan(tcl.IN_TF32, tcl.OUT_F32, 4096, 4096, 2048, cfg)["die_split"] == 1
    assert tcl.plan(tcl.IN_TF32, tcl.OUT_F32, 4096, 4096, 1024, cfg)["die_split"] == 0
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 1536, tcl.Config(max_ctas=152, die_split=2))["die_split"] == 1
    # L2 eviction hints (A evict-first, B evict-last) with the die split for deep tiles only
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 8192, cfg)["l2_hints"] == 1
    assert tcl.plan(tcl.IN_TF32, tcl.OUT_F32, 4096, 4096, 4096, cfg)["l2_hints"] == 1
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 4096, cfg)["l2_hints"] == 0
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 8192, 8192, 8192, cfg)["l2_hints"] == 0   # no die split
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 4096, tcl.Config(max_ctas=152, l2_hints=2))["l2_hints"] == 1
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 8192, tcl.Config(max_ctas=152, l2_hints=1))["l2_hints"] == 0
    for bad in (tcl.Config(max_ctas=152, l2_hints=3), tcl.Config(max_ctas=152, l2_hints=2, cta_pair=1)):
        with pytest.raises(tcl.TclError):
            tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 4096, bad)
    on = tcl.Config(max_ctas=152, die_split=2)
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 8192, 8192, 8192, on)
    assert (p["die_split"], p["die_tiles0"]) == (1, 512)
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 8192, tcl.Config(max_ctas=152, die_split=1))["die_split"] == 0
    # uneven dies: the tiles in proportion to the pairs, to the tile (offline: 37 and 38
    # pairs for max_ctas 150: 256 · 37 / 75 rounds to 126 tiles, 7 columns and 14 rows of
    # the 8th; 192 · 37 / 75 to 95)
    p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 8192, tcl.Config(max_ctas=150))
    assert p["die_split"] == 1 and p["die_tiles0"] == 126 and p["grid"] == 150
    assert tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 3072, 8192,
                    tcl.Config(max_ctas=150, die_split=2))["die_tiles0"] == 95
    for bad in (tcl.Config(max_ctas=152, die_split=3), tcl.Config(max_ctas=152, die_split=-1),
                tcl.Config(max_ctas=152, die_split=2, cta_pair=1),
                tcl.Config(max_ctas=152, die_split=2, stream_k=5)):
        with pytest.raises(tcl.TclError):
            tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 4096, bad)
    with pytest.raises(tcl.TclError):   # fewer tiles than pairs: not every pair would take a place
        tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 1024, 1024, 8192, tcl.Config(max_ctas=152, die_split=2, cta_pair=2))


def test_planner_producer_kinds(L):
    for prod in (tcl.PRODUCER_SYNC, tcl.PRODUCER_CPASYNC):
        p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 4096, tcl.Config(max_ctas=152, producer=prod))
        # thread-copy producers: one SM per tile, four producer warps in front of the MMA warp
        assert p["producer"] == prod and p["cta_pair"] == 1 and p["bn"] == 256
    for bad in (3, -1):
        with pytest.raises(tcl.TclError):
            tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 4096, 4096, 4096, tcl.Config(max_ctas=152, producer=bad))
    for kind in (tcl.IN_TF32, tcl.IN_S8):   # the thread-copy producers are bf16 only
        with pytest.raises(tcl.TclError):
            tcl.plan(kind, 0, 512, 512, 512, tcl.Config(max_ctas=152, producer=tcl.PRODUCER_CPASYNC))


def test_every_stage_count_fits_shared_memory(L):
    for bn, stages in [(256, 1), (256, 2), (256, 3), (256, 4), (128, 1), (128, 2), (128, 4), (128, 6)]:
        p = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, 1024, 1024, 1024, tcl.Config(max_ctas=8, bn=bn, stages=stages))
        assert p["smem_bytes"] <= 232448
