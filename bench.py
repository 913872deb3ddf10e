#!/usr/bin/env python3
"""Benchmark: bf16 GEMM TFLOPS at M=N=K=4096 (fp32 accumulate, fp32 C) on GB300,
as a fraction of the tensor roofline, plus the K sweep, through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one C = A·B of the 4096³ workload (A, B row-major bf16, uniform
[-1, 1) from seed 0). Inputs are resident in HBM when the timed region
starts; the step's inputs rotate over enough sets that the footprint exceeds
the 129 MB L2, so no step reads operands another step left in L2. Timing:
CUDA events on the launching stream around exactly K steps, barrier +
synchronize on both sides, max over ranks. Prints one JSON line on rank 0.
The default 12000 steps run about a second back to back, long enough for the
GPU to settle at its power-capped clock; the roofline then divides by the
sustained cuBLAS figure (a timed region under a second uses the burst one).

With --gpus N (under torchrun) every rank runs its own independent problem
(output tiles need no exchange, so there is no collective on the data path):
weak scaling, value = total flops of all ranks / max time.

--impl reference times the CPU oracle (the plain fp64 triple loop in
oracle/) on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

M = N = K = 4096
FLOPS = 2.0 * M * N * K
WORKLOAD = "bf16 GEMM C=A·B, M=N=K=4096, A and B row-major bf16 uniform[-1,1) seed 0, fp32 accumulate, fp32 C"
SWEEP = [(mn, k) for mn in (512, 4096) for k in (256, 512, 1024, 4096, 8192)]
L2_BYTES = 129 * 1000 * 1000
PAGES_REF_TFLOPS = 33.72   # hgemm_bcf_dbf_rw, 4096³ bf16, GPU not stated (context only)
METRIC = "bf16 GEMM TFLOPS at 4096^3 (fp32 accumulate, fp32 C) and fraction of GB300 dense tensor peak"


def base_config():
    return {"workload": WORKLOAD, "M": M, "N": N, "K": K, "out": "f32"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=12000)   # ~1 s of back-to-back GEMMs: the sustained regime
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-sweep", action="store_true", help="skip the K sweep and the extra variants")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline leg")
    ap.add_argument("--ablation", action="store_true",
                    help="instead of the contract line: the producer × ring-depth ablation, one JSON line per run")
    ap.add_argument("--peak", action="store_true",
                    help="instead of the contract line: the tensor-pipe rate probe (MMA only) per operand layout")
    ap.add_argument("--sweep-launches", action="store_true",
                    help="instead of the contract line: two launches of each K-sweep shape (for an ncu capture)")
    ap.add_argument("--simt", action="store_true",
                    help="instead of the contract line: the CUDA-core fp32 GEMM anchor at 4096^3")
    ap.add_argument("--trace", action="store_true",
                    help="instead of the contract line: per-shape load/MMA overlap from the in-kernel timeline")
    ap.add_argument("--compare", choices=sorted(COMPARE_GROUPS),
                    help="instead of the contract line: planner alternatives timed round robin (CUDA graphs)")
    ap.add_argument("--variant-launches", choices=sorted(VARIANT_LAUNCHES),
                    help="instead of the contract line: one call per alternative after an L2 flush (for ncu)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def max_over_ranks(ms, dist, device):
    """The slowest rank's timed-region length; every rank receives it."""
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(flops_per_step, world, steps, ms_max):
    """Whole-job throughput in TFLOPS: every rank ran `steps` steps of the same
    problem (weak scaling), all done when the slowest rank finished."""
    return flops_per_step * world * steps / (ms_max * 1e-3) / 1e12


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# The sources that define the headline kernel (the two-SM GEMM, its epilogue
# helpers and PTX wrappers, its launch): a recorded ncu traffic figure stays
# valid while these are unchanged and the planner still picks the same launch.
KERNEL_SOURCES = ("ptx.cuh", "gemm_kernel.cuh", "gemm_kernel_pair.cuh", "k_pair.cu")
PLAN_KEYS = ("bn", "stages", "cta_pair", "splits", "sk_tiles", "sk_pieces", "kblocks_per_stage", "die_split",
             "l2_hints")


def _code_only(text):
    """Source text without comments and whitespace: what the compiler sees of it
    (a comment inside a string literal would be dropped too; the kernel sources
    have none that matter)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return re.sub(r"\s+", "", text)


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tensor_core_loop_gb300", "csrc")
    for name in KERNEL_SOURCES:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key, plan):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current
    kernel sources and for the launch the planner makes now."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(kernel_key)
        if (e and e.get("source_hash") == kernel_source_hash()
                and all(e.get("plan", {}).get(k) == plan.get(k) for k in PLAN_KEYS)):
            return e.get("bytes_per_launch")
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)   # let the sampler's first query land before the region opens

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]), "power": float(parts[3]),
                             "hw": parts[5], "hw_thermal": parts[6], "sw_thermal": parts[7], "sw_power": parts[8]})
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "samples_under_load": 0}
        # a sample counts as under load when the board draws more than 300 W (idle is ~150 W);
        # a timed region shorter than the sampling interval may contain none, and then the
        # nvidia-smi clock is reported as unknown rather than taken from idle samples
        loaded = [r for r in rows if r["power"] > 300.0]
        sms = sorted(r["sm"] for r in loaded)
        reasons = set()
        for r in rows:   # a throttle reason seen anywhere in the window counts
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": sms[len(sms) // 2] if sms else None, "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": max(r["power"] for r in rows)}


def cpu_oracle_sample(target_s=12.0, max_rows=4096):
    """Times the CPU oracle on whole rows of the 4096³ workload; returns (tflops, rows, seconds, cores)."""
    import oracle
    from tensor_core_loop_gb300 import inputs
    oracle.build()
    a, b = inputs.bf16_pair(M, N, K, seed=0)
    ab, bb = inputs.bf16_bits(a), inputs.bf16_bits(b)
    cores = oracle.num_threads()
    rows = max(4, cores)
    t0 = time.perf_counter()
    oracle.gemm_bf16(ab, bb, rows=(0, rows), with_abs=False)
    dt = time.perf_counter() - t0
    more = int(min(max_rows - rows, max(rows, rows * target_s / max(dt, 1e-3))))
    more = max(1, min(M - rows, (more // cores) * cores if more >= cores else more))
    t0 = time.perf_counter()
    oracle.gemm_bf16(ab, bb, rows=(rows, rows + more), with_abs=False)
    dt = time.perf_counter() - t0
    return 2.0 * more * N * K / dt / 1e12, more, dt, cores


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the platform module)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def oracle_per_config(target_s=3.0):
    """The CPU oracle timed on each workload, all host cores: the bf16 256³ case whole, and
    whole-row samples of the int8 and TF32 4096³ cases (rows scaled so each takes about
    target_s seconds). Seconds and GFLOP/s (GOP/s for int8) per workload."""
    import oracle
    from tensor_core_loop_gb300 import inputs
    oracle.build()
    res = {}
    a, b = inputs.bf16_pair(256, 256, 256, seed=0)
    ab, bb = inputs.bf16_bits(a), inputs.bf16_bits(b)
    secs = min(_timed(lambda: oracle.gemm_bf16(ab, bb, with_abs=False)) for _ in range(3))
    res["bf16 256^3 (whole C)"] = {"seconds": secs, "gflops": 2.0 * 256 ** 3 / secs / 1e9}
    cores = oracle.num_threads()
    for name, pair, fn in (("int8 4096^3", inputs.s8_pair, lambda x, y, r: oracle.gemm_s8(x, y, rows=r)),
                           ("tf32 4096^3", inputs.tf32_pair,
                            lambda x, y, r: oracle.gemm_tf32(x, y, rows=r, with_abs=False))):
        x, y = pair(M, N, K, seed=0)
        x, y = x.numpy(), y.numpy()
        rows = max(4, cores)
        dt = _timed(lambda: fn(x, y, (0, rows)))
        more = max(cores, min(M - rows, int(rows * target_s / max(dt, 1e-3)) // cores * cores))
        dt = _timed(lambda: fn(x, y, (rows, rows + more)))
        res[name] = {"seconds": dt, "rows": more, "gflops": 2.0 * more * N * K / dt / 1e9,
                     "sample": f"{more} of {M} rows of C (all {N} columns, full K={K})"}
    return res


def run_reference(args, rank, world):
    if rank != 0:
        return
    per_step = []
    rows_used = 0
    import oracle
    from tensor_core_loop_gb300 import inputs
    oracle.build()
    a, b = inputs.bf16_pair(M, N, K, seed=0)
    ab, bb = inputs.bf16_bits(a), inputs.bf16_bits(b)
    cores = oracle.num_threads()
    rows = max(16, cores)  # one bounded sample of whole C rows per step
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.gemm_bf16(ab, bb, rows=(0, rows), with_abs=False)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            per_step.append(dt)
            rows_used = rows
    total = sum(per_step)
    value = 2.0 * rows_used * N * K * len(per_step) / total / 1e12
    sample = f"{rows_used} of {M} rows of C per step (all {N} columns, full K={K})"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / len(per_step), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": base_config(),
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def oracle_one_core_256():
    """The oracle on a single host core at the small workload (bf16 256³): TFLOPS, best of 3."""
    import oracle
    from tensor_core_loop_gb300 import inputs
    a, b = inputs.bf16_pair(256, 256, 256, seed=0)
    ab, bb = inputs.bf16_bits(a), inputs.bf16_bits(b)
    threads = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        best = min(_timed(lambda: oracle.gemm_bf16(ab, bb, with_abs=False)) for _ in range(3))
    finally:
        oracle.set_num_threads(threads)
    return {"value": 2.0 * 256 ** 3 / best / 1e12, "unit": "TFLOPS", "cores": 1, "seconds": best}


def _timed(fn):
    t0 = time.perf_counter()
    fn()
    return time.perf_counter() - t0


def time_rotating(fn, sets, steps, warmup, stream, torch):
    """Back-to-back launches over rotating input sets; returns ms per step."""
    for i in range(warmup):
        fn(*sets[i % len(sets)])
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        fn(*sets[i % len(sets)])
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / steps


def time_graph_rotating(fn, sets, launches, replays, torch):
    """Back-to-back launches over rotating input sets captured into one CUDA graph (the
    host's per-call launch cost removed); returns ms per launch over `replays` replays.
    Every call runs once outside capture first, so that library scratch is in place."""
    for i in range(len(sets)):
        fn(*sets[i])
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for i in range(launches):
            fn(*sets[i % len(sets)])
    g.replay()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(replays):
        g.replay()
    end.record()
    end.synchronize()
    return start.elapsed_time(end) / (replays * launches)


def time_flushed(fn, args_, iters, stream, torch, flush):
    """Per-launch event timing with an L2 flush (a write larger than L2) before each launch."""
    times = []
    for _ in range(iters):
        flush.zero_()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn(*args_)
        e.record(stream)
        e.synchronize()
        times.append(s.elapsed_time(e))
    times.sort()
    return times[len(times) // 2]


ABLATION = [  # (label, producer, ring depth): the pages' ladder, sync copy, then cp.async, then TMA
    ("sync, 1 stage", 1, 1), ("sync, 2 stages", 1, 2), ("sync, 4 stages", 1, 4),
    ("cp.async, 1 stage", 2, 1), ("cp.async, 2 stages", 2, 2), ("cp.async, 3 stages", 2, 3),
    ("cp.async, 4 stages", 2, 4),
    ("TMA, 1 stage", 0, 1), ("TMA, 2 stages", 0, 2), ("TMA, 3 stages", 0, 3), ("TMA, 4 stages", 0, 4)]
PRODUCER_NAMES = {0: "tma", 1: "sync", 2: "cp.async"}


def compute_load_ratio(bm, bn, bk, esize):
    """Flops per loaded byte of one k-block ("流水化 GPU 内核", step 2)."""
    return 2.0 * bm * bn * bk / ((bm * bk + bk * bn) * esize)


def stage_bytes(bm, bn, bk, esize):
    """Shared-memory bytes of one ring stage: the A tile (bm × bk) and the B tile (bk × bn)."""
    a = bm * bk * esize
    b = bk * bn * esize
    return a, b, a + b


def wave_blocks(sms, blocks_per_sm):
    """Thread blocks that run at once: one wave of the grid ("4.1 CUDA GEMM 算子性能优化", §2.3)."""
    return sms * blocks_per_sm


def tile_waves(plan, sms):
    """Output tiles over the tiles one wave holds (one CTA per SM; a two-SM tile takes two)."""
    return round(plan["num_tiles"] / (wave_blocks(sms, 1) // plan["cta_pair"]), 2)


def run_ablation(args):
    import torch
    import tensor_core_loop_gb300 as tcl
    from tensor_core_loop_gb300 import inputs
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(int(2 * L2_BYTES) // 4, dtype=torch.float32, device=dev)
    shapes = [(4096, 4096, 4096)] + [(mn, mn, k) for mn, k in SWEEP if (mn, k) != (4096, 4096)]
    ratio = compute_load_ratio(128, 256, 64, 2)
    ref_out = None
    for (m, n, k) in shapes:
        ah, bh = inputs.bf16_pair(m, n, k, seed=0)
        a, b = ah.to(dev), bh.to(dev)
        c = torch.empty((m, n), dtype=torch.float32, device=dev)
        prev = None
        for label, prod, stages in ABLATION:
            cfg = tcl.Config(bn=256, stages=stages, producer=prod)
            f = (lambda cfg=cfg: tcl.gemm_into(a, b, c, cfg=cfg))
            for _ in range(3):
                f()
            ms = time_flushed(f, (), 20, stream, torch, flush)
            if (m, n, k) == (4096, 4096, 4096):
                if ref_out is None:
                    ref_out = c.clone()
                elif not torch.equal(c, ref_out):
                    raise RuntimeError(f"ablation variant {label} changed the result bits")
            tf = 2.0 * m * n * k / (ms * 1e-3) / 1e12
            line = {"ablation": label, "shape": f"{m}x{n}x{k}", "tflops": round(tf, 1), "us": round(ms * 1e3, 2),
                    "delta_vs_prev_pct": None if prev is None else round(100.0 * (tf / prev - 1.0), 1),
                    "compute_load_ratio": round(ratio, 1), "stage_bytes": stage_bytes(128, 256, 64, 2)[2],
                    "bn": 256, "stages": stages,
                    "producer": PRODUCER_NAMES[prod]}
            prev = tf
            print(json.dumps(line), flush=True)


def measure_simt(tcl, torch, dev, stream, a, b, c, flush):
    """The CUDA-core fp32 GEMM (no tensor cores) at 4096³: back to back for ~0.5 s with the SM
    clock sampled, against the FFMA peak: SMs × 128 fp32 lanes × 2 flop per fused multiply-add
    × clock."""
    fs = (lambda: tcl.gemm_simt_into(a, b, c))
    for _ in range(3):
        fs()
    ms_s = time_flushed(fs, (), 5, stream, torch, flush)
    reps = max(10, int(500.0 / max(ms_s, 1e-3)))
    smp = ClockSampler(dev.index)
    smp.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        fs()
    e1.record(stream)
    e1.synchronize()
    cl = smp.stop()
    ms_b2b = e0.elapsed_time(e1) / reps
    tf_s = FLOPS / (ms_b2b * 1e-3) / 1e12
    mhz = cl.get("sm_mhz") if cl else None
    sms = tcl.num_sms()
    peak_at = (lambda f: sms * 128 * 2 * f * 1e6 / 1e12)
    return {"tflops": round(tf_s, 2), "tflops_single_flushed": round(FLOPS / (ms_s * 1e-3) / 1e12, 2),
            "bound": "alu", "ffma_peak_at_max_clock": round(peak_at(2070.0), 2), "sm_mhz": mhz,
            "ffma_peak_at_sampled_clock": round(peak_at(mhz), 2) if mhz else None,
            "frac": round(tf_s / peak_at(mhz), 3) if mhz else None,
            "reasons": cl.get("reasons") if cl else None}


def run_sweep_launches(args):
    """Each K-sweep shape (bf16, fp32 C, the planner's launch) twice, one after the other:
    a short program for an ncu capture of the whole sweep."""
    import torch
    import tensor_core_loop_gb300 as tcl
    from tensor_core_loop_gb300 import inputs
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    for mn, k in SWEEP:
        ah, bh = inputs.bf16_pair(mn, mn, k, seed=0)
        a, b = ah.to(dev), bh.to(dev)
        c = torch.empty((mn, mn), dtype=torch.float32, device=dev)
        for _ in range(2):
            tcl.gemm_into(a, b, c)
        torch.cuda.synchronize()
        print(json.dumps({"shape": f"{mn}x{mn}x{k}", "plan": tcl.plan(tcl.IN_BF16, tcl.OUT_F32, mn, mn, k)}),
              flush=True)
        del a, b, c
    st, code = tcl.last_device_error()
    if st:
        raise RuntimeError(f"device status {st} (code {code})")


# Planner alternatives compared by --compare: per group, the workloads and the
# tcl_config_t settings; each workload's settings are timed round robin (CUDA graphs
# of back-to-back calls over rotating input sets twice the L2), median of 7 rounds,
# so that the power-capped clock's drift falls on every setting alike.
COMPARE_GROUPS = {
    "raster": ([("bf16", 4096, 4096, 4096), ("bf16", 4096, 4096, 8192), ("bf16", 8192, 8192, 4096),
                ("tf32", 4096, 4096, 4096)],
               [("group 8, K ascending", dict(group_m=8, k_order=1)), ("group 1, K ascending", dict(group_m=1, k_order=1)),
                ("group 1, K alternating", dict(group_m=1, k_order=2)),
                ("group 8, K alternating", dict(group_m=8, k_order=2))]),
    "stream_k": ([("bf16", 4096, 4096, 4096), ("bf16->bf16", 4096, 4096, 4096), ("bf16", 4096, 4096, 8192),
                  ("bf16", 4096, 4096, 2048)],
                 [("equal pieces", dict(stream_k=2)), ("balanced", dict(stream_k=5)), ("none", dict(stream_k=1))]),
    "int8": ([("s8", 4096, 4096, 4096), ("s8", 8192, 8192, 4096), ("s8", 4096, 4096, 8192)],
             [("widening pass", dict(s8_path=1)), ("in-kernel widening", dict(s8_path=2))]),
    "small": ([("bf16", 512, 512, k) for k in (256, 512, 1024, 2048, 4096, 8192)],
              [("automatic", dict()), ("64 wide", dict(bn=64, split_k=1, cluster_k=1)),
               ("64 wide, no programmatic launch", dict(bn=64, split_k=1, cluster_k=1, serial_launch=1)),
               ("64×64 tiles", dict(tile_m=64)),
               ("64 wide, cluster of 2", dict(cluster_k=2)), ("64 wide, cluster of 4", dict(cluster_k=4)),
               ("128 wide", dict(bn=128, split_k=1)),
               ("64 wide, 4 K ranges", dict(bn=64, split_k=4, cluster_k=1)),
               ("128 wide, 4 K ranges", dict(bn=128, split_k=4)),
               ("128 wide, 8 K ranges", dict(bn=128, split_k=8))]),
    "mid": ([("bf16", 1024, 4096, 4096), ("bf16", 2048, 2048, 4096), ("bf16", 1024, 4096, 1024),
             ("bf16", 2048, 2048, 1024), ("bf16", 1536, 3072, 2048), ("bf16", 3072, 3072, 1024)],
            [("automatic", dict()), ("one SM, 128 wide", dict(cta_pair=1, bn=128)),
             ("one SM, 256 wide", dict(cta_pair=1, bn=256)), ("two SMs, 256 wide", dict(cta_pair=2, bn=256)),
             ("two SMs, 224 wide", dict(cta_pair=2, bn=224))]),
    "mid_tf32": ([("tf32", 1024, 4096, 4096), ("tf32", 2048, 2048, 4096), ("tf32", 1024, 4096, 1024),
                  ("tf32", 3072, 3072, 2048)],
                 [("automatic", dict()), ("one SM, 128 wide", dict(cta_pair=1, bn=128)),
                  ("one SM, 256 wide", dict(cta_pair=1, bn=256)), ("two SMs, 256 wide", dict(cta_pair=2, bn=256)),
                  ("two SMs, 224 wide", dict(cta_pair=2, bn=224))]),
    "mid_s8": ([("s8", 1024, 4096, 4096), ("s8", 2048, 2048, 4096), ("s8", 1024, 4096, 1024),
                ("s8", 3072, 3072, 2048)],
               [("automatic", dict()), ("one SM, 128 wide", dict(cta_pair=1, bn=128)),
                ("two SMs, 256 wide", dict(cta_pair=2, bn=256)), ("two SMs, 128 wide", dict(cta_pair=2, bn=128))]),
    "short_k": ([("bf16", 4096, 4096, k) for k in (256, 512, 1024)],
                [("automatic", dict()), ("one SM, 128 wide", dict(cta_pair=1, bn=128)),
                 ("one SM, 256 wide", dict(cta_pair=1, bn=256)),
                 ("one SM, 256 wide, group 2", dict(cta_pair=1, bn=256, group_m=2)),
                 ("one SM, 256 wide, group 32", dict(cta_pair=1, bn=256, group_m=32)),
                 ("two SMs, 256 wide", dict(cta_pair=2, bn=256, stream_k=1)),
                 ("two SMs, 224 wide", dict(cta_pair=2, bn=224, stream_k=1))]),
    # the shapes the two-SM cycle constants were fitted to (the planner's pair or one-SM pick)
    "pair_fit": ([("bf16", 4096, 4096, k) for k in (768, 1024, 1536, 2048)] +
                 [("bf16", 3072, 3072, 1024), ("bf16", 3072, 3072, 2048), ("bf16", 3072, 3072, 4096),
                  ("bf16", 2048, 2048, 4096), ("bf16", 2048, 2048, 8192), ("bf16", 6144, 6144, 2048),
                  ("bf16", 1024, 1024, 8192), ("tf32", 4096, 4096, 512), ("tf32", 4096, 4096, 1024),
                  ("tf32", 2048, 2048, 2048), ("tf32", 2048, 2048, 4096), ("tf32", 3072, 3072, 2048),
                  ("s8", 4096, 4096, 1024)],
                 [("automatic", dict()), ("one SM", dict(cta_pair=1)), ("two SMs, 256 wide", dict(cta_pair=2, bn=256)),
                  ("two SMs, 224 wide", dict(cta_pair=2, bn=224))]),
    # each die's pairs on their own block of tile columns, against all pairs on all tiles
    "die_split": ([("bf16", 4096, 4096, 4096), ("bf16->bf16", 4096, 4096, 4096), ("s8", 4096, 4096, 4096),
                   ("tf32", 4096, 4096, 4096), ("bf16", 4096, 4096, 8192), ("bf16", 4096, 4096, 3072),
                   ("bf16", 6144, 4096, 4096), ("bf16", 8192, 4096, 4096), ("bf16", 3072, 3072, 4096),
                   ("bf16", 4096, 2048, 4096), ("bf16", 8192, 8192, 8192)],
                  [("automatic", dict()), ("die split off", dict(die_split=1)), ("die split on", dict(die_split=2))]),
    # the die split against K depth (two SMs per tile asked for, so that K ≤ 1024 is covered too)
    "die_split_depth": ([("bf16", 4096, 4096, k) for k in (256, 512, 1536, 2048, 2560, 3072)] +
                        [("bf16", 6144, 4096, 2048), ("bf16", 8192, 4096, 2048)] +
                        [("tf32", 4096, 4096, k) for k in (768, 1024, 2048)] + [("tf32", 6144, 4096, 1024)],
                        [("two SMs, die split off", dict(cta_pair=2, bn=256, die_split=1)),
                         ("two SMs, die split on", dict(cta_pair=2, bn=256, die_split=2))]),
    # L2 eviction priorities on the two-SM kernel's loads (A evict-first, B evict-last)
    "l2_hints": ([("bf16", 4096, 4096, 8192), ("tf32", 4096, 4096, 4096), ("bf16->bf16", 4096, 4096, 8192),
                  ("s8", 4096, 4096, 8192), ("bf16", 4096, 4096, 4096)],
                 [("automatic", dict()), ("hints off", dict(l2_hints=1)), ("hints on", dict(l2_hints=2))]),
    # tensor copies per k-block: two k-blocks per copy (two-SM 256-wide tiles), a CTA's B boxes
    # in one copy, or one copy per box and k-block
    "copies": ([("bf16", 4096, 4096, 4096), ("bf16", 4096, 4096, 8192), ("tf32", 4096, 4096, 4096),
                ("s8", 4096, 4096, 4096), ("bf16", 4096, 4096, 512), ("bf16", 8192, 8192, 512),
                ("tf32", 4096, 4096, 512), ("tf32", 2048, 2048, 2048)],
               [("automatic", dict()), ("one k-block per copy", dict(kblocks_per_stage=1)),
                ("one copy per B box", dict(kblocks_per_stage=1, b_copy=1))]),
}

# --variant-launches: one call of each alternative (after an L2 flush) for an ncu
# capture of DRAM bytes per call.
VARIANT_LAUNCHES = {
    "raster": ([("bf16", 4096, 4096, 8192), ("tf32", 4096, 4096, 4096)], COMPARE_GROUPS["raster"][1]),
    "raster_groups": ([("bf16", 4096, 4096, 8192), ("tf32", 4096, 4096, 4096)],
                      [(f"group {g}, K alternating", dict(group_m=g, k_order=2)) for g in (1, 2, 3, 4, 6, 16)]),
    "int8": ([("s8", 4096, 4096, 4096)], COMPARE_GROUPS["int8"][1]),
    "tf32": ([("tf32", 4096, 4096, 4096)], [("automatic", dict())]),
    "die_split": ([("bf16", 4096, 4096, 8192), ("tf32", 4096, 4096, 4096), ("bf16", 4096, 4096, 4096)],
                  [("die split off", dict(die_split=1)), ("die split on", dict(die_split=2))]),
    "l2_hints": ([("bf16", 4096, 4096, 8192), ("tf32", 4096, 4096, 4096), ("bf16", 4096, 4096, 4096)],
                 [("hints off", dict(l2_hints=1)), ("hints on", dict(l2_hints=2))]),
}


def _compare_operands(kind, m, n, k, dev, torch, inputs, footprint):
    gen = {"bf16": inputs.bf16_pair, "bf16->bf16": inputs.bf16_pair, "tf32": inputs.tf32_pair,
           "s8": inputs.s8_pair}[kind]
    out = {"bf16": torch.float32, "bf16->bf16": torch.bfloat16, "tf32": torch.float32, "s8": torch.int32}[kind]
    ah, bh = gen(m, n, k, seed=0)
    a0, b0 = ah.to(dev), bh.to(dev)
    per = (m * k + k * n) * a0.element_size() + m * n * torch.empty((), dtype=out).element_size()
    nset = max(2, -(-footprint // per))
    return [(a0 if i == 0 else a0.clone(), b0 if i == 0 else b0.clone(), torch.empty((m, n), dtype=out, device=dev))
            for i in range(nset)]


def run_compare(args):
    import statistics
    import torch
    import tensor_core_loop_gb300 as tcl
    from tensor_core_loop_gb300 import inputs
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    shapes, settings = COMPARE_GROUPS[args.compare]
    for kind, m, n, k in shapes:
        sets = _compare_operands(kind, m, n, k, dev, torch, inputs, 2 * L2_BYTES if kind != "s8" else L2_BYTES)
        launches = max(len(sets), 20)
        in_kind = {"bf16": tcl.IN_BF16, "bf16->bf16": tcl.IN_BF16, "tf32": tcl.IN_TF32, "s8": tcl.IN_S8}[kind]
        out = tcl.OUT_BF16 if kind == "bf16->bf16" else tcl.OUT_F32
        graphs = []
        for name, kw in settings:
            cfg = tcl.Config(**kw)
            try:   # a setting this shape or type does not allow (e.g. 224-wide int8 tiles) is skipped
                tcl.plan(in_kind, out, m, n, k, cfg)
            except tcl.TclError:
                continue
            fn = (lambda a, b, c, cfg=cfg: tcl.gemm_into(a, b, c, cfg=cfg))
            for i in range(len(sets)):
                fn(*sets[i])
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream()
            with torch.cuda.graph(g, stream=side):
                for i in range(launches):
                    fn(*sets[i % len(sets)])
            g.replay()
            torch.cuda.synchronize()
            graphs.append((name, kw, g))
        times = {name: [] for name, _, _ in graphs}
        for _ in range(7):
            for name, _, g in graphs:
                s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s_.record()
                for _ in range(3):
                    g.replay()
                e_.record()
                e_.synchronize()
                times[name].append(s_.elapsed_time(e_) * 1e3 / (3 * launches))
        st, code = tcl.last_device_error()
        if st:
            raise RuntimeError(f"device status {st} (code {code})")
        for name, kw, _ in graphs:
            med = statistics.median(times[name])
            print(json.dumps({"compare": args.compare, "workload": f"{kind} {m}x{n}x{k}", "setting": name,
                              "us_median": round(med, 2), "us_min": round(min(times[name]), 2),
                              "tflops": round(2.0 * m * n * k / med / 1e6, 1),
                              "plan": tcl.plan(in_kind, out, m, n, k, tcl.Config(**kw))}), flush=True)
        del graphs, sets


def run_variant_launches(args):
    import torch
    import tensor_core_loop_gb300 as tcl
    from tensor_core_loop_gb300 import inputs
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    flush = torch.empty(int(2 * L2_BYTES) // 4, dtype=torch.float32, device=dev)
    shapes, settings = VARIANT_LAUNCHES[args.variant_launches]
    for kind, m, n, k in shapes:
        a, b, c = _compare_operands(kind, m, n, k, dev, torch, inputs, 0)[0]
        for name, kw in settings:
            flush.zero_()
            tcl.gemm_into(a, b, c, cfg=tcl.Config(**kw))
            torch.cuda.synchronize()
            print(json.dumps({"launch": f"{kind} {m}x{n}x{k}", "setting": name}), flush=True)
        del a, b, c
    st, code = tcl.last_device_error()
    if st:
        raise RuntimeError(f"device status {st} (code {code})")


def run_simt(args):
    import torch
    import tensor_core_loop_gb300 as tcl
    from tensor_core_loop_gb300 import inputs
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(int(2 * L2_BYTES) // 4, dtype=torch.float32, device=dev)
    ah, bh = inputs.tf32_pair(M, N, K, seed=0)
    a, b = ah.to(dev), bh.to(dev)
    c = torch.empty((M, N), dtype=torch.float32, device=dev)
    line = {"simt": "fp32 GEMM on the CUDA cores, 4096^3, fp32 N(0,1) operands"}
    line.update(measure_simt(tcl, torch, dev, stream, a, b, c, flush))
    print(json.dumps(line), flush=True)


def trace_stats(t, stages, bn, num_kb, bm=128):
    """Pipeline statistics of one CTA's per-k-block stamps (issued, landed, MMAs issued, MMAs done);
    bm × bn is the CTA's share of a tile (the ideal MMA time at the pipe's 8192 flop/clk)."""
    import numpy as np
    issued, landed, mma, done = t[:, 0], t[:, 1], t[:, 2], t[:, 3]
    n = len(t)
    nd = int((done > 0).sum())
    out = {"kblocks_traced": n, "ideal_mma_cycles_per_kblock": bm * bn * 64 * 2 / 8192}
    idx = np.arange(max(0, min(nd, n - 1)))
    out["load_issued_before_prev_mma_done"] = float((issued[idx + 1] < done[idx]).mean()) if len(idx) else None
    idx2 = np.arange(max(0, min(nd, n - (stages - 1))))
    out["load_k_plus_stages_minus_1_before_mma_k_done"] = (
        float((issued[idx2 + stages - 1] < done[idx2]).mean()) if len(idx2) and stages > 1 else None)
    if n <= stages - 1 and nd >= 1:
        # a walk shorter than the ring: were all of its loads in flight before the first MMAs finished?
        out["all_loads_issued_before_first_mma_done"] = bool(issued[n - 1] < done[0])
    issue = mma - landed                     # MMA warp: issue 4 MMAs + commit
    out["mma_issue_cycles"] = {"p50": float(np.median(issue)), "mean": float(issue.mean())}
    if n > 1:
        gap = landed[1:] - mma[:-1]          # MMA warp: waiting for the next stage's barrier
        out["mma_wait_cycles"] = {"p50": float(np.median(gap)), "mean": float(gap.mean()),
                                  "p90": float(np.percentile(gap, 90))}
    lat = landed - issued
    out["load_latency_cycles"] = {"mean": float(lat.mean()), "p50": float(np.median(lat)),
                                  "p90": float(np.percentile(lat, 90))}
    if nd >= 2:
        d = done[:nd]
        busy_iv = np.diff(d)
        out["mma_done_interval_cycles"] = {"mean": float(busy_iv.mean()), "p50": float(np.median(busy_iv)),
                                           "p90": float(np.percentile(busy_iv, 90))}
        # tensor pipe idle before block k: its data landed after block k-1 had finished
        starve = np.maximum(0, landed[1:nd] - d[:nd - 1])
        span = float(d[nd - 1] - landed[0])
        out["pipe_starved_frac"] = float(starve.sum()) / span if span > 0 else None
        tile_starts = np.arange(num_kb, nd, num_kb)
        out["starved_cycles_at_tile_starts"] = float(starve[tile_starts - 1].sum()) if len(tile_starts) else 0.0
        out["busy_frac_of_span"] = (nd * out["ideal_mma_cycles_per_kblock"]) / span if span > 0 else None
    return out


def run_trace(args):
    import numpy as np
    import torch
    import tensor_core_loop_gb300 as tcl
    from tensor_core_loop_gb300 import inputs
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    shapes = [(mn, mn, k) for mn, k in SWEEP]
    for (m, n, k) in shapes:
        ah, bh = inputs.bf16_pair(m, n, k, seed=0)
        a, b = ah.to(dev), bh.to(dev)
        for pair in ((1, 2) if m >= 4096 else (1,)):
            cfg0 = tcl.Config(cta_pair=pair, split_k=1)
            pl = tcl.plan(tcl.IN_BF16, tcl.OUT_F32, m, n, k, cfg0)
            num_kb = -(-k // 64)
            clusters = pl["grid"] // (2 if pl["cta_pair"] == 2 else 1)
            tiles_cta0 = -(-pl["num_tiles"] // clusters)
            cap = min(8192, tiles_cta0 * num_kb)
            trace = torch.zeros(4 * cap + 4, dtype=torch.int64, device=dev)
            cfg = tcl.Config(cta_pair=pair, split_k=1, trace=trace.data_ptr(), trace_cap=cap)
            for _ in range(3):
                trace.zero_()
                tcl.gemm(a, b, cfg=cfg)
            torch.cuda.synchronize()
            tt = trace.cpu().numpy().astype(np.int64)
            t = tt[:4 * cap].reshape(cap, 4)
            t = t[:int((t[:, 0] > 0).sum())]   # k-blocks CTA 0 actually ran (a stream-K tail makes fewer)
            c0, g0, c1, g1 = tt[4 * cap:]
            line = {"trace": f"{m}x{n}x{k}", "sm_mhz_in_kernel": round(1e3 * (c1 - c0) / max(1, g1 - g0), 1),
                    "cta_pair": pl["cta_pair"], "tile_m": pl["tile_m"], "bn": pl["bn"], "stages": pl["stages"],
                    "tiles_cta0": tiles_cta0}
            # each SM computes 128 rows (64 on 64-row tiles) × bn columns per k-block
            line.update(trace_stats(t, pl["stages"], pl["bn"], num_kb, bm=64 if pl["tile_m"] == 64 else 128))
            print(json.dumps(line), flush=True)


def run_peak(args):
    import torch
    import tensor_core_loop_gb300 as tcl
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sms = tcl.num_sms()
    sampler = ClockSampler(0)
    sampler.start()
    rows = []
    combos = [(0, 256, 1), (0, 256, 0), (0, 224, 1), (0, 192, 1), (0, 128, 1), (0, 128, 0), (1, 256, 0),
              (1, 128, 0)]
    # flags: 2 = walk operands like a k-loop; 11 = also one chained accumulator and the
    # rest of a GEMM issue loop (barrier wait, fence, commit per four MMAs)
    for kind, n, b_mn, flags in [c + (f,) for c in combos for f in (2, 11)]:
        tcl.mma_peak(kind, n, b_mn, iters=512, flags=flags)          # warm-up
        cyc, rate, ms = tcl.mma_peak(kind, n, b_mn, iters=16384, flags=flags)
        k = 16 if kind == 0 else 8
        flops = 2.0 * 128 * n * k * 16384 * sms
        rows.append({"peak": "bf16" if kind == 0 else "tf32", "n": n, "b_major": "MN" if b_mn else "K",
                     "one_accumulator": bool(flags & 1), "walk_operands": bool(flags & 2),
                     "gemm_issue_loop": bool(flags & 8),
                     "flop_per_clk_per_sm": round(rate, 1), "cycles_per_mma": round(max(cyc) / 16384, 2),
                     "tflops_all_sms": round(flops / (ms * 1e-3) / 1e12, 1), "sms": sms})
    # the warp-level mma.sync forms the pages' kernels use: int8 m16n8k32 (the only int8
    # tensor instruction sm_103a has) and bf16 m16n8k16
    for kind, flags, name, ops in ((2, 0, "int8 mma.sync m16n8k32", 8192), (0, 128, "bf16 mma.sync m16n8k16", 4096)):
        tcl.mma_peak(kind, 128, 0, iters=512, flags=flags)
        cyc, rate, ms = tcl.mma_peak(kind, 128, 0, iters=16384, flags=flags)
        total = 64.0 * 16384 * ops * sms
        rows.append({"peak": name, "op_per_clk_per_sm": round(rate, 1),
                     "tops_all_sms": round(total / (ms * 1e-3) / 1e12, 1), "sms": sms})
    clocks = sampler.stop()
    for r in rows:
        r["clocks"] = clocks
        print(json.dumps(r), flush=True)


def in_kernel_clock_mhz(tcl, torch, sets, stream, steps):
    """SM clock inside the GEMM under the timed workload: back-to-back launches with CTA 0
    stamping %clock64 and %globaltimer at its start and end; median over the last launches."""
    import ctypes
    cap = 1
    bufs = [torch.zeros(4 * cap + 4, dtype=torch.int64, device=sets[0][0].device) for _ in range(8)]
    L = tcl.lib()
    mhz = []
    for i in range(steps):
        buf = bufs[i % len(bufs)]
        cfg = tcl.Config(trace=buf.data_ptr(), trace_cap=cap)
        a, b, c = sets[i % len(sets)]
        st = L.gemm_bf16_ex(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N, tcl.OUT_F32,
                            ctypes.byref(cfg), ctypes.c_void_p(stream.cuda_stream))
        if st:
            return None
    torch.cuda.synchronize()
    for buf in bufs:
        c0, g0, c1, g1 = buf[4 * cap:].cpu().tolist()
        if g1 > g0:
            mhz.append(1e3 * (c1 - c0) / (g1 - g0))
    mhz.sort()
    return mhz[len(mhz) // 2] if mhz else None


def measured_mma_rate(tcl):
    """flop/clk/SM of the bf16 N=256 tensor pipe, from the MMA-only probe (None on failure)."""
    try:
        tcl.mma_peak(0, 256, 1, iters=256)
        return tcl.mma_peak(0, 256, 1, iters=4096, flags=2)[1]
    except Exception:
        return None


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.ablation:
        run_ablation(args)
        return
    if args.trace:
        run_trace(args)
        return
    if args.peak:
        run_peak(args)
        return
    if args.simt:
        run_simt(args)
        return
    if args.sweep_launches:
        run_sweep_launches(args)
        return
    if args.compare:
        run_compare(args)
        return
    if args.variant_launches:
        run_variant_launches(args)
        return

    import torch
    import torch.distributed as dist

    import tensor_core_loop_gb300 as tcl
    from tensor_core_loop_gb300 import inputs

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    stream = torch.cuda.current_stream(dev)
    peaks, peak_src = measured_peaks()

    # ---- inputs: rotate over sets whose total footprint exceeds L2
    a_h, b_h = inputs.bf16_pair(M, N, K, seed=0)
    set_bytes = M * K * 2 + K * N * 2 + M * N * 4
    nsets = max(2, -(-3 * L2_BYTES // set_bytes))
    a0, b0 = a_h.to(dev), b_h.to(dev)
    sets = []
    for i in range(nsets):
        ai = a0 if i == 0 else a0.clone()
        bi = b0 if i == 0 else b0.clone()
        sets.append((ai, bi, torch.empty((M, N), dtype=torch.float32, device=dev)))
    L = tcl.lib()

    def step(a, b, c):
        st = L.gemm_bf16(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N, tcl.OUT_F32,
                         stream.cuda_stream)
        if st:
            raise tcl.TclError(st, "gemm_bf16")

    for i in range(max(3, args.warmup)):
        step(*sets[i % nsets])
    torch.cuda.synchronize()

    sampler = ClockSampler(dev.index if world == 1 else local)
    if rank == 0:
        sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        step(*sets[i % nsets])
    end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms_total = start.elapsed_time(end)
    clocks = sampler.stop() if rank == 0 else None
    if world > 1:
        ms_total = max_over_ranks(ms_total, dist, dev)
    st, code = tcl.last_device_error()
    if st:
        raise RuntimeError(f"device status {st} (code {code}) after the timed region")
    kernel_mhz = None
    if rank == 0:
        kernel_mhz = in_kernel_clock_mhz(tcl, torch, sets, stream, steps=min(args.steps, 2000))
    ms_step = ms_total / args.steps
    if rank == 0:
        print(f"[bench] {args.steps} steps, {ms_step * 1e3:.2f} us/step, "
              f"{FLOPS / (ms_step * 1e-3) / 1e12:.1f} TFLOPS per GPU; clocks {clocks}", file=sys.stderr, flush=True)
    value = job_value(FLOPS, world, args.steps, ms_total)
    per_launch_s = ms_step * 1e-3
    achieved = FLOPS / per_launch_s / 1e12

    extra = {}
    if rank == 0 and not args.no_sweep:
        # bf16 output variant of the same workload
        sets16 = [(s[0], s[1], torch.empty((M, N), dtype=torch.bfloat16, device=dev)) for s in sets]

        def step16(a, b, c):
            st_ = L.gemm_bf16(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N, tcl.OUT_BF16,
                              stream.cuda_stream)
            if st_:
                raise tcl.TclError(st_, "gemm_bf16")
        ms16 = time_rotating(step16, sets16, 500, 20, stream, torch)
        extra["bf16_out_tflops"] = FLOPS / (ms16 * 1e-3) / 1e12
        del sets16
        # K sweep: back-to-back launches over rotating input/output sets whose footprint is
        # twice the L2, so every launch starts cold in L2 (single-launch event timing is
        # quantised at ~2 µs on this GPU, too coarse for the smallest shapes). "us" is
        # taken from a CUDA graph of those launches (what the GPU takes per call);
        # "us_host_launch" from the same launches issued one by one from Python, whose
        # per-call host cost (ctypes and the library's host code) shows at the small shapes
        sweep = {}
        for mn, k in SWEEP:
            ah, bh = inputs.bf16_pair(mn, mn, k, seed=0)
            a0_, b0_ = ah.to(dev), bh.to(dev)
            sbytes = 2 * mn * k * 2 + mn * mn * 4
            nset = max(2, -(-2 * L2_BYTES // sbytes))
            ssets = [(a0_ if i == 0 else a0_.clone(), b0_ if i == 0 else b0_.clone(),
                      torch.empty((mn, mn), dtype=torch.float32, device=dev)) for i in range(nset)]

            def f(a, b, c, mn=mn, k=k):
                st_ = L.gemm_bf16(mn, mn, k, a.data_ptr(), k, b.data_ptr(), mn, c.data_ptr(), mn, tcl.OUT_F32,
                                  torch.cuda.current_stream().cuda_stream)
                if st_:
                    raise tcl.TclError(st_, "gemm_bf16")
            ms_host = time_rotating(f, ssets, max(60, 2 * nset), 2 * nset, stream, torch)
            ms = time_graph_rotating(f, ssets, max(40, 2 * nset), 5, torch)
            tf = 2.0 * mn * mn * k / (ms * 1e-3) / 1e12
            alg_bytes = (mn * k + k * mn) * 2 + mn * mn * 4
            sweep[f"{mn}x{mn}x{k}"] = {"tflops": round(tf, 1), "us": round(ms * 1e3, 2),
                                        "us_host_launch": round(ms_host * 1e3, 2),
                                        "alg_gbs": round(alg_bytes / (ms * 1e-3) / 1e9, 1),
                                        "plan": tcl.plan(tcl.IN_BF16, tcl.OUT_F32, mn, mn, k)}
            del ssets, a0_, b0_
        extra["k_sweep"] = sweep
        extra["k_sweep_timing"] = ("us: mean of back-to-back launches over rotating sets (footprint 2x L2) "
                                   "captured in a CUDA graph; us_host_launch: the same launches issued one "
                                   "by one from Python")
        flush = torch.empty(int(2 * L2_BYTES) // 4, dtype=torch.float32, device=dev)
        # the other two workloads at 4096³, whole call (int8 → exact int32: widening pass +
        # GEMM; TF32: the GEMM alone, B read in place), timed like the headline (back-to-back
        # launches over rotating input sets whose footprint exceeds L2) and, beside it, each
        # launch alone after an L2 flush (host launch latency included)
        def whole_call(pair_fn, out_dtype):
            xh, yh = pair_fn(M, N, K, seed=0)
            x0, y0 = xh.to(dev), yh.to(dev)
            per = (x0.numel() + y0.numel()) * x0.element_size() + M * N * 4
            nset_ = max(2, -(-2 * L2_BYTES // per))
            sets_ = [(x0 if i == 0 else x0.clone(), y0 if i == 0 else y0.clone(),
                      torch.empty((M, N), dtype=out_dtype, device=dev)) for i in range(nset_)]
            fn = (lambda x, y, z: tcl.gemm_into(x, y, z))
            ms_rot = time_rotating(fn, sets_, 200, 20, stream, torch)
            ms_graph = time_graph_rotating(fn, sets_, max(40, 2 * nset_), 5, torch)
            x, y, z = sets_[0]
            ms_one = time_flushed(lambda: fn(x, y, z), (), 20, stream, torch, flush)
            return ms_rot, ms_graph, ms_one, sets_[0]
        ms8, ms8_graph, ms8_one, _ = whole_call(inputs.s8_pair, torch.int32)
        extra["int8_tops_4096"] = round(FLOPS / (ms8 * 1e-3) / 1e12, 1)
        extra["int8_tops_4096_graph"] = round(FLOPS / (ms8_graph * 1e-3) / 1e12, 1)
        extra["int8_tops_4096_single_flushed"] = round(FLOPS / (ms8_one * 1e-3) / 1e12, 1)
        mst, mst_graph, mst_one, (at, bt, ct) = whole_call(inputs.tf32_pair, torch.float32)
        extra["tf32_tflops_4096"] = round(FLOPS / (mst * 1e-3) / 1e12, 1)
        extra["tf32_tflops_4096_graph"] = round(FLOPS / (mst_graph * 1e-3) / 1e12, 1)
        extra["tf32_tflops_4096_single_flushed"] = round(FLOPS / (mst_one * 1e-3) / 1e12, 1)
        extra["int8_tf32_timing"] = ("*_4096: back-to-back whole calls over rotating input sets (footprint "
                                     "> 2x L2), issued one by one from Python, as the headline; *_graph: the "
                                     "same calls captured in a CUDA graph (the host's per-call cost removed; "
                                     "int8: widening pass and GEMM per call); *_single_flushed: one call "
                                     "after an L2 flush")
        extra["sgemm_simt_4096"] = measure_simt(tcl, torch, dev, stream, at, bt, ct, flush)
        del at, bt, ct
        del flush

    # ---- end to end through the public API with host buffers
    e2e = None
    if rank == 0:
        # the host-buffer call of the C ABI: it uploads A and B, runs the GEMM and
        # downloads C, pipelined over row chunks, every step inside the timed region
        a_pin = a_h.pin_memory()
        b_pin = b_h.pin_memory()
        c_pin = torch.empty((M, N), dtype=torch.float32).pin_memory()

        def e2e_step():
            tcl.gemm_host_into(a_pin, b_pin, c_pin, stream=stream)
        e2e_steps = max(5, min(50, args.steps))
        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e.record(stream)
        e.synchronize()
        ms_e2e = s.elapsed_time(e) / e2e_steps
        e2e = {"value": FLOPS / (ms_e2e * 1e-3) / 1e12, "unit": "TFLOPS",
               "h2d_bytes_per_step": a_pin.numel() * 2 + b_pin.numel() * 2,
               "d2h_bytes_per_step": c_pin.numel() * 4, "ms_per_step": ms_e2e}

    cpu = None
    if rank == 0 and not args.no_cpu:
        tf, rows, secs, cores = cpu_oracle_sample()
        cpu = {"value": tf, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
               "sample": f"{rows} of {M} rows of C (all {N} columns, full K={K}), {secs:.1f} s",
               "seconds": secs, "gflops": tf * 1e3,
               "host_cpu_count": os.cpu_count(), "cpu_model": cpu_model(),
               "one_core_256": oracle_one_core_256(),
               "per_config": oracle_per_config()}

    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return

    # The denominator follows the regime the timed region ran in: a region of a
    # second or more of back-to-back launches runs at the power-capped sustained
    # clock, like the sustained cuBLAS figure; a shorter one compares with the burst.
    sustained = ms_total >= 1000.0 and "bf16_tflops_sustained" in peaks
    peak = float(peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"])
    sms = tcl.num_sms()
    sm_mhz = clocks.get("sm_mhz") if clocks else None
    rate = measured_mma_rate(tcl) or 8192.0
    clk = kernel_mhz or sm_mhz
    cc_peak = (sms * rate * clk * 1e6 / 1e12) if clk else None
    # the same pipe rate at the GPU's maximum SM clock (nvidia-smi clocks.max.sm)
    max_mhz = clocks.get("sm_max_mhz") if clocks else None
    max_peak = (sms * rate * max_mhz * 1e6 / 1e12) if max_mhz else None
    if clocks is not None:
        # the primary clock is the one measured inside the GEMM on the timed workload; the
        # nvidia-smi median (samples drawing > 300 W during the timed region) sits beside
        # it and is null when the region was too short to be sampled under load
        clocks["sm_mhz_nvidia_smi"] = clocks.get("sm_mhz")
        clocks["sm_mhz_in_kernel"] = kernel_mhz
        if kernel_mhz:
            clocks["sm_mhz"] = round(kernel_mhz, 1)
            clocks["sm_mhz_source"] = ("in kernel: CTA 0's %clock64 over %globaltimer, median of back-to-back "
                                       "launches of the timed workload")
        else:
            clocks["sm_mhz_source"] = "nvidia-smi, samples under load during the timed region"
    line = {
        "metric": METRIC,
        "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": value / world / PAGES_REF_TFLOPS,
        "dtype": "bf16", "data": "synthetic",
        "config": {**base_config(),
                   "l2": f"inputs rotated over {nsets} sets of {set_bytes >> 20} MiB (> 129 MB L2)",
                   "vs_baseline_ref": "pages' hgemm_bcf_dbf_rw 4096^3 bf16 33.72 TFLOPS, GPU not stated (context)",
                   "plan": tcl.plan(tcl.IN_BF16, tcl.OUT_F32, M, N, K), "sms": sms,
                   "tile_waves": tile_waves(tcl.plan(tcl.IN_BF16, tcl.OUT_F32, M, N, K), sms)},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": recorded_traffic("gemm_bf16_f32_4096", tcl.plan(tcl.IN_BF16, tcl.OUT_F32, M, N, K)),
                     "peak_source": (f"{peak_src} bf16_tflops_sustained (cuBLAS 8192^3 back to back for 4 s; "
                                     f"the timed region ran {ms_total / 1e3:.2f} s back to back)") if sustained
                                    else f"{peak_src} bf16_tflops (cuBLAS 8192^3 burst)",
                     "frac_of_burst": achieved / float(peaks["bf16_tflops"]),
                     "frac_of_sustained": (achieved / float(peaks["bf16_tflops_sustained"])
                                           if "bf16_tflops_sustained" in peaks else None),
                     "mma_rate_flop_per_clk_per_sm": rate,
                     "clock_corrected_peak": cc_peak,
                     "clock_corrected_peak_def": "SMs x probe-measured flop/clk/SM x SM clock measured inside "
                                                 "the kernel (%clock64 / %globaltimer) on the timed workload",
                     "frac_clock_corrected": (achieved / cc_peak) if cc_peak else None,
                     "max_clock_peak": max_peak,
                     "frac_of_max_clock": (achieved / max_peak) if max_peak else None},
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "cpu_baseline": cpu,
    }
    line.update(extra)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
