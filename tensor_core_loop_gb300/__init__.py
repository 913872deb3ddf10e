"""GB300 (sm_103a) pipelined tensor-core GEMM: Python binding of the C ABI.

The work happens in ``libtcl_gb300.so`` (built from ``csrc/`` by
``_build.build()``); this module only marshals arguments: it passes device
pointers, leading dimensions and the current CUDA stream of PyTorch tensors to
the C entry points declared in ``include/tcl_gemm.h`` and turns a nonzero
status into an exception. PyTorch supplies device memory and streams only.
There is no fallback: if the library is missing or the device is not an
sm_103 GPU, calls raise.

    C = gemm(A, B)                      # bf16 -> fp32, tf32 (fp32 in) -> fp32, int8 -> int32
    C = gemm(A, B, out_dtype=torch.bfloat16)
"""
from __future__ import annotations

import ctypes
import os
import threading

from ._build import LIB_PATH

__all__ = ["gemm", "gemm_into", "gemm_host_into", "gemm_simt_into", "plan", "lib", "Config", "last_device_error", "num_sms", "version",
           "TclError", "STATUS", "EXPORTED_SYMBOLS"]

STATUS = {
    0: "TCL_OK", 1: "TCL_ERR_NULL", 2: "TCL_ERR_DIMS", 3: "TCL_ERR_LD", 4: "TCL_ERR_ALIGN",
    5: "TCL_ERR_K_TOO_LARGE", 6: "TCL_ERR_LAUNCH", 7: "TCL_ERR_DEVICE_TIMEOUT", 8: "TCL_ERR_CONFIG",
    9: "TCL_ERR_NO_MEMORY", 10: "TCL_ERR_DEVICE", 11: "TCL_ERR_STATIC_LIMIT", 12: "TCL_ERR_CAPTURE",
}
OUT_F32, OUT_BF16 = 0, 1
PRODUCER_TMA, PRODUCER_SYNC, PRODUCER_CPASYNC = 0, 1, 2
IN_BF16, IN_TF32, IN_S8 = 0, 1, 2

EXPORTED_SYMBOLS = ("gemm_bf16", "gemm_tf32", "gemm_s8", "gemm_bf16_ex", "gemm_tf32_ex", "gemm_s8_ex",
                    "tcl_plan", "tcl_status_string", "tcl_last_device_error", "tcl_num_sms", "tcl_die_pairs",
                    "tcl_shutdown", "tcl_version", "gemm_s8_static", "tcl_mma_peak", "gemm_f32_simt",
                    "gemm_bf16_host", "tcl_stream_release")


class TclError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        text = STATUS.get(status, str(status))
        try:
            text += ": " + lib().tcl_status_string(status).decode()
        except Exception:
            pass
        super().__init__(f"{what}{' ' if what else ''}failed with {text}")


class Config(ctypes.Structure):
    """Mirror of ``tcl_config_t`` (zero = automatic)."""
    _fields_ = [
        ("bn", ctypes.c_int),
        ("stages", ctypes.c_int),
        ("one_cta_per_tile", ctypes.c_int),
        ("group_m", ctypes.c_int),
        ("max_ctas", ctypes.c_int),
        ("timeout_ns", ctypes.c_ulonglong),
        ("trace", ctypes.c_void_p),
        ("trace_cap", ctypes.c_int),
        ("producer", ctypes.c_int),
        ("split_k", ctypes.c_int),
        ("cta_pair", ctypes.c_int),
        ("epi_slots", ctypes.c_int),
        ("debug_skip_kblock", ctypes.c_int),
        ("stream_k", ctypes.c_int),
        ("serial_launch", ctypes.c_int),
        ("debug_stream_k_stall", ctypes.c_int),
        ("k_order", ctypes.c_int),
        ("s8_path", ctypes.c_int),
        ("cluster_k", ctypes.c_int),
        ("tile_m", ctypes.c_int),
        ("kblocks_per_stage", ctypes.c_int),
        ("b_copy", ctypes.c_int),
        ("die_split", ctypes.c_int),
        ("l2_hints", ctypes.c_int),
    ]


class PlanInfo(ctypes.Structure):
    """Mirror of ``tcl_plan_t``."""
    _fields_ = [
        ("bn", ctypes.c_int),
        ("stages", ctypes.c_int),
        ("grid", ctypes.c_int),
        ("num_tiles", ctypes.c_int),
        ("smem_bytes", ctypes.c_int),
        ("cta_pair", ctypes.c_int),
        ("splits", ctypes.c_int),
        ("producer", ctypes.c_int),
        ("workspace_bytes", ctypes.c_ulonglong),
        ("sk_tiles", ctypes.c_int),
        ("sk_pieces", ctypes.c_int),
        ("sk_balanced", ctypes.c_int),
        ("group_m", ctypes.c_int),
        ("k_serpentine", ctypes.c_int),
        ("s8_in_kernel", ctypes.c_int),
        ("cluster_k", ctypes.c_int),
        ("tile_m", ctypes.c_int),
        ("kblocks_per_stage", ctypes.c_int),
        ("die_split", ctypes.c_int),
        ("die_tiles0", ctypes.c_int),
        ("l2_hints", ctypes.c_int),
    ]


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        I, P = ctypes.c_int, ctypes.c_void_p
        CP = ctypes.POINTER(Config)
        L.gemm_bf16.argtypes = [I, I, I, P, I, P, I, P, I, I, P]
        L.gemm_bf16_ex.argtypes = [I, I, I, P, I, P, I, P, I, I, CP, P]
        for name in ("gemm_tf32", "gemm_s8"):
            getattr(L, name).argtypes = [I, I, I, P, I, P, I, P, I, P]
            getattr(L, name + "_ex").argtypes = [I, I, I, P, I, P, I, P, I, CP, P]
        L.gemm_s8_static.argtypes = [I, I, I, P, I, P, I, P, I, P]
        L.gemm_f32_simt.argtypes = [I, I, I, P, I, P, I, P, I, P]
        L.gemm_bf16_host.argtypes = [I, I, I, P, I, P, I, P, I, I, P]
        L.tcl_mma_peak.argtypes = [I, I, I, I, I, I, P, P]
        IP = ctypes.POINTER(ctypes.c_int)
        L.tcl_plan.argtypes = [I, I, I, I, I, CP, ctypes.POINTER(PlanInfo)]
        L.tcl_status_string.argtypes = [I]
        L.tcl_status_string.restype = ctypes.c_char_p
        L.tcl_last_device_error.argtypes = [P, IP]
        L.tcl_num_sms.argtypes = []
        L.tcl_die_pairs.argtypes = [IP, IP]
        L.tcl_shutdown.argtypes = []
        L.tcl_shutdown.restype = None
        L.tcl_stream_release.argtypes = [P]
        L.tcl_version.restype = ctypes.c_char_p
        _lib = L
        return L


def version() -> str:
    return lib().tcl_version().decode()


def num_sms() -> int:
    return int(lib().tcl_num_sms())


def die_pairs() -> tuple:
    """Pairs of SMs on each die of the current device as the die split measured them
    ((0, 0): not known, no die split)."""
    n0, n1 = ctypes.c_int(0), ctypes.c_int(0)
    st = lib().tcl_die_pairs(ctypes.byref(n0), ctypes.byref(n1))
    if st:
        raise TclError(st, "tcl_die_pairs")
    return n0.value, n1.value


def plan(in_kind: int, out: int, M: int, N: int, K: int, cfg: Config | None = None) -> dict:
    """The launch the library would make (tile width, ring depth, grid, tiles, shared memory,
    one or two SMs per tile, split-K ranges, producer kind, workspace bytes)."""
    info = PlanInfo()
    st = lib().tcl_plan(in_kind, out, M, N, K, ctypes.byref(cfg) if cfg else None, ctypes.byref(info))
    if st:
        raise TclError(st, "tcl_plan")
    return {name: getattr(info, name) for name, _ in PlanInfo._fields_}


def mma_peak(in_kind: int = IN_BF16, n: int = 256, b_mn: int = 0, iters: int = 4096, grid: int | None = None,
             flags: int = 0):
    """Runs the tensor-pipe probe on every SM; returns (cycles per CTA as a list, flop/clk/SM of the
    slowest CTA, elapsed ms of the launch measured with CUDA events). ``in_kind=IN_S8`` (or
    ``flags=128`` with bf16) times the warp-level ``mma.sync`` forms instead."""
    import torch
    grid = grid or num_sms()
    cyc = torch.zeros(grid, dtype=torch.int64, device="cuda")
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    st = lib().tcl_mma_peak(in_kind, n, b_mn, flags, iters, grid, cyc.data_ptr(), ctypes.c_void_p(s.cuda_stream))
    e1.record(s)
    if st:
        raise TclError(st, "tcl_mma_peak")
    e1.synchronize()
    c = cyc.cpu().tolist()
    worst = max(c) if min(c) > 0 else 0
    if in_kind == IN_S8 or flags & 128:   # warp-level mma.sync: 8 warps × 8 chains × iters per CTA
        rate = 64.0 * iters * (8192 if in_kind == IN_S8 else 4096) / worst if worst else 0.0
    else:
        k = 16 if in_kind == IN_BF16 else 8
        rate = 2.0 * 128 * n * k * iters / worst if worst else 0.0
    return c, rate, e0.elapsed_time(e1)


def last_device_error(stream=None) -> tuple[int, int]:
    """(status, raw device code) after synchronising the stream; clears the word."""
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    detail = ctypes.c_int(0)
    st = lib().tcl_last_device_error(ctypes.c_void_p(s.cuda_stream), ctypes.byref(detail))
    return int(st), int(detail.value)


def stream_release(stream) -> None:
    """Frees the scratch and stream-K flags the library holds for `stream` (a torch
    stream), after synchronising it; call before destroying a stream."""
    st = lib().tcl_stream_release(ctypes.c_void_p(stream.cuda_stream))
    if st:
        raise TclError(st, "tcl_stream_release")


def _ld(t) -> int:
    """Leading dimension in elements. A one-row matrix never steps to a second
    row, so its leading dimension is free: report the row width rounded up to
    16 bytes, which satisfies the library's alignment rule."""
    if t.dim() != 2:
        raise ValueError("expected a 2-D tensor")
    if t.stride(1) != 1 and t.shape[1] > 1:
        raise ValueError("rows must be contiguous (stride(1) == 1)")
    if t.shape[0] > 1:
        return max(t.stride(0), t.shape[1])
    q = max(1, 16 // t.element_size())
    return -(-t.shape[1] // q) * q


def gemm_host_into(a, b, c, stream=None) -> None:
    """C = A·B for bf16 CPU tensors (page-locked for overlap) into the CPU tensor ``c``
    (float32 or bfloat16): uploads, GEMMs and downloads pipelined by the library.
    Asynchronous on ``stream`` (default: the current CUDA stream): ``c`` is ready
    once that stream is synchronised."""
    import torch
    if a.is_cuda or b.is_cuda or c.is_cuda:
        raise ValueError("a, b and c must be CPU tensors")
    if a.dtype != torch.bfloat16 or b.dtype != torch.bfloat16:
        raise TypeError("the host-buffer GEMM takes bf16 a and b")
    out = {torch.float32: OUT_F32, torch.bfloat16: OUT_BF16}.get(c.dtype)
    if out is None:
        raise TypeError("c must be float32 or bfloat16")
    M, K = a.shape
    K2, N = b.shape
    if K != K2 or tuple(c.shape) != (M, N):
        raise ValueError(f"shape mismatch: {tuple(a.shape)} x {tuple(b.shape)} -> {tuple(c.shape)}")
    s = stream if stream is not None else torch.cuda.current_stream()
    st = lib().gemm_bf16_host(M, N, K, a.data_ptr(), _ld(a), b.data_ptr(), _ld(b), c.data_ptr(), _ld(c), out,
                              ctypes.c_void_p(s.cuda_stream))
    if st:
        raise TclError(st, "gemm_bf16_host")


def gemm_simt_into(a, b, c, stream=None) -> None:
    """C = A·B for fp32 CUDA tensors on the CUDA cores (fp32 FMA, no tensor cores), into ``c``."""
    import torch
    if not (a.is_cuda and b.is_cuda and c.is_cuda):
        raise ValueError("a, b and c must be CUDA tensors")
    if not (a.dtype == b.dtype == c.dtype == torch.float32):
        raise TypeError("the SIMT GEMM takes and writes float32")
    M, K = a.shape
    K2, N = b.shape
    if K != K2 or tuple(c.shape) != (M, N):
        raise ValueError(f"shape mismatch: {tuple(a.shape)} x {tuple(b.shape)} -> {tuple(c.shape)}")
    s = stream if stream is not None else torch.cuda.current_stream(a.device)
    with torch.cuda.device(a.device):
        st = lib().gemm_f32_simt(M, N, K, a.data_ptr(), _ld(a), b.data_ptr(), _ld(b), c.data_ptr(), _ld(c),
                                 ctypes.c_void_p(s.cuda_stream))
    if st:
        raise TclError(st, "gemm_f32_simt")


def gemm_into(a, b, c, cfg: Config | None = None, stream=None) -> None:
    """C = A·B written into the preallocated CUDA tensor ``c`` (overwritten)."""
    import torch
    if not (a.is_cuda and b.is_cuda and c.is_cuda):
        raise ValueError("a, b and c must be CUDA tensors")
    M, K = a.shape
    K2, N = b.shape
    if K != K2 or tuple(c.shape) != (M, N):
        raise ValueError(f"shape mismatch: {tuple(a.shape)} x {tuple(b.shape)} -> {tuple(c.shape)}")
    if b.dtype != a.dtype:
        raise TypeError("a and b must have the same dtype")
    s = stream if stream is not None else torch.cuda.current_stream(a.device)
    sp = ctypes.c_void_p(s.cuda_stream)
    cp = ctypes.byref(cfg) if cfg is not None else None
    L = lib()
    with torch.cuda.device(a.device):
        if a.dtype == torch.bfloat16:
            if c.dtype == torch.float32:
                out = OUT_F32
            elif c.dtype == torch.bfloat16:
                out = OUT_BF16
            else:
                raise TypeError("bf16 GEMM writes float32 or bfloat16")
            st = L.gemm_bf16_ex(M, N, K, a.data_ptr(), _ld(a), b.data_ptr(), _ld(b), c.data_ptr(), _ld(c),
                                out, cp, sp)
        elif a.dtype == torch.float32:
            if c.dtype != torch.float32:
                raise TypeError("tf32 GEMM writes float32")
            st = L.gemm_tf32_ex(M, N, K, a.data_ptr(), _ld(a), b.data_ptr(), _ld(b), c.data_ptr(), _ld(c),
                                cp, sp)
        elif a.dtype == torch.int8:
            if c.dtype != torch.int32:
                raise TypeError("int8 GEMM writes int32")
            st = L.gemm_s8_ex(M, N, K, a.data_ptr(), _ld(a), b.data_ptr(), _ld(b), c.data_ptr(), _ld(c),
                              cp, sp)
        else:
            raise TypeError(f"unsupported input dtype {a.dtype}")
    if st:
        raise TclError(st, "gemm")


def gemm(a, b, out_dtype=None, cfg: Config | None = None, stream=None):
    """C = A·B on the GPU. bf16 inputs -> float32 (or ``out_dtype=torch.bfloat16``);
    float32 inputs (consumed as TF32) -> float32; int8 inputs -> int32 (exact)."""
    import torch
    if out_dtype is None:
        out_dtype = {torch.bfloat16: torch.float32, torch.float32: torch.float32,
                     torch.int8: torch.int32}.get(a.dtype)
        if out_dtype is None:
            raise TypeError(f"unsupported input dtype {a.dtype}")
    c = torch.empty((a.shape[0], b.shape[1]), dtype=out_dtype, device=a.device)
    gemm_into(a, b, c, cfg=cfg, stream=stream)
    return c
