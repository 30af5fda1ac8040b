"""Python binding of the GB300 SGEMM library (``_build/libsgemm.so``).

Argument marshalling only: every step of the product runs in the library's CUDA
kernels. PyTorch is used for device memory and streams. If the compiled library is
missing, every call raises; there is no CPU fallback.

    import torch, dense_fp32_gemm_sgemm_gb300 as sg
    A = torch.randn(512, 256, device="cuda"); B = torch.randn(256, 384, device="cuda")
    C = sg.matmul(A, B)                      # FP32-accurate
    C = sg.matmul(A, B, mode=sg.MODE_TF32)   # explicit 1xTF32
    C = sg.matmul(A, B, mode="3xfp16")       # scaled FP16 pieces (bound in the C header)
"""

from __future__ import annotations

import ctypes
import os
import re
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB_PATH = os.path.join(PKG, "_build", "libsgemm.so")
HEADER = os.path.join(ROOT, "include", "sgemm.h")

OK = 0
ERR_ARG = -1
ERR_OVERLAP = -2
ERR_CUDA = -3
ERR_NO_DEVICE = -4
ERR_TIMEOUT = -5
ERR_UNSUPPORTED = -6

MODE_FP32 = 0
MODE_TF32 = 1
MODE_FP32_SIMT = 2
MODE_FP32_3XTF32 = 3
MODE_3XFP16_SCALED = 4
MODES = {"fp32": MODE_FP32, "tf32": MODE_TF32, "simt": MODE_FP32_SIMT,
         "3xtf32": MODE_FP32_3XTF32, "3xfp16": MODE_3XFP16_SCALED}

KERNEL_SIMT = 1
KERNEL_GEVM = 2
KERNEL_GEMV = 3
KERNEL_TC_1XTF32 = 4
KERNEL_TC_3XTF32 = 5
KERNEL_SMALLN = 6
KERNEL_TC_3XFP16 = 7

PROBE_FFMA = 0
PROBE_FFMA2 = 1
PROBE_TF32_MMA = 2
PROBE_F16_MMA = 3

_lock = threading.Lock()
_lib = None


class SgemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        text = lib().sgemm_status_string(status).decode()
        super().__init__(f"{what + ': ' if what else ''}{text} (status {status})")


def exported_names() -> list[str]:
    """Function names declared in include/sgemm.h (the C ABI)."""
    src = open(HEADER, encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", src, flags=re.M)


def lib() -> ctypes.CDLL:
    """Loads the compiled library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it first (python -m "
                    "dense_fp32_gemm_sgemm_gb300.build, or __graft_entry__.build())")
            L = ctypes.CDLL(LIB_PATH)
            vp, i = ctypes.c_void_p, ctypes.c_int
            L.solve.argtypes = [vp, vp, vp, i, i, i]
            L.solve.restype = None
            L.solve_ex.argtypes = [vp, vp, vp, i, i, i, i, vp]
            L.solve_ex.restype = i
            L.solve_host.argtypes = [vp, vp, vp, i, i, i, i, vp]
            L.solve_host.restype = i
            L.sgemm_set_stream.argtypes = [vp]
            L.sgemm_set_stream.restype = i
            L.sgemm_last_status.argtypes = []
            L.sgemm_last_status.restype = i
            L.sgemm_status_string.argtypes = [i]
            L.sgemm_status_string.restype = ctypes.c_char_p
            L.sgemm_device_error.argtypes = [vp]
            L.sgemm_device_error.restype = i
            L.sgemm_plan.argtypes = [i, i, i, i, i, ctypes.POINTER(i)]
            L.sgemm_plan.restype = i
            L.sgemm_plan_units.argtypes = [i, i, i, i, i, ctypes.POINTER(i), i]
            L.sgemm_plan_units.restype = i
            L.sgemm_launch_count.argtypes = []
            L.sgemm_launch_count.restype = ctypes.c_longlong
            L.sgemm_set_kernel_events.argtypes = [vp, vp]
            L.sgemm_set_kernel_events.restype = i
            L.sgemm_release_pool.argtypes = []
            L.sgemm_release_pool.restype = i
            L.sgemm_selftest_wait_timeout.argtypes = [ctypes.c_longlong, vp]
            L.sgemm_selftest_wait_timeout.restype = i
            L.solve_row_noalloc.argtypes = [vp, vp, vp, i, i, vp]
            L.solve_row_noalloc.restype = i
            L.sgemm_peak_probe.argtypes = [i, i, vp, ctypes.POINTER(ctypes.c_double),
                                           ctypes.POINTER(ctypes.c_float)]
            L.sgemm_peak_probe.restype = i
            L.sgemm_tc_clock_mhz.argtypes = [vp, ctypes.POINTER(ctypes.c_double)]
            L.sgemm_tc_clock_mhz.restype = i
            L.sgemm_simt_clock_mhz.argtypes = [vp, ctypes.POINTER(ctypes.c_double)]
            L.sgemm_simt_clock_mhz.restype = i
            _lib = L
    return _lib


def _mode(mode) -> int:
    if isinstance(mode, str):
        return MODES[mode.lower()]
    return int(mode)


def _stream_handle(stream=None) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _check_operands(A, B, C):
    import torch
    for name, t in (("A", A), ("B", B), ("C", C)):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if t.dtype != torch.float32 or not t.is_cuda or t.dim() != 2 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 2-D float32 CUDA tensor")
    M, N = A.shape
    if B.shape[0] != N or C.shape != (M, B.shape[1]):
        raise ValueError(f"shapes do not chain: A {tuple(A.shape)}, B {tuple(B.shape)}, "
                         f"C {tuple(C.shape)}")
    return M, N, B.shape[1]


def solve(A, B, C, mode=MODE_FP32, stream=None) -> None:
    """C = A . B for float32 CUDA tensors (A: M x N, B: N x K, C: M x K), enqueued on
    ``stream`` (default: torch's current stream). Raises SgemmError on a bad status."""
    M, N, K = _check_operands(A, B, C)
    rc = lib().solve_ex(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, _mode(mode),
                        _stream_handle(stream))
    if rc != OK:
        raise SgemmError(rc, "solve_ex")


def matmul(A, B, mode=MODE_FP32, stream=None):
    """Returns a new M x K tensor holding A . B."""
    import torch
    C = torch.empty((A.shape[0], B.shape[1]), dtype=torch.float32, device=A.device)
    solve(A, B, C, mode=mode, stream=stream)
    return C


def solve_host(A, B, mode=MODE_FP32, C=None, stream=None):
    """Round trip through the library for host numpy arrays: upload A and B, multiply,
    download C. Returns C (float32 numpy array)."""
    import numpy as np
    A = np.ascontiguousarray(A, dtype=np.float32)
    B = np.ascontiguousarray(B, dtype=np.float32)
    M, N = A.shape
    K = B.shape[1]
    if B.shape[0] != N:
        raise ValueError("inner dimensions differ")
    if C is None:
        C = np.empty((M, K), dtype=np.float32)
    rc = lib().solve_host(A.ctypes.data, B.ctypes.data, C.ctypes.data, M, N, K, _mode(mode),
                          _stream_handle(stream))
    if rc != OK:
        raise SgemmError(rc, "solve_host")
    return C


def plan(M: int, N: int, K: int, mode=MODE_FP32, aligned: bool = True):
    """(kernel id, tile count) that solve would use; host-only, needs no GPU."""
    tiles = ctypes.c_int(0)
    k = lib().sgemm_plan(M, N, K, _mode(mode), int(aligned), ctypes.byref(tiles))
    return k, tiles.value


def plan_units(M: int, N: int, K: int, mode=MODE_FP32, sm_count: int = 0):
    """The tensor-core GEMM's units for this shape and mode, in the order CTA pairs take
    them round-robin: a list of (row0, col0, cols, kb0, kb1, slot). Host-only."""
    n = lib().sgemm_plan_units(M, N, K, _mode(mode), int(sm_count), None, 0)
    if n < 0:
        raise SgemmError(n, "sgemm_plan_units")
    buf = (ctypes.c_int * (6 * n))()
    lib().sgemm_plan_units(M, N, K, _mode(mode), int(sm_count), buf, n)
    return [tuple(buf[6 * u:6 * u + 6]) for u in range(n)]


def launch_count() -> int:
    return int(lib().sgemm_launch_count())


def device_error(stream=None) -> int:
    return int(lib().sgemm_device_error(_stream_handle(stream)))


def tc_clock_mhz(stream=None) -> float:
    """SM clock (MHz) of the last tensor-core GEMM or TF32 probe launch, measured by the
    kernel itself (clock64 cycles over globaltimer nanoseconds on CTA 0)."""
    mhz = ctypes.c_double(0.0)
    rc = lib().sgemm_tc_clock_mhz(_stream_handle(stream), ctypes.byref(mhz))
    if rc != OK:
        raise SgemmError(rc, "sgemm_tc_clock_mhz")
    return mhz.value


def simt_clock_mhz(stream=None) -> float:
    """SM clock (MHz) of the last CUDA-core GEMM or FFMA probe launch, measured by the
    kernel itself (thread 0 of CTA 0, from its start to its end)."""
    mhz = ctypes.c_double(0.0)
    rc = lib().sgemm_simt_clock_mhz(_stream_handle(stream), ctypes.byref(mhz))
    if rc != OK:
        raise SgemmError(rc, "sgemm_simt_clock_mhz")
    return mhz.value


def peak_probe(probe: int, iters: int, stream=None):
    """Runs one rate probe (PROBE_*) on the current device; returns (flop, ms)."""
    flop = ctypes.c_double(0.0)
    ms = ctypes.c_float(0.0)
    rc = lib().sgemm_peak_probe(int(probe), int(iters), _stream_handle(stream),
                                ctypes.byref(flop), ctypes.byref(ms))
    if rc != OK:
        raise SgemmError(rc, "sgemm_peak_probe")
    return flop.value, float(ms.value)
