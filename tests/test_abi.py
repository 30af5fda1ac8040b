"""C-ABI checks that need no GPU: the library loads, exports every function that
include/sgemm.h declares, rejects bad arguments on the host before touching a device,
and plans the expected kernel for each shape class."""

import ctypes

import pytest

import dense_fp32_gemm_sgemm_gb300 as sg
from dense_fp32_gemm_sgemm_gb300 import build as sg_build


@pytest.fixture(scope="module")
def L():
    try:
        sg_build.nvcc()
    except RuntimeError:
        if not sg_build.up_to_date():
            pytest.skip("no nvcc and no prebuilt library")
    sg_build.build()
    return sg.lib()


def test_exports_every_declared_symbol(L):
    names = sg.exported_names()
    assert {"solve", "solve_ex", "solve_host"} <= set(names)
    for name in names:
        assert hasattr(L, name), f"{name} declared in sgemm.h but not exported"


def test_status_strings(L):
    for code in (sg.OK, sg.ERR_ARG, sg.ERR_OVERLAP, sg.ERR_CUDA, sg.ERR_NO_DEVICE,
                 sg.ERR_TIMEOUT, sg.ERR_UNSUPPORTED, 12345):
        s = L.sgemm_status_string(code)
        assert isinstance(s, bytes) and len(s) > 0


# Fake, never dereferenced addresses: validation must reject these before any CUDA call.
A_FAKE, B_FAKE, C_FAKE = 0x10000000, 0x20000000, 0x30000000


@pytest.mark.parametrize("dims", [(0, 4, 4), (4, 0, 4), (4, 4, 0), (8193, 4, 4),
                                  (4, 8193, 4), (4, 4, 8193), (-1, 4, 4)])
def test_bad_dims_rejected(L, dims):
    M, N, K = dims
    assert L.solve_ex(A_FAKE, B_FAKE, C_FAKE, M, N, K, 0, None) == sg.ERR_ARG


def test_null_and_mode_rejected(L):
    assert L.solve_ex(None, B_FAKE, C_FAKE, 4, 4, 4, 0, None) == sg.ERR_ARG
    assert L.solve_ex(A_FAKE, None, C_FAKE, 4, 4, 4, 0, None) == sg.ERR_ARG
    assert L.solve_ex(A_FAKE, B_FAKE, None, 4, 4, 4, 0, None) == sg.ERR_ARG
    assert L.solve_ex(A_FAKE, B_FAKE, C_FAKE, 4, 4, 4, 7, None) == sg.ERR_ARG
    assert L.solve_ex(A_FAKE, B_FAKE, C_FAKE, 4, 4, 4, -1, None) == sg.ERR_ARG


def test_overlap_rejected(L):
    # C = [A + 8 floats, +16 floats) overlaps A = [A, +16 floats)
    assert L.solve_ex(A_FAKE, B_FAKE, A_FAKE + 32, 4, 4, 4, 0, None) == sg.ERR_OVERLAP
    assert L.solve_ex(A_FAKE, B_FAKE, B_FAKE - 32, 4, 4, 4, 0, None) == sg.ERR_OVERLAP


def test_solve_void_sets_last_status(L):
    L.solve(A_FAKE, B_FAKE, C_FAKE, 0, 1, 1)
    assert L.sgemm_last_status() == sg.ERR_ARG


def test_solve_host_validation(L):
    assert L.solve_host(None, None, None, 1, 1, 1, 0, None) == sg.ERR_ARG
    assert L.solve_host(A_FAKE, B_FAKE, C_FAKE, 9000, 1, 1, 0, None) == sg.ERR_ARG


def test_plan_shape_classes(L):
    assert sg.plan(1, 8192, 8192)[0] == sg.KERNEL_GEVM
    assert sg.plan(8192, 8192, 1)[0] == sg.KERNEL_GEMV
    assert sg.plan(1, 1, 1)[0] == sg.KERNEL_GEMV
    assert sg.plan(8192, 6144, 4096)[0] == sg.KERNEL_TC_3XTF32
    # small products: the CUDA-core kernel on 16 x 64 tiles (32 x 64 without 16-byte rows)
    assert sg.plan(512, 512, 512) == (sg.KERNEL_SIMT, 32 * 8)
    assert sg.plan(510, 512, 512) == (sg.KERNEL_SIMT, 32 * 8)
    assert sg.plan(512, 512, 512, aligned=False) == (sg.KERNEL_SIMT, 16 * 8)
    assert sg.plan(17, 19, 31)[0] == sg.KERNEL_SIMT
    assert sg.plan(64, 64, 127)[0] == sg.KERNEL_SIMT
    assert sg.plan(64, 128, 128)[0] == sg.KERNEL_SIMT
    assert sg.plan(640, 640, 640) == (sg.KERNEL_TC_3XTF32, 9)
    assert sg.plan(128, 8192, 128)[0] == sg.KERNEL_TC_3XTF32  # long reduction, 8 tiles
    assert sg.plan(8192, 6144, 4096, mode=sg.MODE_TF32)[0] == sg.KERNEL_TC_1XTF32
    assert sg.plan(1, 8192, 8192, mode=sg.MODE_TF32)[0] == sg.KERNEL_GEVM
    assert sg.plan(1, 8192, 8192, mode=sg.MODE_FP32_3XTF32)[0] == sg.KERNEL_TC_3XTF32
    assert sg.plan(512, 512, 512, mode=sg.MODE_FP32_SIMT) == (sg.KERNEL_SIMT, 32 * 8)
    assert sg.plan(8191, 6143, 4097, mode=sg.MODE_FP32_SIMT) == (sg.KERNEL_SIMT, 64 * 33)
    assert sg.plan(4097, 1, 4095) == (sg.KERNEL_SMALLN, 32 * 65)
    assert sg.plan(1000, 4, 777, mode=sg.MODE_TF32)[0] == sg.KERNEL_SMALLN
    assert sg.plan(8192, 5, 8192)[0] == sg.KERNEL_TC_3XTF32
    assert sg.plan(4097, 1, 4095, mode=sg.MODE_FP32_3XTF32)[0] == sg.KERNEL_TC_3XTF32
    # the FP16 three-product mode is forced for every shape, with the 256 x 256 tiles
    assert sg.plan(8192, 6144, 4096, mode=sg.MODE_3XFP16_SCALED) == (sg.KERNEL_TC_3XFP16, 32 * 16)
    assert sg.plan(1, 8192, 8192, mode=sg.MODE_3XFP16_SCALED)[0] == sg.KERNEL_TC_3XFP16
    assert sg.plan(17, 19, 31, mode="3xfp16")[0] == sg.KERNEL_TC_3XFP16
    assert sg.plan(0, 1, 1)[0] == sg.ERR_ARG
    tiles = ctypes.c_int(-7)
    assert L.sgemm_plan(4, 4, 4, 9, 1, ctypes.byref(tiles)) == sg.ERR_ARG
    assert tiles.value == -7


def test_launch_count_starts_readable(L):
    assert sg.launch_count() >= 0


def test_selftest_limits_checked_on_host(L):
    assert L.sgemm_selftest_wait_timeout(10, None) == sg.ERR_ARG
    assert L.sgemm_selftest_wait_timeout(3_000_000_000, None) == sg.ERR_ARG


def test_peak_probe_arguments_checked_on_host(L):
    flop, ms = ctypes.c_double(-1.0), ctypes.c_float(-1.0)
    assert L.sgemm_peak_probe(7, 16, None, ctypes.byref(flop), ctypes.byref(ms)) == sg.ERR_ARG
    assert L.sgemm_peak_probe(sg.PROBE_FFMA, 0, None, ctypes.byref(flop),
                              ctypes.byref(ms)) == sg.ERR_ARG
    assert L.sgemm_peak_probe(sg.PROBE_FFMA2, (1 << 20) + 1, None, ctypes.byref(flop),
                              ctypes.byref(ms)) == sg.ERR_ARG
    assert L.sgemm_peak_probe(sg.PROBE_TF32_MMA, (1 << 18) + 1, None, ctypes.byref(flop),
                              ctypes.byref(ms)) == sg.ERR_ARG
    assert L.sgemm_peak_probe(sg.PROBE_TF32_MMA, 16, None, None, ctypes.byref(ms)) == sg.ERR_ARG
    assert flop.value == -1.0 and ms.value == -1.0


def test_clock_readings_check_their_argument_on_host(L):
    assert L.sgemm_tc_clock_mhz(None, None) == sg.ERR_ARG
    assert L.sgemm_simt_clock_mhz(None, None) == sg.ERR_ARG
