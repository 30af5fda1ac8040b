"""Failure detection on the GPU without faulting it: every wait inside the kernels is
bounded, and a wait that runs out sets the device error word and lets the kernel
return. sgemm_selftest_wait_timeout runs that exact wait on an mbarrier that nothing
completes; the status must come back as a timeout, and the context must stay usable."""

import numpy as np
import pytest

import dense_fp32_gemm_sgemm_gb300 as sg
from tests.gpu_util import assert_within, inputs, run_gpu, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_fp32_gemm_sgemm_gb300 import build
    build.build()
    torch_cuda()


def test_bounded_wait_times_out_and_context_survives():
    import oracle
    torch = torch_cuda()
    stream = int(torch.cuda.current_stream().cuda_stream)
    assert sg.lib().sgemm_selftest_wait_timeout(50_000_000, stream) == sg.ERR_TIMEOUT
    # the word was cleared by the read, and the context still runs products
    assert sg.device_error() == sg.OK
    A, B = inputs(300, 200, 260, 15, "uniform")
    C_ref, S = oracle.gemm(A, B)
    for mode in (sg.MODE_FP32, sg.MODE_FP32_3XTF32, sg.MODE_TF32):
        tol = 2e-3 if mode == sg.MODE_TF32 else 1e-5
        assert_within(run_gpu(A, B, mode), C_ref, S, tol, f"after timeout, mode {mode}")
    assert sg.device_error() == sg.OK
