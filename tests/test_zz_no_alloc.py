"""The allocation-free one-row entry point, solve_row_noalloc.

It serves callers that cannot allocate device memory (their own allocator holds the
memory, or allocation latency is not allowed), so its partial sums live in a fixed
device array shared by all calls. This checks, through the C ABI, that two calls in a
row - the second over whatever the first left in that array - match what solve_ex
returns for the same one-row products, within the FP32 bound used by every other
test (|difference| <= 1e-5 * (|A|.|B|)).

Collected last on purpose: a failure here must not stop a first-failure run before the
other tests have run.
"""

import numpy as np
import pytest

import dense_fp32_gemm_sgemm_gb300 as sg
from tests.gpu_util import assert_within, inputs, to_dev, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_fp32_gemm_sgemm_gb300 import build
    build.build()
    torch_cuda()


def _row_products(N, K, seed):
    import oracle
    torch = torch_cuda()
    A, B = inputs(1, N, K, seed, "normal")
    _, S = oracle.gemm(A, B)
    dA, dB = to_dev(A), to_dev(B)
    stream = int(torch.cuda.current_stream().cuda_stream)
    L = sg.lib()
    ref = torch.empty(1, K, device="cuda")
    got = torch.full((1, K), float("nan"), device="cuda")
    assert L.solve_ex(dA.data_ptr(), dB.data_ptr(), ref.data_ptr(), 1, N, K,
                      sg.MODE_FP32, stream) == sg.OK
    assert L.solve_row_noalloc(dA.data_ptr(), dB.data_ptr(), got.data_ptr(), N, K,
                               stream) == sg.OK
    torch.cuda.synchronize()
    return got.cpu().numpy(), ref.cpu().numpy(), S


def test_two_calls_match_solve_ex():
    # first call fills the shared array with 8192-wide partial rows; the second, narrower
    # and unaligned, runs over what the first left behind
    for N, K, seed in [(8192, 8192, 3), (3000, 257, 4)]:
        got, ref, S = _row_products(N, K, seed)
        assert_within(got, ref.astype(np.float64), S, 1e-5, f"noalloc {N}x{K}")


def test_rejects_sizes_beyond_the_array():
    L = sg.lib()
    assert L.solve_row_noalloc(0x1000, 0x2000, 0x3000, 8193, 16, None) == sg.ERR_ARG
    assert L.solve_row_noalloc(0x1000, 0x2000, 0x3000, 16, 8193, None) == sg.ERR_ARG
    assert L.solve_row_noalloc(0x1000, 0x2000, 0x3000, 0, 16, None) == sg.ERR_ARG
