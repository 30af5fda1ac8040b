"""The allocation-free one-row entry point, solve_row_noalloc.

It serves callers that cannot allocate device memory: an application whose own
allocator has reserved nearly all of it, one that must account every device byte, or a
loop that cannot take an allocation's possible synchronisation. Its partial sums live in
a fixed device array shared by all calls. This checks, through the C ABI, two calls in a
row (the second over whatever the first left in that array) against the CPU oracle,
within the FP32 bound used by every other test (|C - C_exact| <= 1e-5 * (|A|.|B|)), and
against what solve_ex returns for the same products; and that the two calls leave the
device's free memory exactly as it was.

Collected last on purpose: a failure here must not stop a first-failure run before the
other tests have run.
"""

import numpy as np
import pytest

import dense_fp32_gemm_sgemm_gb300 as sg
from tests.gpu_util import assert_within, inputs, to_dev, torch_cuda

pytestmark = pytest.mark.gpu

# the first call fills the shared array with 8192-wide partial rows; the second, narrower
# and with K not a multiple of 4 (the 4-byte loader), runs over what the first left behind
CASES = [(8192, 8192, 3), (3000, 257, 4)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_fp32_gemm_sgemm_gb300 import build
    build.build()
    torch_cuda()


def test_two_calls_match_the_oracle_and_allocate_nothing():
    import oracle
    torch = torch_cuda()
    L = sg.lib()
    stream = int(torch.cuda.current_stream().cuda_stream)
    cases = []
    for N, K, seed in CASES:
        A, B = inputs(1, N, K, seed, "normal")
        C_ref, S = oracle.gemm(A, B)
        dA, dB = to_dev(A), to_dev(B)
        got = torch.full((1, K), float("nan"), device="cuda")
        ex = torch.empty(1, K, device="cuda")
        cases.append((N, K, dA, dB, got, ex, C_ref, S))
    # every buffer exists before the measured window; a warm-up call per case loads the
    # device code (both loaders and the reduction) and looks up the array; solve_ex's
    # results are taken now, and its pool is trimmed, so nothing else changes the free
    # memory while the two calls run
    for N, K, dA, dB, got, ex, _, _ in cases:
        assert L.solve_row_noalloc(dA.data_ptr(), dB.data_ptr(), got.data_ptr(), N, K,
                                   stream) == sg.OK
        assert L.solve_ex(dA.data_ptr(), dB.data_ptr(), ex.data_ptr(), 1, N, K, sg.MODE_FP32,
                          stream) == sg.OK
    torch.cuda.synchronize()
    assert L.sgemm_release_pool() == sg.OK
    for _, _, _, _, got, _, _, _ in cases:
        got.fill_(float("nan"))
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for N, K, dA, dB, got, _, _, _ in cases:
        assert L.solve_row_noalloc(dA.data_ptr(), dB.data_ptr(), got.data_ptr(), N, K,
                                   stream) == sg.OK
    torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    assert free_after == free_before, f"device free memory changed by {free_before - free_after} B"
    for N, K, _, _, got, ex, C_ref, S in cases:
        g = got.cpu().numpy()
        assert_within(g, C_ref, S, 1e-5, f"noalloc {N}x{K} against the oracle")
        # and the pool-backed entry point on the same product, within the same bound
        assert_within(g, ex.cpu().numpy().astype(np.float64), S, 1e-5, f"noalloc {N}x{K} vs solve_ex")
    assert sg.device_error() == sg.OK


def test_rejects_sizes_beyond_the_array():
    L = sg.lib()
    assert L.solve_row_noalloc(0x1000, 0x2000, 0x3000, 8193, 16, None) == sg.ERR_ARG
    assert L.solve_row_noalloc(0x1000, 0x2000, 0x3000, 16, 8193, None) == sg.ERR_ARG
    assert L.solve_row_noalloc(0x1000, 0x2000, 0x3000, 0, 16, None) == sg.ERR_ARG
