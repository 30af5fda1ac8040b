"""CUDA graph capture of the library's calls: solve_ex enqueues only stream-ordered work
(pool allocations and frees, a memset, kernel launches), so a product captured into a graph
and replayed equals, bit for bit, the same product computed directly, for every kernel
class, and replays pick up new operand values written into the same buffers."""

import numpy as np
import pytest

import dense_fp32_gemm_sgemm_gb300 as sg
from tests.gpu_util import inputs, torch_cuda

pytestmark = pytest.mark.gpu

# one shape per dispatch class: 3xTF32 with a pre-pass and split tiles, 3xTF32 with the
# fused split, a recut last round, 1xTF32 on 256 x 256 and on 256 x 512 tiles, FFMA on
# small and on 128 x 128 tiles, GEVM (split reduction), GEMV, short reduction
CASES = [((512, 512, 512), sg.MODE_FP32_3XTF32), ((8192, 1024, 4096), sg.MODE_FP32),
         ((2048, 512, 8192), sg.MODE_FP32), ((1000, 333, 777), sg.MODE_TF32),
         ((8192, 2048, 8192), sg.MODE_TF32),
         ((300, 200, 100), sg.MODE_FP32), ((2048, 512, 2048), sg.MODE_FP32_SIMT),
         ((1, 8192, 8192), sg.MODE_FP32), ((8192, 8192, 1), sg.MODE_FP32),
         ((4097, 1, 4095), sg.MODE_FP32)]


@pytest.mark.parametrize("shape,mode", CASES, ids=[f"{m}x{n}x{k}-mode{md}" for (m, n, k), md in CASES])
def test_graph_replay_matches_direct(shape, mode):
    torch = torch_cuda()
    M, N, K = shape
    A0, B0 = inputs(M, N, K, 50, "uniform")
    A1, B1 = inputs(M, N, K, 51, "uniform")
    dA = torch.from_numpy(A0).cuda()
    dB = torch.from_numpy(B0).cuda()
    dC = torch.empty((M, K), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()

    def call():
        rc = sg.lib().solve_ex(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), M, N, K, mode,
                               int(torch.cuda.current_stream().cuda_stream))
        assert rc == sg.OK, sg.lib().sgemm_status_string(rc)

    with torch.cuda.stream(s):
        call()  # warm-up outside capture: lazy module loads, attributes, the pool
    torch.cuda.synchronize()
    direct0 = dC.cpu().numpy().copy()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    dC.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(dC.cpu().numpy(), direct0), "replay differs from the direct call"

    # new operands in the same buffers: the replay computes the new product
    dA.copy_(torch.from_numpy(A1))
    dB.copy_(torch.from_numpy(B1))
    g.replay()
    torch.cuda.synchronize()
    replay1 = dC.cpu().numpy().copy()
    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    assert np.array_equal(replay1, dC.cpu().numpy())
    assert not np.array_equal(replay1, direct0)
    assert sg.device_error() == sg.OK
