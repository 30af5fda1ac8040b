"""Seeded random shapes through every mode: each product is checked against the oracle,
bit for bit on integer entries and within the mode's bound on uniform ones. The shapes
are drawn log-uniformly, so that one-row, one-column, short-reduction, few-tile (split),
unaligned and multi-round shapes all occur, with the kernels and schedules each implies."""

import numpy as np
import pytest

import dense_fp32_gemm_sgemm_gb300 as sg
from tests.gpu_util import TOL, assert_exact, assert_within, check_sampled, inputs, run_gpu

pytestmark = pytest.mark.gpu

MODES = [sg.MODE_FP32, sg.MODE_TF32, sg.MODE_FP32_SIMT, sg.MODE_FP32_3XTF32]


def shapes(count, seed, max_dim=1500, max_work=2.0e9):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < count:
        M, N, K = (int(round(np.exp(rng.uniform(0.0, np.log(max_dim))))) for _ in range(3))
        if M * N * K <= max_work:
            out.append((M, N, K))
    return out


CASES = [(s, m) for i, s in enumerate(shapes(24, 7)) for m in [MODES[i % 4]]]
# the FP16 three-product mode on shapes of its own
CASES += [(s, sg.MODE_3XFP16_SCALED) for s in shapes(10, 17)]


@pytest.mark.parametrize("shape,mode", CASES, ids=[f"{m}x{n}x{k}-mode{md}" for (m, n, k), md in CASES])
def test_random_shape(shape, mode):
    import oracle
    M, N, K = shape
    Ai, Bi = inputs(M, N, K, 77, "int8")
    Ci, _ = oracle.gemm(Ai, Bi)
    assert_exact(run_gpu(Ai, Bi, mode), Ci, f"{shape} int8")
    A, B = inputs(M, N, K, 78, "uniform")
    C_ref, S = oracle.gemm(A, B)
    assert_within(run_gpu(A, B, mode, offset=(M + N + K) % 3), C_ref, S, TOL[mode], f"{shape} uniform")
    assert sg.device_error() == sg.OK


def large_shapes(count, seed):
    """Large seeded shapes (2048..8192 rows, 512..6144 reduction, 1024..8192 columns): the
    fused split (every other shape has a reduction length divisible by 4, which the fused
    path needs), split reductions and ragged tails, at random."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(count):
        M, N, K = (int(rng.integers(2048, 8193)), int(rng.integers(512, 6145)),
                   int(rng.integers(1024, 8193)))
        out.append((M, N - N % 4 if i % 2 == 0 else N, K))
    return out


LARGE_CASES = [(s, m) for i, s in enumerate(large_shapes(6, 9))
               for m in [(sg.MODE_FP32, sg.MODE_TF32)[i % 2]]]
LARGE_CASES += [(s, sg.MODE_3XFP16_SCALED) for s in large_shapes(3, 19)]


@pytest.mark.parametrize("shape,mode", LARGE_CASES,
                         ids=[f"{m}x{n}x{k}-mode{md}" for (m, n, k), md in LARGE_CASES])
def test_random_large_shape(shape, mode):
    M, N, K = shape
    A, B = inputs(M, N, K, 80, "uniform")
    check_sampled(run_gpu(A, B, mode), A, B, TOL[mode], seed=81, count=2048, rows_full=4,
                  what=f"{shape} uniform")
    Ai, Bi = inputs(M, N, K, 82, "int8")
    check_sampled(run_gpu(Ai, Bi, mode), Ai, Bi, 0.0, seed=83, count=1024, rows_full=2,
                  exact=True, what=f"{shape} int8")
    assert sg.device_error() == sg.OK
