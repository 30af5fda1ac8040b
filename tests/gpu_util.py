"""Helpers shared by the GPU parity tests: run the library through its C ABI on
seeded inputs and compare with the CPU oracle under the stated tolerances."""

import numpy as np
import pytest

import dense_fp32_gemm_sgemm_gb300 as sg
from dense_fp32_gemm_sgemm_gb300.inputs import make_inputs, sample_indices

# Elementwise bounds |C - C_exact| <= TOL * (|A|.|B|): FP32-accurate paths 1e-5, the
# explicit 1xTF32 path 2e-3 (inputs rounded to 11 significant bits: at most 2^-11
# relative error per input, so about 2^-10 per product, plus FP32 accumulation).
TOL = {sg.MODE_FP32: 1e-5, sg.MODE_FP32_SIMT: 1e-5, sg.MODE_FP32_3XTF32: 1e-5,
       sg.MODE_3XFP16_SCALED: 1e-5, sg.MODE_TF32: 2e-3}
MODE_IDS = {sg.MODE_FP32: "fp32", sg.MODE_FP32_SIMT: "simt", sg.MODE_FP32_3XTF32: "3xtf32",
            sg.MODE_3XFP16_SCALED: "3xfp16", sg.MODE_TF32: "tf32"}


def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def to_dev(x, offset=0):
    """Copies a numpy matrix to the GPU. With offset > 0 the tensor starts `offset`
    floats into a larger buffer, so its address is not 16-byte aligned."""
    torch = torch_cuda()
    flat = torch.empty(x.size + offset, dtype=torch.float32, device="cuda")
    view = flat[offset:offset + x.size].view(x.shape)
    view.copy_(torch.from_numpy(np.ascontiguousarray(x)))
    return view


def run_gpu(A, B, mode, offset=0, stream=None):
    """C = A . B through solve_ex; returns C as a numpy float32 array."""
    torch = torch_cuda()
    dA = to_dev(A, offset)
    dB = to_dev(B, offset)
    M, K = A.shape[0], B.shape[1]
    flat = torch.empty(M * K + offset, dtype=torch.float32, device="cuda")
    flat.fill_(float("nan"))
    dC = flat[offset:offset + M * K].view(M, K)
    rc = sg.lib().solve_ex(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), M, A.shape[1], K,
                           mode, int((stream or torch.cuda.current_stream()).cuda_stream))
    assert rc == sg.OK, sg.lib().sgemm_status_string(rc)
    torch.cuda.synchronize()
    return dC.cpu().numpy()


def fp16_scale_term(A, B):
    """The absolute part of the FP16 three-product mode's bound: an element far below the
    largest of its row of A (128-column block of B) keeps a lo piece below FP16's normal
    range, whose spacing is at most 2^-39 of that largest magnitude after the power-of-two
    scale; over a term this adds 2^-39 (max_n |A[m][n]| * sum_n |B[n][k]| +
    sum_n |A[m][n]| * maxB(k)), taken here with a factor 4 of margin."""
    a = np.abs(A.astype(np.float64))
    b = np.abs(B.astype(np.float64))
    K = b.shape[1]
    # B shares one scale per block of 128 columns: the largest |B| of k's block
    bmax = np.concatenate([np.full(min(128, K - k0), b[:, k0:k0 + 128].max())
                           for k0 in range(0, K, 128)])[None, :]
    return 2.0 ** -37 * (a.max(axis=1, keepdims=True) * b.sum(axis=0, keepdims=True) +
                         a.sum(axis=1, keepdims=True) * bmax)


def assert_within(C, C_ref, S, tol, what="", extra=None):
    C = np.asarray(C, dtype=np.float64)
    assert np.all(np.isfinite(C)), f"{what}: non-finite output"
    err = np.abs(C - C_ref)
    bound = tol * S if extra is None else tol * S + extra
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        worst = float(np.max(err / np.maximum(bound, 1e-300)))
        raise AssertionError(f"{what}: {int(bad.sum())} elements outside {tol}*S, "
                             f"worst ratio {worst:.3g}, first at {idx.tolist()}")


def assert_exact(C, C_ref, what=""):
    C = np.asarray(C, dtype=np.float64)
    assert np.all(np.isfinite(C)), f"{what}: non-finite output"
    if not np.array_equal(C, C_ref):
        bad = np.argwhere(C != C_ref)[:5]
        raise AssertionError(f"{what}: {int((C != C_ref).sum())} elements differ, "
                             f"first at {bad.tolist()}")


def check_sampled(C, A, B, tol, seed, count=512, rows_full=8, exact=False, what=""):
    """Compares sampled entries (and `rows_full` whole rows) of a large product with the
    oracle, entry by entry."""
    import oracle
    M, K = C.shape
    r, c = sample_indices(M, K, count, seed)
    c_ref, s_ref = oracle.entries(A, B, r, c)
    got = C[r, c]
    if exact:
        assert_exact(got, c_ref, what + " samples")
    else:
        assert_within(got, c_ref, s_ref, tol, what + " samples")
    if rows_full:
        rows = np.unique(np.concatenate([[0, M - 1], r[:rows_full]]))
        C_rows, S_rows = oracle.gemm(A[rows], B)
        if exact:
            assert_exact(C[rows], C_rows, what + " rows")
        else:
            assert_within(C[rows], C_rows, S_rows, tol, what + " rows")


def split_elements(M, N, K, mode, chunk_rows=None):
    """Boolean mask of the elements of C whose reduction the tensor-core schedule splits
    into parts (added by the last part in a fixed order) for the whole product, or, with
    chunk_rows, for any of the row chunks the pipelined host round trip computes one by
    one. Elsewhere every element is summed in the same order by both paths."""
    mask = np.zeros((M, K), dtype=bool)
    spans = [(0, M)]
    if chunk_rows:
        spans += [(r0, min(chunk_rows, M - r0)) for r0 in range(0, M, chunk_rows)]
    for r0, rows in spans:
        for row, col, cols, _, _, slot in sg.plan_units(rows, N, K, mode):
            if slot >= 0:
                mask[r0 + row:r0 + row + 256, col:col + cols] = True
    return mask


def inputs(M, N, K, seed, dist):
    return make_inputs(M, N, K, seed, dist)
