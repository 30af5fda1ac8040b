"""Host checks of the two split-precision schemes' representation error, emulated in
numpy and summed in fp64 (no GPU, and nothing from the CUDA path): the claims the design
makes about them before any tensor-core accumulation error.

3xTF32: hi = x truncated to TF32 (13 low mantissa bits cleared), lo = x - hi rounded to TF32
with ties away from zero; the product is A_lo.B_hi + A_hi.B_lo + A_hi.B_hi.
3xFP16: each row of A and each block of 128 columns of B scaled by the power of two that
puts its largest magnitude in [2^14, 2^15), hi = rn_fp16(x), lo = rn_fp16(x - hi), the same three products,
then the scales undone.
"""

import numpy as np
import pytest

from dense_fp32_gemm_sgemm_gb300.inputs import make_inputs


def tf32_trunc(x):
    return (x.astype(np.float32).view(np.uint32) & np.uint32(0xFFFFE000)).view(np.float32)


def tf32_rna(x):
    u = x.astype(np.float32).view(np.uint32)
    sign = u & np.uint32(0x80000000)
    mag = (u & np.uint32(0x7FFFFFFF)) + np.uint32(0x1000)  # half an ulp of TF32: ties away
    return ((mag & np.uint32(0x7FFFE000)) | sign).view(np.float32)


def split_tf32(X):
    hi = tf32_trunc(X)
    lo = tf32_rna(X.astype(np.float32) - hi)  # x - hi is exact in FP32
    return hi.astype(np.float64), lo.astype(np.float64)


def split_fp16(X, axis):
    """Scaled FP16 pieces: one scale per row (axis=1) or per block of 128 columns (axis=0)."""
    if axis == 1:
        m = np.max(np.abs(X), axis=1, keepdims=True).astype(np.float64)
    else:
        m = np.concatenate([np.full(min(128, X.shape[1] - k0), np.abs(X[:, k0:k0 + 128]).max())
                            for k0 in range(0, X.shape[1], 128)])[None, :].astype(np.float64)
    e = np.where(m > 0, 14 - np.floor(np.log2(np.where(m > 0, m, 1.0))), 0.0)
    Xs = (X.astype(np.float64) * np.exp2(e)).astype(np.float32)  # exact: a power of two
    hi = Xs.astype(np.float16)
    lo = (Xs - hi.astype(np.float32)).astype(np.float16)
    return hi.astype(np.float64), lo.astype(np.float64), e


def three_tf32(A, B):
    ah, al = split_tf32(A)
    bh, bl = split_tf32(B)
    return al @ bh + ah @ bl + ah @ bh


def three_fp16(A, B):
    ah, al, ea = split_fp16(A, 1)
    bh, bl, eb = split_fp16(B, 0)
    return (al @ bh + ah @ bl + ah @ bh) * np.exp2(-ea) * np.exp2(-eb)


def reference(A, B):
    a, b = A.astype(np.float64), B.astype(np.float64)
    return a @ b, np.abs(a) @ np.abs(b)


CASES = [(128, 3072, 96, 2, "uniform"), (96, 4096, 64, 3, "normal"), (128, 64, 128, 3, "normal"),
         (100, 1000, 77, 4, "uniform"), (64, 2048, 64, 5, "int8")]


@pytest.mark.parametrize("M,N,K,seed,dist", CASES)
def test_split_error_far_below_the_bound(M, N, K, seed, dist):
    """On the workloads' distributions each scheme stays within its per-product bound, far
    below the 1e-5 of (|A|.|B|) allowed: 3xTF32 2^-19 (hi truncated, so lo carries up to
    2^-10 of x and the dropped lo.lo term up to 2^-20 of |a||b|), 3xFP16 2^-22 (pieces
    rounded to nearest, 2^-12 each); integers are exact in both."""
    A, B = make_inputs(M, N, K, seed, dist)
    C, S = reference(A, B)
    for name, got, bound in (("3xtf32", three_tf32(A, B), 2.0 ** -19),
                             ("3xfp16", three_fp16(A, B), 2.0 ** -22)):
        if dist == "int8":
            assert np.array_equal(got, C), name
        else:
            assert np.max(np.abs(got - C) / S) <= bound, name


def test_tf32_split_keeps_21_bits_per_element():
    """hi + lo reproduces any normal float to within 2^-21 of its magnitude (truncation
    leaves at most 2^-10 relative to lo, which then keeps 11 bits)."""
    x = make_inputs(1, 50000, 1, 6, "normal")[0].ravel()
    hi, lo = split_tf32(x)
    rel = np.abs(hi + lo - x.astype(np.float64)) / np.abs(x.astype(np.float64))
    assert rel.max() <= 2.0 ** -21


def test_fp16_split_needs_its_absolute_term_for_tiny_elements():
    """An element far below its row's largest magnitude loses bits in the FP16 scheme, so
    A.I can miss the relative bound; the stated absolute term
    2^-37 (max_n|A_mn| sum_n|B_nk| + sum_n|A_mn| max_n|B_nk|) covers it, and 3xTF32 needs
    no such term."""
    n = 64
    A = np.full((1, n), 0.75, dtype=np.float32)
    A[0, 5] = np.float32(3.0e-8)  # about 2^-25 of the row's largest
    eye = np.eye(n, dtype=np.float32)
    C, S = reference(A, eye)
    err16 = np.abs(three_fp16(A, eye) - C)
    assert err16[0, 5] > 1e-5 * S[0, 5], "the relative bound alone is missed"
    a, b = np.abs(A.astype(np.float64)), np.abs(eye.astype(np.float64))
    extra = 2.0 ** -37 * (a.max(axis=1, keepdims=True) * b.sum(axis=0, keepdims=True) +
                          a.sum(axis=1, keepdims=True) * b.max())  # one 128-column block
    assert np.all(err16 <= 1e-5 * S + extra)
    assert np.all(np.abs(three_tf32(A, eye) - C) <= 1e-5 * S)
