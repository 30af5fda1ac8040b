"""Pins for the CPU oracle: each check ties it to something other than itself.

* the worked examples printed on the pages (tests/golden/worked_examples.txt);
* exact rational sums (fractions.Fraction) on tiny shapes, within the double-rounding
  bound of a recursive sum;
* integer-valued inputs against numpy's exact int64 matrix product;
* identity, permutation and transpose invariants, which hold bit for bit;
* closed forms (all-ones, and A = 1 with B[n][k] = n);
* the integer/8 input pattern of "分块计算与矩阵乘法", section "3. 完整对照程序",
  on that page's shapes, against exact integer arithmetic;
* properties of the scale S = |A|.|B| used by every tolerance.

The last test plants plausible mistakes in copies of the oracle (transposed operand,
dropped term, wrong sign, float32 accumulation, transposed output) and checks that
every one of them fails at least one pin.
"""

from fractions import Fraction

import numpy as np
import pytest

from dense_fp32_gemm_sgemm_gb300.inputs import make_inputs, make_permutation
from tests.golden.load import worked_examples

U53 = 2.0 ** -53


# ---------------------------------------------------------------------------------
# Pins written as checks on any gemm function f(A, B) -> C (float64), so that the
# same checks can be run against planted mistakes below.
# ---------------------------------------------------------------------------------

def pin_worked_examples(f):
    for case in worked_examples():
        C = f(case["A"], case["B"])
        assert C.shape == case["C"].shape, case["name"]
        assert np.array_equal(C, case["C"].astype(np.float64)), case["name"]


def _exact(A, B):
    M, N = A.shape
    K = B.shape[1]
    Af = [[Fraction(float(x)) for x in row] for row in A]
    Bf = [[Fraction(float(x)) for x in row] for row in B]
    C = [[sum((Af[m][n] * Bf[n][k] for n in range(N)), Fraction(0)) for k in range(K)]
         for m in range(M)]
    S = [[sum((abs(Af[m][n]) * abs(Bf[n][k]) for n in range(N)), Fraction(0))
          for k in range(K)] for m in range(M)]
    return C, S


def pin_exact_rational(f):
    for (M, N, K), seed in [((1, 1, 1), 1), ((2, 2, 2), 1), ((1, 3, 1), 1),
                            ((17, 19, 31), 1), ((5, 40, 3), 7)]:
        A, B = make_inputs(M, N, K, seed, "uniform")
        C = f(A, B)
        assert C.shape == (M, K)
        Ce, Se = _exact(A, B)
        # recursive summation in double: |err| <= (N-1) u / (1 - (N-1) u) * sum |terms|
        g = (N - 1) * U53 / (1 - (N - 1) * U53)
        for m in range(M):
            for k in range(K):
                err = abs(Fraction(float(C[m, k])) - Ce[m][k])
                assert err <= Fraction(g) * Se[m][k] + Fraction(0), (M, N, K, m, k)


def pin_integer_exact(f):
    for (M, N, K), dist in [((17, 19, 31), "int8"), ((127, 129, 65), "int8"),
                            ((64, 300, 50), "int4"), ((3, 1, 7), "int8")]:
        A, B = make_inputs(M, N, K, 1, dist)
        ref = A.astype(np.int64) @ B.astype(np.int64)
        C = f(A, B)
        assert C.shape == ref.shape
        assert np.array_equal(C, ref.astype(np.float64)), (M, N, K)


def pin_identity(f):
    A, _ = make_inputs(33, 33, 1, 3, "normal")
    eye = np.eye(33, dtype=np.float32)
    assert np.array_equal(f(A, eye), A.astype(np.float64))
    _, B = make_inputs(1, 21, 45, 4, "uniform")
    eye = np.eye(21, dtype=np.float32)
    assert np.array_equal(f(eye, B), B.astype(np.float64))


def pin_permutation(f):
    # (P.B)[i] = B[p[i]] where P[i, p[i]] = 1; (A.P)[:, p[i]] = A[:, i]
    A, B = make_inputs(13, 29, 11, 5, "uniform")
    p = make_permutation(29, 5)
    P = np.zeros((29, 29), dtype=np.float32)
    P[np.arange(29), p] = 1.0
    assert np.array_equal(f(P, B), B[p].astype(np.float64))
    AP = f(A, P)
    expect = np.empty_like(A)
    expect[:, p] = A
    assert np.array_equal(AP, expect.astype(np.float64))


def pin_transpose(f):
    A, B = make_inputs(9, 23, 14, 6, "uniform")
    assert np.array_equal(f(np.ascontiguousarray(B.T), np.ascontiguousarray(A.T)),
                          f(A, B).T)


def pin_closed_forms(f):
    for N in (1, 7, 1000):
        ones_a = np.ones((3, N), dtype=np.float32)
        ones_b = np.ones((N, 5), dtype=np.float32)
        assert np.array_equal(f(ones_a, ones_b), np.full((3, 5), float(N)))
        ramp = np.repeat(np.arange(N, dtype=np.float32)[:, None], 5, axis=1)
        assert np.array_equal(f(ones_a, ramp), np.full((3, 5), N * (N - 1) / 2.0))


def _dyadic(M, N, K):
    a = ((np.arange(M * N, dtype=np.int64) * 17) % 13 - 6).reshape(M, N)
    b = ((np.arange(N * K, dtype=np.int64) * 29) % 11 - 5).reshape(N, K)
    return a, b


def pin_dyadic_pattern(f):
    # Shapes of that page's run_case list and exercise, relabelled to (M, N, K).
    for M, N, K in [(3, 5, 4), (17, 19, 23), (257, 129, 193), (255, 257, 129)]:
        a, b = _dyadic(M, N, K)
        C = f((a / 8.0).astype(np.float32), (b / 8.0).astype(np.float32))
        assert np.array_equal(C, (a @ b).astype(np.float64) / 64.0), (M, N, K)


PINS = [pin_worked_examples, pin_exact_rational, pin_integer_exact, pin_identity,
        pin_permutation, pin_transpose, pin_closed_forms, pin_dyadic_pattern]


def _oracle_c(oracle_mod):
    return lambda A, B: oracle_mod.gemm(A, B, with_scale=False)[0]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(oracle_mod, pin):
    pin(_oracle_c(oracle_mod))


def test_dyadic_512_cube(oracle_mod):
    a, b = _dyadic(512, 512, 512)
    C, _ = oracle_mod.gemm((a / 8.0).astype(np.float32), (b / 8.0).astype(np.float32),
                           with_scale=False)
    assert np.array_equal(C, (a @ b).astype(np.float64) / 64.0)


def test_scale_properties(oracle_mod):
    A, B = make_inputs(31, 77, 19, 8, "normal")
    C, S = oracle_mod.gemm(A, B)
    assert np.all(S >= np.abs(C))
    # S is the product of the absolute values: equal to C on non-negative inputs
    C_abs, S_abs = oracle_mod.gemm(np.abs(A), np.abs(B))
    assert np.array_equal(C_abs, S)
    assert np.array_equal(S_abs, S)
    # flipping the sign of A flips C and leaves S alone
    C_neg, S_neg = oracle_mod.gemm(-A, B)
    assert np.array_equal(C_neg, -C)
    assert np.array_equal(S_neg, S)
    # exact integer check of S
    Ai, Bi = make_inputs(12, 40, 9, 2, "int8")
    _, Si = oracle_mod.gemm(Ai, Bi)
    assert np.array_equal(Si, (np.abs(Ai.astype(np.int64)) @ np.abs(Bi.astype(np.int64))).astype(np.float64))


def test_entries_match_full(oracle_mod):
    A, B = make_inputs(40, 300, 50, 9, "uniform")
    C, S = oracle_mod.gemm(A, B)
    rows = np.array([0, 39, 17, 5, 39], dtype=np.int64)
    cols = np.array([0, 49, 23, 0, 0], dtype=np.int64)
    c, s = oracle_mod.entries(A, B, rows, cols)
    assert np.array_equal(c, C[rows, cols])
    assert np.array_equal(s, S[rows, cols])


def test_thread_count_invariance(oracle_mod):
    A, B = make_inputs(37, 200, 41, 10, "normal")
    C1, S1 = oracle_mod.gemm(A, B, threads=1)
    C7, S7 = oracle_mod.gemm(A, B, threads=7)
    assert np.array_equal(C1, C7) and np.array_equal(S1, S7)


def test_rejects_bad_shapes(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.gemm(np.zeros((2, 3), np.float32), np.zeros((4, 2), np.float32))
    with pytest.raises(RuntimeError):
        oracle_mod.entries(np.zeros((2, 3), np.float32), np.zeros((3, 2), np.float32),
                           [2], [0])


# ---------------------------------------------------------------------------------
# Planted mistakes: each must fail at least one pin.
# ---------------------------------------------------------------------------------

def _loop_gemm(A, B, acc_dtype=np.float64, n_stop=0, last_sign=1.0, swap_out=False,
               a_transposed=False):
    A = np.asarray(A, dtype=np.float32)
    B = np.asarray(B, dtype=np.float32)
    if a_transposed:
        A = A.T
    M, N = A.shape
    K = B.shape[1]
    C = np.zeros((M, K), dtype=acc_dtype)
    for n in range(N - n_stop):
        sign = last_sign if n == N - 1 else 1.0
        term = np.outer(A[:, n].astype(acc_dtype), B[n, :].astype(acc_dtype))
        C = (C + acc_dtype(sign) * term).astype(acc_dtype)
    C = C.astype(np.float64)
    return C.T if swap_out else C


MUTANTS = {
    "b_transposed": lambda A, B: _loop_gemm(A, np.ascontiguousarray(B.T)),
    "a_transposed": lambda A, B: _loop_gemm(A, B, a_transposed=True),
    "dropped_last_term": lambda A, B: _loop_gemm(A, B, n_stop=1),
    "wrong_sign_last_term": lambda A, B: _loop_gemm(A, B, last_sign=-1.0),
    "float32_accumulator": lambda A, B: _loop_gemm(A, B, acc_dtype=np.float32),
    "transposed_output": lambda A, B: _loop_gemm(A, B, swap_out=True),
}


def test_planted_reference_passes_pins():
    # the unmutated loop form must pass every pin, or the mutant test proves nothing
    for pin in PINS:
        pin(_loop_gemm)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    f = MUTANTS[name]
    failed = []
    for pin in PINS:
        try:
            pin(f)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
