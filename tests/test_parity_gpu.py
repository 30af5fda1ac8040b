"""GPU parity: the library (through its C ABI) against the CPU oracle.

Shapes and inputs follow the workloads: the 512^3 cube (seed 0), the ragged sweep
(seed 1), the performance shape 8192 x 6144 x 4096 (seed 2), the one-row/one-column
and thin shapes (seed 3, normal entries) and the largest/aspect sweep (seed 4).
Integer-valued inputs must match bit for bit; uniform and normal inputs must satisfy
|C - C_exact| <= tol * (|A|.|B|) elementwise (tol 1e-5 for the FP32-accurate modes,
2e-3 for 1xTF32). Every configuration of the workloads, up to 8192^3, is checked element
by element against the oracle's full product; same-sign inputs over long reductions
(where accumulation errors add up instead of cancelling) are checked the same way.
Integer products at full size, too slow to repeat for every mode on the CPU, are checked
on sampled entries and whole rows, plus exact properties on the full output.
"""

import numpy as np
import pytest

import dense_fp32_gemm_sgemm_gb300 as sg
from tests.golden.load import worked_examples
from tests.gpu_util import (MODE_IDS, TOL, assert_exact, assert_within, check_sampled,
                            fp16_scale_term, inputs, run_gpu, split_elements, to_dev,
                            torch_cuda)

pytestmark = pytest.mark.gpu

ALL_MODES = [sg.MODE_FP32, sg.MODE_FP32_SIMT, sg.MODE_FP32_3XTF32, sg.MODE_3XFP16_SCALED,
             sg.MODE_TF32]
MODE_PARAMS = [pytest.param(m, id=MODE_IDS[m]) for m in ALL_MODES]

RAGGED = [(1, 1, 1), (2, 2, 2), (1, 3, 1), (17, 19, 31), (127, 129, 65), (1000, 333, 777),
          (4097, 1, 4095)]
# shapes from the pages' checks, relabelled to (M, N, K): partial tiles, several blocks,
# and the tiled-chapter cases
PAGE_SHAPES = [(129, 96, 132), (256, 96, 256), (3, 5, 4), (17, 19, 23), (257, 129, 193),
               (255, 257, 129)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_fp32_gemm_sgemm_gb300 import build
    build.build()
    torch_cuda()


def _oracle(A, B):
    import oracle
    return oracle.gemm(A, B)


_FULL_REF = {}


def _full_reference(M, N, K, seed, dist):
    """Inputs and the oracle's full product and |A|.|B| for one workload, kept until a
    different workload is asked for (the tests of one shape run one after another, so
    each full product is computed once for all modes)."""
    key = (M, N, K, seed, dist)
    if key not in _FULL_REF:
        _FULL_REF.clear()
        A, B = inputs(M, N, K, seed, dist)
        C_ref, S = _oracle(A, B)
        _FULL_REF[key] = dict(A=A, B=B, C_ref=C_ref, S=S)
    return _FULL_REF[key]


def _bound_extra(mode, A, B):
    """The absolute term of the scaled FP16 mode's stated bound (None for every other
    mode, whose bound is tol * S alone)."""
    return fp16_scale_term(A, B) if mode == sg.MODE_3XFP16_SCALED else None


@pytest.mark.parametrize("mode", MODE_PARAMS)
def test_worked_examples(mode):
    for case in worked_examples():
        C = run_gpu(case["A"], case["B"], mode)
        assert_exact(C, case["C"].astype(np.float64), case["name"])


@pytest.mark.parametrize("mode", MODE_PARAMS)
def test_cube_512(mode):
    A, B = inputs(512, 512, 512, 0, "uniform")
    C_ref, S = _oracle(A, B)
    assert_within(run_gpu(A, B, mode), C_ref, S, TOL[mode], "512^3 uniform")
    Ai, Bi = inputs(512, 512, 512, 0, "int4")
    Ci_ref, _ = _oracle(Ai, Bi)
    assert_exact(run_gpu(Ai, Bi, mode), Ci_ref, "512^3 int4")


@pytest.mark.parametrize("mode", MODE_PARAMS)
@pytest.mark.parametrize("shape", RAGGED, ids=[f"{m}x{n}x{k}" for m, n, k in RAGGED])
def test_ragged_sweep(mode, shape):
    M, N, K = shape
    A, B = inputs(M, N, K, 1, "uniform")
    C_ref, S = _oracle(A, B)
    assert_within(run_gpu(A, B, mode), C_ref, S, TOL[mode], f"{shape} uniform")
    Ai, Bi = inputs(M, N, K, 1, "int8")
    Ci_ref, _ = _oracle(Ai, Bi)
    assert_exact(run_gpu(Ai, Bi, mode), Ci_ref, f"{shape} int8")


@pytest.mark.parametrize("mode", MODE_PARAMS)
@pytest.mark.parametrize("shape", PAGE_SHAPES, ids=[f"{m}x{n}x{k}" for m, n, k in PAGE_SHAPES])
def test_page_shapes(mode, shape):
    M, N, K = shape
    A, B = inputs(M, N, K, 5, "uniform")
    C_ref, S = _oracle(A, B)
    assert_within(run_gpu(A, B, mode), C_ref, S, TOL[mode], f"{shape}")
    # the integer/8 pattern of the tiled-multiplication chapter: exact
    a = ((np.arange(M * N) * 17) % 13 - 6).reshape(M, N) / 8.0
    b = ((np.arange(N * K) * 29) % 11 - 5).reshape(N, K) / 8.0
    a = a.astype(np.float32)
    b = b.astype(np.float32)
    Cd_ref, _ = _oracle(a, b)
    assert_exact(run_gpu(a, b, mode), Cd_ref, f"{shape} eighths")


@pytest.mark.parametrize("mode", MODE_PARAMS)
@pytest.mark.parametrize("shape", [(130, 129, 131), (64, 64, 64), (300, 500, 260), (1, 9, 7),
                                   (9, 7, 1)])
def test_unaligned_pointers(mode, shape):
    M, N, K = shape
    A, B = inputs(M, N, K, 6, "uniform")
    C_ref, S = _oracle(A, B)
    for off in (1, 2, 3):
        assert_within(run_gpu(A, B, mode, offset=off), C_ref, S, TOL[mode],
                      f"{shape} offset {off}")


@pytest.mark.parametrize("mode", MODE_PARAMS)
def test_unaligned_pointers_large(mode):
    """Operands and C one float off 16-byte alignment at a size where every mode takes its
    large-product path with the copies that such pointers force: the operand pre-pass's
    row-by-row split instead of the fused one, no raw A plane, the row-wise epilogue
    instead of TMA stores of C, 1xTF32 on 256 x 512 tiles, and the 128 x 128 FFMA kernel's
    4-byte copies. Every element against the oracle."""
    M, N, K = 4096, 2048, 8192
    ref = _full_reference(M, N, K, 6, "uniform")
    got = run_gpu(ref["A"], ref["B"], mode, offset=1)
    assert_within(got, ref["C_ref"], ref["S"], TOL[mode], f"{(M, N, K)} offset 1",
                  extra=_bound_extra(mode, ref["A"], ref["B"]))


@pytest.mark.parametrize("mode", MODE_PARAMS)
@pytest.mark.parametrize("shape", [(200, 77, 130), (1, 300, 259), (259, 300, 1), (128, 128, 128)])
def test_guard_bands(mode, shape):
    """C sits inside a NaN-filled buffer: every C element must be written and no float
    outside C may change."""
    torch = torch_cuda()
    M, N, K = shape
    A, B = inputs(M, N, K, 7, "uniform")
    C_ref, S = _oracle(A, B)
    guard = 1024
    buf = torch.full((guard + M * K + guard,), float("nan"), device="cuda")
    dC = buf[guard:guard + M * K].view(M, K)
    dA, dB = to_dev(A), to_dev(B)
    rc = sg.lib().solve_ex(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), M, N, K, mode,
                           int(torch.cuda.current_stream().cuda_stream))
    assert rc == sg.OK
    host = buf.cpu().numpy()
    assert np.all(np.isnan(host[:guard])) and np.all(np.isnan(host[-guard:]))
    assert_within(host[guard:guard + M * K].reshape(M, K), C_ref, S, TOL[mode], "inside")


# Small FFMA products with 16-byte rows: the reduction split among four groups of threads
# per CTA, in stages of 64 reduction elements (16 per group). Shapes: one stage and one
# CTA; a ragged second stage that only group 0 reaches (N = 68) with ragged rows and
# columns; reductions shorter than one group's slice (N = 12); 16 x 32 tiles (fewer
# 16 x 64 tiles than SMs) and 16 x 64 tiles with a ragged last stage; a reduction just
# under the 1024 limit of the default mode's choice.
SPLIT_SMALL = [(16, 64, 64), (33, 68, 100), (1000, 12, 1000), (160, 1020, 640),
               (384, 260, 1024), (200, 1016, 360)]


@pytest.mark.parametrize("mode", [pytest.param(m, id=MODE_IDS[m])
                                  for m in (sg.MODE_FP32, sg.MODE_FP32_SIMT)])
@pytest.mark.parametrize("shape", SPLIT_SMALL, ids=[f"{m}x{n}x{k}" for m, n, k in SPLIT_SMALL])
def test_small_split_reduction(mode, shape):
    M, N, K = shape
    assert sg.plan(M, N, K, mode)[0] == sg.KERNEL_SIMT
    A, B = inputs(M, N, K, 1, "uniform")
    C_ref, S = _oracle(A, B)
    assert_within(run_gpu(A, B, mode), C_ref, S, TOL[mode], f"{shape} uniform")
    A, B = inputs(M, N, K, 1, "normal")
    C_ref, S = _oracle(A, B)
    assert_within(run_gpu(A, B, mode), C_ref, S, TOL[mode], f"{shape} normal")
    Ai, Bi = inputs(M, N, K, 1, "int8")
    Ci_ref, _ = _oracle(Ai, Bi)
    assert_exact(run_gpu(Ai, Bi, mode), Ci_ref, f"{shape} int8")


@pytest.mark.parametrize("mode", MODE_PARAMS)
def test_thin_shapes(mode):
    """One-row, one-column and thin-reduction shapes, N(0,1) entries, seed 3."""
    import oracle
    A, B = inputs(1, 8192, 8192, 3, "normal")
    C_ref, S = oracle.gemm(A, B)
    assert_within(run_gpu(A, B, mode), C_ref, S, TOL[mode], "1x8192x8192")
    A, B = inputs(8192, 8192, 1, 3, "normal")
    C_ref, S = oracle.gemm(A, B)
    assert_within(run_gpu(A, B, mode), C_ref, S, TOL[mode], "8192x8192x1")
    ref = _full_reference(8192, 64, 8192, 3, "normal")
    assert_within(run_gpu(ref["A"], ref["B"], mode), ref["C_ref"], ref["S"], TOL[mode],
                  "8192x64x8192")


SHORT_N = [(1000, 1, 777), (129, 2, 4095), (64, 3, 130), (2, 4, 2), (333, 4, 1001),
           (257, 5, 63), (1000, 8, 777), (4097, 16, 5)]


@pytest.mark.parametrize("mode", MODE_PARAMS)
@pytest.mark.parametrize("shape", SHORT_N, ids=[f"{m}x{n}x{k}" for m, n, k in SHORT_N])
def test_short_reductions(mode, shape):
    """Short reductions (N <= 4 take the short-reduction kernel in the FP32 and TF32
    modes, larger N the GEMM kernels): within the mode's bound on uniform entries,
    bit-exact on integers, also from pointers that are not 16-byte aligned."""
    import oracle
    M, N, K = shape
    A, B = inputs(M, N, K, 23, "uniform")
    C_ref, S = oracle.gemm(A, B)
    assert_within(run_gpu(A, B, mode), C_ref, S, TOL[mode], f"{shape} uniform")
    assert_within(run_gpu(A, B, mode, offset=1), C_ref, S, TOL[mode], f"{shape} offset")
    Ai, Bi = inputs(M, N, K, 23, "int8")
    Ci_ref, _ = oracle.gemm(Ai, Bi)
    assert_exact(run_gpu(Ai, Bi, mode), Ci_ref, f"{shape} int8")
    if N == 1 and mode in (sg.MODE_FP32, sg.MODE_FP32_SIMT):
        # FP32 FMA kernels form one correctly rounded product per element: the exact
        # product rounded to float
        np.testing.assert_array_equal(run_gpu(A, B, mode), C_ref.astype(np.float32))


@pytest.mark.parametrize("mode", MODE_PARAMS)
def test_short_reduction_full_size(mode):
    """8192 x 4 x 8192 (C is 256 MiB): every element against the oracle."""
    ref = _full_reference(8192, 4, 8192, 24, "normal")
    assert_within(run_gpu(ref["A"], ref["B"], mode), ref["C_ref"], ref["S"], TOL[mode],
                  "8192x4x8192")


# shapes where neither the device schedule nor the host round trip's 1024-row chunks split
# tiles along the reduction, so that both compute every tile whole; the fused split
# claims rows in 1024-column chunks, and the last two shapes end in a partial chunk
FUSED = [(7000, 4096, 4096), (8000, 2048, 4096), (7000, 3000, 4096), (8000, 5000, 4096)]


@pytest.mark.parametrize("mode", [sg.MODE_FP32, sg.MODE_TF32], ids=["fp32", "tf32"])
@pytest.mark.parametrize("shape", FUSED, ids=[f"{m}x{n}x{k}" for m, n, k in FUSED])
def test_fused_operand_split(mode, shape):
    """Large aligned A whose first round of tiles reads under half of its rows: the GEMM
    kernel splits A itself, and the last 256-row block is partial (88 and 64 rows). The
    result must equal, bit for bit, the host round trip, which splits A in a separate
    pass, wherever neither path's schedule splits the reduction of an element's tile (the
    two schedules differ: the round trip computes 1024-row chunks); every element of both
    must meet the oracle's bound; integers (sampled entries and whole rows) exactly."""
    M, N, K = shape
    ref = _full_reference(M, N, K, 31, "uniform")
    A, B = ref["A"], ref["B"]
    C = run_gpu(A, B, mode)
    C_host = sg.solve_host(A, B, mode=mode)
    same = ~split_elements(M, N, K, mode, chunk_rows=1024)
    assert same.mean() > 0.5, "too few elements summed alike to compare"
    np.testing.assert_array_equal(C_host[same], C[same])
    assert_within(C, ref["C_ref"], ref["S"], TOL[mode], str(shape))
    assert_within(C_host, ref["C_ref"], ref["S"], TOL[mode], f"{shape} host round trip")
    Ai, Bi = inputs(M, N, K, 31, "int8")
    check_sampled(run_gpu(Ai, Bi, mode), Ai, Bi, 0.0, seed=32, count=1024, rows_full=4,
                  exact=True, what=f"{shape} int8")
    assert sg.device_error() == sg.OK


_HEADLINE_REF = {}


def _headline_reference():
    """The oracle's full 8192 x 6144 x 4096 product and |A|.|B| (computed once)."""
    if not _HEADLINE_REF:
        import oracle
        A, B = inputs(8192, 6144, 4096, 2, "uniform")
        C_ref, S = oracle.gemm(A, B)
        _HEADLINE_REF.update(A=A, B=B, C_ref=C_ref, S=S)
    return _HEADLINE_REF


@pytest.mark.parametrize("mode", MODE_PARAMS)
def test_headline_shape(mode):
    """8192 x 6144 x 4096, uniform, seed 2: every element of the device result and of the
    pipelined host round trip against the oracle's full product."""
    ref = _headline_reference()
    A, B = ref["A"], ref["B"]
    assert_within(run_gpu(A, B, mode), ref["C_ref"], ref["S"], TOL[mode], "headline")
    assert_within(sg.solve_host(A, B, mode=mode), ref["C_ref"], ref["S"], TOL[mode],
                  "headline host round trip")


@pytest.mark.parametrize("mode", MODE_PARAMS)
def test_row_permutation_exact(mode):
    """An exact property on a full output: with every tile computed whole (7000 x 4096 x
    4096 is cut neither along the reduction nor into chunks), permuting the rows of A
    permutes the rows of C bit for bit."""
    torch = torch_cuda()
    from dense_fp32_gemm_sgemm_gb300.inputs import make_permutation
    M, N, K = 7000, 4096, 4096
    A, B = inputs(M, N, K, 2, "uniform")
    dA, dB = to_dev(A), to_dev(B)
    dC = torch.empty(M, K, device="cuda")
    stream = int(torch.cuda.current_stream().cuda_stream)
    assert sg.lib().solve_ex(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), M, N, K, mode,
                             stream) == sg.OK
    p = torch.from_numpy(make_permutation(M, 2)).cuda()
    dAp = dA[p].contiguous()
    dCp = torch.empty_like(dC)
    assert sg.lib().solve_ex(dAp.data_ptr(), dB.data_ptr(), dCp.data_ptr(), M, N, K, mode,
                             stream) == sg.OK
    assert torch.equal(dCp, dC[p])


@pytest.mark.parametrize("mode", MODE_PARAMS)
def test_headline_shape_integer_exact(mode):
    M, N, K = 8192, 6144, 4096
    A, B = inputs(M, N, K, 2, "int8")
    C = run_gpu(A, B, mode)
    check_sampled(C, A, B, 0.0, seed=12, count=1024, rows_full=4, exact=True,
                  what="headline int8")


SPLIT = [(64, 8192, 64), (256, 8192, 256), (200, 4000, 300), (1024, 2048, 1000)]


@pytest.mark.parametrize("mode", MODE_PARAMS)
@pytest.mark.parametrize("shape", SPLIT, ids=[f"{m}x{n}x{k}" for m, n, k in SPLIT])
def test_long_reduction_few_tiles(mode, shape):
    """Shapes whose output tiles cannot fill the GPU: the tensor-core path splits the
    reduction and adds the split partials in a fixed order. Exact on integers, within
    the bound otherwise, and reproducible bit for bit."""
    M, N, K = shape
    A, B = inputs(M, N, K, 16, "uniform")
    C_ref, S = _oracle(A, B)
    C1 = run_gpu(A, B, mode)
    assert_within(C1, C_ref, S, TOL[mode], f"{shape} uniform")
    assert np.array_equal(C1, run_gpu(A, B, mode))
    Ai, Bi = inputs(M, N, K, 16, "int8")
    Ci_ref, _ = _oracle(Ai, Bi)
    assert_exact(run_gpu(Ai, Bi, mode), Ci_ref, f"{shape} int8")


@pytest.mark.parametrize("mode", MODE_PARAMS)
@pytest.mark.parametrize("shape", [(2560, 1024, 2048), (8191, 6143, 4097)],
                         ids=["2560x1024x2048", "8191x6143x4097"])
def test_nearly_empty_last_round(mode, shape):
    """Tile counts whose last round of CTA pairs is nearly empty: the tensor-core path
    splits those tiles' reductions across the idle pairs. Every element against the
    oracle's full product; bit-exact on integers (sampled entries and whole rows)."""
    M, N, K = shape
    ref = _full_reference(M, N, K, 17, "uniform")
    A, B = ref["A"], ref["B"]
    assert_within(run_gpu(A, B, mode), ref["C_ref"], ref["S"], TOL[mode], f"{shape} uniform",
                  _bound_extra(mode, A, B))
    Ai, Bi = inputs(M, N, K, 17, "int8")
    check_sampled(run_gpu(Ai, Bi, mode), Ai, Bi, 0.0, seed=18, count=1024, rows_full=4,
                  exact=True, what=f"{shape} int8")


# shapes whose last round the 3xTF32 schedule recuts into narrower pieces: ragged right
# edges that pieces run past (K = 4001, 4095, 4097), C rows that are not 16-byte aligned
# (odd K, or a C pointer offset by one float: row-by-row stores), the narrowest pieces (32
# columns) and the aligned TMA-store path
RECUT = [((3000, 700, 4001), 0), ((4097, 129, 4095), 0), ((8191, 64, 4097), 0),
         ((4000, 1000, 4000), 0), ((4000, 1000, 4000), 1), ((2048, 512, 8192), 3)]


@pytest.mark.parametrize("shape,offset", RECUT,
                         ids=[f"{m}x{n}x{k}+{o}" for (m, n, k), o in RECUT])
def test_recut_last_round(shape, offset):
    """Every element of a product whose last round is recut into pieces (one per CTA pair,
    the pair MMA's N set to the piece width) against the oracle; bit-exact on integers."""
    M, N, K = shape
    mode = sg.MODE_FP32
    assert sg.plan(M, N, K, mode)[0] == sg.KERNEL_TC_3XTF32
    assert any(u[2] != 256 for u in sg.plan_units(M, N, K, mode)), "no longer recut"
    A, B = inputs(M, N, K, 40, "uniform")
    C_ref, S = _oracle(A, B)
    assert_within(run_gpu(A, B, mode, offset=offset), C_ref, S, TOL[mode], f"{shape} uniform")
    Ai, Bi = inputs(M, N, K, 41, "int8")
    Ci_ref, _ = _oracle(Ai, Bi)
    assert_exact(run_gpu(Ai, Bi, mode, offset=offset), Ci_ref, f"{shape} int8")


LARGE = [(8192, 8192, 8192), (8192, 8192, 1024), (1024, 8192, 8192), (8191, 6143, 4097)]


@pytest.mark.parametrize("mode", MODE_PARAMS)
@pytest.mark.parametrize("shape", LARGE, ids=[f"{m}x{n}x{k}" for m, n, k in LARGE])
def test_large_sweep(mode, shape):
    """The largest allowed cube and the aspect sweep, uniform entries, seed 4: every
    element against the oracle's full product (these shapes run the recut and split last
    rounds and, at 8191 x 6143 x 4097, the loaders for rows that are not 16-byte aligned,
    all at full size)."""
    ref = _full_reference(*shape, 4, "uniform")
    A, B = ref["A"], ref["B"]
    assert_within(run_gpu(A, B, mode), ref["C_ref"], ref["S"], TOL[mode], str(shape),
                  _bound_extra(mode, A, B))


SAME_SIGN = [(512, 8192, 512), (8192, 6144, 4096)]


@pytest.mark.parametrize("mode", MODE_PARAMS)
@pytest.mark.parametrize("shape", SAME_SIGN, ids=[f"{m}x{n}x{k}" for m, n, k in SAME_SIGN])
def test_same_sign_long_reduction(mode, shape):
    """All entries in [0, 1): no term cancels another, so every rounding error of the
    accumulation adds up, and more so the longer the reduction. This is where a biased
    accumulator would break the elementwise bound first (the pages ask for the error
    budget to be re-checked for longer reductions and other input distributions). Every
    element against the oracle's full product, in every mode under its own bound."""
    ref = _full_reference(*shape, 50, "uniform01")
    A, B = ref["A"], ref["B"]
    assert_within(run_gpu(A, B, mode), ref["C_ref"], ref["S"], TOL[mode],
                  f"{shape} same-sign", _bound_extra(mode, A, B))


@pytest.mark.parametrize("mode", MODE_PARAMS)
def test_identity_full_size(mode):
    """A . I = A and I . B = B: bit for bit on the CUDA-core kernel (every product is x*1
    or x*0 and every other addend is zero); the TF32-based kernels see rounded or split
    inputs, so there the bound |C - A| <= tol * |A| applies. Here each output has a single
    nonzero term, so the FP16 three-product mode's absolute term (an element of A far below
    its row's largest keeps fewer bits) decides, and its full bound applies."""
    n = 2048
    A, _ = inputs(3000, n, 1, 8, "normal")
    eye = np.eye(n, dtype=np.float32)
    exact = sg.plan(3000, n, n, mode)[0] == sg.KERNEL_SIMT
    f16 = mode == sg.MODE_3XFP16_SCALED
    got = run_gpu(A, eye, mode)
    if exact:
        assert np.array_equal(got, A)
    else:
        assert_within(got, A.astype(np.float64), np.abs(A).astype(np.float64), TOL[mode], "A.I",
                      fp16_scale_term(A, eye) if f16 else None)
    _, B = inputs(1, n, 1500, 9, "uniform")
    got = run_gpu(eye, B, mode)
    if exact:
        assert np.array_equal(got, B)
    else:
        assert_within(got, B.astype(np.float64), np.abs(B).astype(np.float64), TOL[mode], "I.B",
                      fp16_scale_term(eye, B) if f16 else None)


@pytest.mark.parametrize("mode", MODE_PARAMS)
def test_deterministic(mode):
    A, B = inputs(1000, 2000, 1500, 10, "uniform")
    C1 = run_gpu(A, B, mode)
    C2 = run_gpu(A, B, mode)
    assert np.array_equal(C1, C2)


def test_solve_uses_thread_stream():
    import oracle
    torch = torch_cuda()
    A, B = inputs(300, 200, 100, 11, "uniform")
    dA, dB = to_dev(A), to_dev(B)
    dC = torch.empty(300, 100, device="cuda")
    s = torch.cuda.Stream()
    L = sg.lib()
    L.sgemm_set_stream(int(s.cuda_stream))
    try:
        L.solve(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), 300, 200, 100)
        assert L.sgemm_last_status() == sg.OK
        s.synchronize()
    finally:
        L.sgemm_set_stream(None)
    C_ref, S = oracle.gemm(A, B)
    assert_within(dC.cpu().numpy(), C_ref, S, 1e-5, "solve on side stream")


def test_solve_host_round_trip():
    import oracle
    A, B = inputs(333, 444, 555, 12, "uniform")
    C = sg.solve_host(A, B)
    C_ref, S = oracle.gemm(A, B)
    assert_within(C, C_ref, S, 1e-5, "solve_host")


@pytest.mark.parametrize("mode", [sg.MODE_FP32, sg.MODE_TF32], ids=["fp32", "tf32"])
@pytest.mark.parametrize("shape", [(2304, 300, 520), (2049, 129, 257)], ids=["2304x300x520", "2049x129x257"])
def test_solve_host_pipelined(mode, shape):
    """Host round trips of tensor-core products with M >= 2048 upload, multiply and
    download in overlapping row chunks (the last one ragged); results must match the
    oracle like the device-pointer path, bit-exact on integers."""
    import oracle
    M, N, K = shape
    A, B = inputs(M, N, K, 19, "uniform")
    C_ref, S = oracle.gemm(A, B)
    assert_within(sg.solve_host(A, B, mode=mode), C_ref, S, TOL[mode], f"{shape} uniform")
    Ai, Bi = inputs(M, N, K, 19, "int8")
    Ci_ref, _ = oracle.gemm(Ai, Bi)
    assert_exact(sg.solve_host(Ai, Bi, mode=mode), Ci_ref, f"{shape} int8")
    assert sg.device_error() == sg.OK


def test_concurrent_host_round_trips():
    """Two threads run pipelined host round trips at the same time; they share the
    library's internal copy and compute streams and must both get their own product."""
    import threading
    import oracle
    shapes = [(2304, 256, 520), (2048, 300, 264)]
    data = [inputs(M, N, K, 40 + i, "int8") for i, (M, N, K) in enumerate(shapes)]
    out = [None, None]
    errors = []

    def work(i):
        try:
            torch = torch_cuda()
            with torch.cuda.stream(torch.cuda.Stream()):
                for _ in range(3):
                    out[i] = sg.solve_host(*data[i], mode=sg.MODE_FP32)
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i in range(2):
        C_ref, _ = oracle.gemm(*data[i])
        assert_exact(out[i], C_ref, f"thread {i}")


# one product of each dispatch class that chains launches (pre-pass -> GEMM -> split
# reduction, the 256 x 512 1xTF32 kernel with its split tail, the small FFMA kernel, a
# fused split), enqueued back to back
BACK_TO_BACK = [((512, 512, 512), sg.MODE_FP32_3XTF32), ((2048, 2048, 4096), sg.MODE_TF32),
                ((300, 200, 100), sg.MODE_FP32), ((4096, 4096, 4096), sg.MODE_FP32),
                ((8192, 2048, 4096), sg.MODE_TF32), ((1000, 333, 777), sg.MODE_TF32),
                ((7000, 4096, 2048), sg.MODE_FP32)]


def test_back_to_back_calls_without_sync():
    """Products of different shapes and kernels enqueued on one stream with no
    synchronisation between them, twice round, each into its own C: every launch chain
    (pre-pass, GEMM started early by programmatic dependent launch, split reduction) must
    wait for its own inputs, and workspace blocks the pool hands from one call to the
    next must not be overwritten early. Every result within the bound of its mode."""
    import oracle
    torch = torch_cuda()
    stream = torch.cuda.Stream()
    cases = []
    for i, ((M, N, K), mode) in enumerate(BACK_TO_BACK):
        A, B = inputs(M, N, K, 60 + i, "uniform")
        cases.append((A, B, mode, to_dev(A), to_dev(B),
                      [torch.full((M, K), float("nan"), device="cuda") for _ in range(2)]))
    torch.cuda.synchronize()
    h = int(stream.cuda_stream)
    for rnd in range(2):
        for A, B, mode, dA, dB, outs in cases:
            M, N, K = A.shape[0], A.shape[1], B.shape[1]
            rc = sg.lib().solve_ex(dA.data_ptr(), dB.data_ptr(), outs[rnd].data_ptr(), M, N, K,
                                   mode, h)
            assert rc == sg.OK, sg.lib().sgemm_status_string(rc)
    stream.synchronize()
    for A, B, mode, _, _, outs in cases:
        C_ref, S = _oracle(A, B)
        for rnd in range(2):
            assert_within(outs[rnd].cpu().numpy(), C_ref, S, TOL[mode],
                          f"{A.shape[0]}x{A.shape[1]}x{B.shape[1]} mode {mode} round {rnd}")
    assert sg.device_error() == sg.OK


def test_two_streams_concurrently():
    """Two streams each running a chain of tensor-core products at the same time (each
    call with its own workspace from the pool): both results within the bound."""
    torch = torch_cuda()
    shapes = [((4096, 4096, 4096), sg.MODE_FP32), ((8192, 2048, 4096), sg.MODE_TF32)]
    data = []
    for i, ((M, N, K), mode) in enumerate(shapes):
        A, B = inputs(M, N, K, 70 + i, "uniform")
        data.append((A, B, mode, to_dev(A), to_dev(B),
                     torch.full((M, K), float("nan"), device="cuda"), torch.cuda.Stream()))
    torch.cuda.synchronize()
    for _ in range(3):
        for A, B, mode, dA, dB, dC, st in data:
            rc = sg.lib().solve_ex(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), A.shape[0],
                                   A.shape[1], B.shape[1], mode, int(st.cuda_stream))
            assert rc == sg.OK, sg.lib().sgemm_status_string(rc)
    torch.cuda.synchronize()
    for A, B, mode, _, _, dC, _ in data:
        C_ref, S = _oracle(A, B)
        assert_within(dC.cpu().numpy(), C_ref, S, TOL[mode], f"{A.shape} mode {mode}")
    assert sg.device_error() == sg.OK


def test_python_wrappers_and_counters():
    import oracle
    torch = torch_cuda()
    A, B = inputs(70, 80, 90, 13, "uniform")
    before = sg.launch_count()
    C = sg.matmul(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda())
    torch.cuda.synchronize()
    assert sg.launch_count() > before
    C_ref, S = oracle.gemm(A, B)
    assert_within(C.cpu().numpy(), C_ref, S, 1e-5, "matmul")
    assert sg.device_error() == sg.OK


def test_kernel_event_hook():
    torch = torch_cuda()
    A, B = inputs(1024, 1024, 1024, 14, "uniform")
    dA, dB = to_dev(A), to_dev(B)
    dC = torch.empty(1024, 1024, device="cuda")
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    # torch creates the CUDA event on first record; record once so the handles exist
    e0.record()
    e1.record()
    sg.lib().sgemm_set_kernel_events(e0.cuda_event, e1.cuda_event)
    sg.solve(dA, dB, dC)
    torch.cuda.synchronize()
    assert e0.elapsed_time(e1) > 0.0


NONFINITE_SHAPES = [(300, 200, 500), (512, 512, 512), (2048, 2048, 2048), (1000, 4, 777)]


@pytest.mark.parametrize("mode", MODE_PARAMS)
@pytest.mark.parametrize("shape", NONFINITE_SHAPES, ids=[f"{m}x{n}x{k}" for m, n, k in NONFINITE_SHAPES])
def test_nonfinite_input_stays_in_its_row_and_column(mode, shape):
    """Inputs are assumed finite, but a non-finite one must not leak: with A[r0][n0] = +Inf
    and B[n1][k1] = NaN, row r0 and column k1 of C are non-finite (3xTF32 turns the Inf
    into NaN through its lo part, Inf - Inf; the other paths give +-Inf or NaN), and every
    other element is finite and within the mode's bound of the oracle's product of the
    unmodified inputs, whatever split parts, recut pieces or skinny kernel the shape uses."""
    M, N, K = shape
    A, B = inputs(M, N, K, 61, "uniform")
    C_ref, S = _oracle(A, B)
    r0, n0, n1, k1 = M // 3, N // 2, (N - 1) // 3, (2 * K) // 3
    A2, B2 = A.copy(), B.copy()
    A2[r0, n0] = np.inf
    B2[n1, k1] = np.nan
    C = run_gpu(A2, B2, mode)
    nonzero = B[n0, :] != 0
    assert not np.isfinite(C[r0, nonzero]).any(), "row of the Inf has finite entries"
    assert not np.isfinite(C[:, k1]).any(), "column of the NaN has finite entries"
    keep = np.ones((M, K), dtype=bool)
    keep[r0, :] = False
    keep[:, k1] = False
    assert_within(C[keep], C_ref[keep], S[keep], TOL[mode], f"{shape} outside the row and column")
    assert sg.device_error() == sg.OK


@pytest.mark.parametrize("scale", [1e5, 1e-5], ids=["x1e5", "x1e-5"])
def test_nonfinite_input_keeps_neighbour_scales_3xfp16(scale):
    """The scaled FP16 mode takes one power-of-two scale per row of A and per 128-column
    block of B from the largest magnitude there. An Inf or a NaN must not count as that
    largest magnitude: with B far from unit scale (1e5: its FP16 hi pieces would overflow
    unscaled; 1e-5: its lo pieces would fall below FP16's normal range), every element
    outside the non-finite input's row and column must still meet the mode's bound."""
    mode = sg.MODE_3XFP16_SCALED
    M, N, K = 300, 200, 500
    A, B = inputs(M, N, K, 62, "uniform")
    A = (A * np.float32(scale)).astype(np.float32)
    B = (B * np.float32(scale)).astype(np.float32)
    C_ref, S = _oracle(A, B)
    r0, n0, n1, k1 = M // 3, N // 2, (N - 1) // 3, (2 * K) // 3
    A2, B2 = A.copy(), B.copy()
    A2[r0, n0] = np.inf
    B2[n1, k1] = np.nan
    C = run_gpu(A2, B2, mode)
    assert not np.isfinite(C[:, k1]).any(), "column of the NaN has finite entries"
    keep = np.ones((M, K), dtype=bool)
    keep[r0, :] = False
    keep[:, k1] = False
    extra = fp16_scale_term(A, B)
    assert_within(C[keep], C_ref[keep], S[keep], TOL[mode], f"x{scale} outside", extra[keep])
    assert sg.device_error() == sg.OK
