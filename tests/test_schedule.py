"""Host checks of the tensor-core GEMM's work schedule (sgemm_plan_units): whatever the
mix of whole tiles, reduction-split parts and recut last-round pieces, every element of C
is computed exactly once over the whole reduction, the pieces are MMA-legal, and no pair
gets more work than the schedule's round count allows."""

import numpy as np
import pytest

import dense_fp32_gemm_sgemm_gb300 as sg


def coverage(M, N, K, sm_count=0, mode=sg.MODE_FP32):
    units = sg.plan_units(M, N, K, mode, sm_count)
    # a block holds 32 reduction elements (TF32 planes) or 64 (FP16 planes)
    kblocks = (N + 63) // 64 if mode == sg.MODE_3XFP16_SCALED else (N + 31) // 32
    # whole-reduction units count once per element; split parts add their block counts
    cover = np.zeros((M, K), dtype=np.int32)
    for row0, col0, cols, kb0, kb1, slot in units:
        assert 0 <= kb0 < kb1 <= kblocks
        # 1xTF32 takes 256 x 512 tiles on long products
        widest = 512 if mode == sg.MODE_TF32 else 256
        assert 32 <= cols <= widest and cols % 32 == 0, "pieces are multiples of 32 columns"
        assert row0 % 256 == 0 and 0 <= row0 < M and 0 <= col0 < K and col0 % 32 == 0
        if slot < 0:
            assert (kb0, kb1) == (0, kblocks), "a unit that writes C takes the whole reduction"
            cover[row0:row0 + 256, col0:col0 + cols] += kblocks
        else:
            # split parts are whole tiles (256 x 256, or 1xTF32's 256 x 512 in its tail)
            assert cols in (256, widest) and col0 % cols == 0, "split parts are whole tiles"
            cover[row0:row0 + 256, col0:col0 + cols] += kb1 - kb0
    return units, cover, kblocks


SHAPES = [(8192, 6144, 4096), (4096, 4096, 4096), (8192, 8192, 8192), (8191, 6143, 4097),
          (2048, 512, 8192), (4000, 1000, 4000), (1000, 333, 777), (7000, 4096, 4096),
          (6144, 4096, 4096), (8192, 64, 8192), (256, 8192, 256), (257, 129, 8192),
          (1, 8192, 8192), (8192, 8192, 1), (5000, 3000, 2500)]


@pytest.mark.parametrize("mode", [sg.MODE_FP32, sg.MODE_TF32, sg.MODE_3XFP16_SCALED],
                         ids=["3xtf32", "tf32", "3xfp16"])
@pytest.mark.parametrize("shape", SHAPES, ids=["x".join(map(str, s)) for s in SHAPES])
def test_every_element_once(shape, mode):
    units, cover, kblocks = coverage(*shape, mode=mode)
    assert np.all(cover == kblocks)


def test_random_shapes_and_sm_counts():
    rng = np.random.default_rng(5)
    for _ in range(150):
        M, N, K = (int(np.exp(rng.uniform(0, np.log(8192)))) for _ in range(3))
        sm = int(rng.choice([2, 16, 64, 132, 148, 152, 160, 264]))
        mode = int(rng.choice([sg.MODE_FP32, sg.MODE_TF32, sg.MODE_3XFP16_SCALED]))
        _, cover, kblocks = coverage(M, N, K, sm, mode)
        assert np.all(cover == kblocks), (M, N, K, sm)


def test_recut_balances_the_last_round():
    """Recut last rounds: 8192x8192x1024 on 76 pairs leaves 52 tiles for a second round,
    recut into 76 pieces of at most 192 columns; 2048x512x8192 (a short reduction) leaves
    28, recut into 76 pieces of at most 96. One piece per pair, right after the whole
    rounds."""
    for shape, widest in [((8192, 8192, 1024), 192), ((2048, 512, 8192), 96)]:
        units = sg.plan_units(*shape, sg.MODE_FP32, 152)
        full = [u for u in units if u[2] == 256]
        pieces = [u for u in units if u[2] != 256]
        assert len(full) % 76 == 0 and 0 < len(pieces) <= 76
        assert max(u[2] for u in pieces) == widest
        assert units[len(full):] == pieces


def test_split_tail_is_part_major():
    """A last round split along the reduction (4096^3: 28 tiles, 5 parts) lists all tiles'
    first parts, then all second parts, and so on, so that the pairs work in one reduction
    range at a time; the parts of a tile cover its reduction exactly once."""
    units = sg.plan_units(4096, 4096, 4096, sg.MODE_FP32, 152)
    parts = [u for u in units if u[5] >= 0]
    assert parts and all(u[2] == 256 for u in parts)
    starts = [u[3] for u in parts]
    assert starts == sorted(starts), "parts are not in reduction order"
    tiles = {(u[0], u[1]) for u in parts}
    assert len(tiles) == 28 and len(parts) == 28 * 5
    kblocks = 4096 // 32
    for t in tiles:
        ranges = sorted((u[3], u[4]) for u in parts if (u[0], u[1]) == t)
        assert ranges[0][0] == 0 and ranges[-1][1] == kblocks
        assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))


def test_schedule_query_rejects_bad_arguments():
    L = sg.lib()
    assert L.sgemm_plan_units(0, 1, 1, 0, 0, None, 0) == sg.ERR_ARG
    assert L.sgemm_plan_units(1, 1, 8193, 0, 0, None, 0) == sg.ERR_ARG
    assert L.sgemm_plan_units(1, 1, 1, 5, 0, None, 0) == sg.ERR_ARG
    assert L.sgemm_plan_units(1, 1, 1, 0, -1, None, 0) == sg.ERR_ARG
    assert L.sgemm_plan_units(1, 1, 1, 0, 0, None, 1) == sg.ERR_ARG
    # 2 x 2 tiles for 76 pairs: each split in two (10 reduction blocks, at least 4 a part)
    assert L.sgemm_plan_units(300, 300, 300, 0, 0, None, 0) == 8
