"""The dense GEMM's tail-split plan and work units, through the library's
host-only queries (the same functions the kernel walks on the device).

Checked for many shapes and SM-pair counts: every (tile, K block) of the
GEMM is computed exactly once; every launched pair gets work; whole tiles
come before the one K range a pair may take; slabs are distinct, one per
split range, and fit the workspace; a split happens only for a last wave of
at most half the pairs with at least 16 K blocks; ranges of one tile cover
its K blocks in slab order.
"""
import itertools

import pytest


@pytest.fixture(scope="module")
def fb():
    from fp8_fine_grained_16_b300 import build
    build.build()
    from fp8_fine_grained_16_b300 import fp8bs
    return fp8bs


SLAB = 256 * 256 * 4          # one pair tile of fp32 partial sums: what the workspace size counts per pair
FORMS = [0, 1]                # FP8_GEMM_FORM_DENSE, FP8_GEMM_FORM_Q8


def _slab(fb, form):
    return 256 * fb.fp8_gemm_tile_cols(form) * 4


def _walk(fb, M, N, K, pairs, ws_bytes, form=0):
    split, tail0, np_ = fb.fp8_gemm_split_plan(M, N, K, pairs, ws_bytes, form)
    bn = fb.fp8_gemm_tile_cols(form)
    num_tiles = ((M + 255) // 256) * ((N + bn - 1) // bn)
    nkb = K // 128
    seen = {}
    slabs = {}
    for c in range(np_):
        units = fb.fp8_gemm_split_units(M, N, K, pairs, ws_bytes, c, form)
        assert units, "pair %d has no work" % c
        for i, (w, kb0, kb1, slab) in enumerate(units):
            assert 0 <= w < num_tiles and 0 <= kb0 < kb1 <= nkb
            if slab < 0:
                assert (kb0, kb1) == (0, nkb) and (split == 0 or w < tail0)
            else:
                assert i == len(units) - 1, "the K range comes after the whole tiles"
                assert w >= tail0 and slab not in slabs
                slabs[slab] = (w, kb0, kb1)
            for kb in range(kb0, kb1):
                assert (w, kb) not in seen, "tile %d K block %d computed twice" % (w, kb)
                seen[(w, kb)] = slab
    assert len(seen) == num_tiles * nkb
    return split, tail0, np_, slabs, num_tiles, nkb


@pytest.mark.parametrize("M,N,K", [(4096, 7168, 7168), (4096, 7168, 2048), (7168, 7168, 8192), (2048, 4096, 8192),
                                   (256, 256, 2048), (300, 384, 4096), (1, 256, 2048), (513, 768, 2048),
                                   (640, 1280, 4096), (4096, 7168, 1024), (128, 256, 128), (10240, 256, 4096),
                                   (4096, 2048, 7168), (5000, 5120, 3072)])
@pytest.mark.parametrize("pairs", [74, 72, 70, 66, 8, 1])
@pytest.mark.parametrize("form", FORMS)
def test_every_k_block_once_and_every_pair_busy(fb, M, N, K, pairs, form):
    ws = pairs * SLAB
    split, tail0, np_, slabs, num_tiles, nkb = _walk(fb, M, N, K, pairs, ws, form)
    assert np_ <= pairs
    tail = num_tiles % pairs
    if split:
        assert nkb >= 16 and 0 < tail and 2 * tail <= pairs and tail0 == num_tiles - tail
        assert 2 <= split <= min(pairs // tail, nkb // 2)
        assert sorted(slabs) == list(range(tail * split))
        # slab j * split + s holds range s of tail tile j; the ranges of a tile run in K order
        for j in range(tail):
            ranges = [slabs[j * split + s] for s in range(split)]
            assert all(r[0] == tail0 + j for r in ranges)
            assert [r[1] for r in ranges] == sorted(r[1] for r in ranges)
            assert ranges[0][1] == 0 and ranges[-1][2] == nkb
            assert all(ranges[s][2] == ranges[s + 1][1] for s in range(split - 1))
    else:
        assert not slabs
        if nkb >= 16 and 0 < tail and 2 * tail <= pairs:
            pytest.fail("a splittable last wave was not split")


def test_tile_widths(fb):
    # every form runs 256-column tiles (two 256-column TMEM accumulators)
    assert [fb.fp8_gemm_tile_cols(f) for f in (0, 1, 2)] == [256, 256, 256]
    assert fb.lib.fp8_gemm_tile_cols(3) == -1


def test_known_plans(fb):
    for form in FORMS:
        # the dense-linear GEMM on 74 pairs: 448 tiles, last wave of 4 cut into 18 ranges
        assert fb.fp8_gemm_split_plan(4096, 7168, 7168, 74, 74 * SLAB, form) == (18, 444, 74)
        # Wgrad: 784 tiles leave 44 on 74 pairs, more than half: whole tiles only
        assert fb.fp8_gemm_split_plan(7168, 7168, 8192, 74, 74 * SLAB, form) == (0, 784, 74)
        # one tile, 16 K blocks: 8 ranges of 2, 8 pairs launched
        assert fb.fp8_gemm_split_plan(256, 256, 2048, 74, 74 * SLAB, form) == (8, 0, 8)
        # no workspace, or too short a K: no split, one pair per tile at most
        assert fb.fp8_gemm_split_plan(4096, 7168, 7168, 74, 0, form) == (0, 448, 74)
        assert fb.fp8_gemm_split_plan(256, 256, 1024, 74, 74 * SLAB, form) == (0, 1, 1)


def test_small_workspace_disables_the_split(fb):
    # 4 tail tiles x 18 ranges need 72 slabs; 71 do not fit
    assert fb.fp8_gemm_split_plan(4096, 7168, 7168, 74, 71 * SLAB)[0] == 0
    assert fb.fp8_gemm_split_plan(4096, 7168, 7168, 74, 72 * SLAB)[0] == 18


def test_plan_argument_errors(fb):
    L = fb.lib
    assert L.fp8_gemm_split_plan(0, 0, 256, 256, 74, 0, None, None, None) == -1
    import ctypes
    out = (ctypes.c_int64 * 3)()
    p = ctypes.addressof(out)
    assert L.fp8_gemm_split_plan(0, 256, 200, 256, 74, 0, p, p + 8, p + 16) == -2
    assert L.fp8_gemm_split_plan(0, 256, 256, 256, 0, 0, p, p + 8, p + 16) == -1
    assert L.fp8_gemm_split_plan(2, 256, 256, 2048, 74, 0, p, p + 8, p + 16) == -1    # grouped: no split
    assert L.fp8_gemm_split_plan(7, 256, 256, 2048, 74, 0, p, p + 8, p + 16) == -1    # unknown form
    assert L.fp8_gemm_split_units(0, 256, 256, 2048, 74, 74 * SLAB, 8, None, 0) == -1    # pair beyond the launch
