"""Pins for the oracle's quantisers (the jp-study.kr page: max-abs taken online per 1x128
activation tile and per 128x128 weight block; the tmdrlife.com and gnrental.net pages: integral power-of-2
scales for some activations; the jp-study.kr page: Wgrad runs in FP8, which needs 128x1
tiles along tokens)."""
import math
import os

import numpy as np
import pytest
import torch

from fp8_fine_grained_16_b300 import synthetic as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_tiles_1x128.txt")


def _bits(t):
    return S.bf16_bits(t)


def _rand_bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def _load_golden():
    tiles = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        f = line.split()
        if f[0] == "tile":
            tiles.append(dict(name=f[1], pow2=f[2] == "pow2", scale=float.fromhex(f[3]), xs=[]))
        else:
            tiles[-1]["xs"].append((int(f[1]), float.fromhex(f[2]), int(f[3], 16)))
    return tiles


@pytest.mark.parametrize("tile", _load_golden(), ids=lambda t: t["name"] + ("-pow2" if t["pow2"] else ""))
def test_worked_tiles(orc, tile):
    x = torch.zeros((1, 128), dtype=torch.float32)
    for i, v, _ in tile["xs"]:
        x[0, i] = v
    xb = x.to(torch.bfloat16)
    assert torch.equal(xb.float(), x)            # fixture values are bf16-exact
    q, s = orc.quant_act_1x128(_bits(xb), flags=1 if tile["pow2"] else 0)
    assert s[0, 0] == np.float32(tile["scale"])
    expect = np.zeros(128, np.uint8)
    for i, _, c in tile["xs"]:
        expect[i] = c
    assert np.array_equal(q[0], expect)


def _decode(orc, q):
    table = orc.e4m3_decode(np.arange(256))
    return table[q]


@pytest.mark.parametrize("pow2", [False, True])
def test_amax_maps_to_448(orc, pow2):
    d = S.tiny_dense()
    xb = _bits(d["x"])
    q, s = orc.quant_act_1x128(xb, flags=int(pow2))
    x = d["x"].float().numpy()
    v = _decode(orc, q)
    M, K = x.shape
    for m in range(M):
        for kb in range(K // 128):
            t = x[m, kb * 128:(kb + 1) * 128]
            qt = v[m, kb * 128:(kb + 1) * 128]
            i = int(np.argmax(np.abs(t)))
            if not pow2:
                assert abs(qt[i]) == 448.0 and math.copysign(1, qt[i]) == math.copysign(1, t[i])
            else:
                sc = float(s[kb, m])
                assert math.frexp(sc)[0] == 0.5                       # exact power of two
                assert 448.0 * sc >= abs(t[i]) > 224.0 * sc           # smallest such power
                assert 224.0 <= np.abs(qt).max() <= 448.0


@pytest.mark.parametrize("pow2", [False, True])
def test_dequant_error_bound(orc, pow2):
    """|x - q*s| <= max(|x| 2^-4, s 2^-10) + |x| 2^-20 for every element."""
    xt = torch.cat([_rand_bf16((64, 1024), 3), _rand_bf16((64, 1024), 4, 1e-3),
                    S.dense_linear(M=64, N=128, K=1024)["x"]])
    q, s = orc.quant_act_1x128(_bits(xt), flags=int(pow2))
    x = xt.double().numpy()
    sc = np.repeat(s.T.astype(np.float64), 128, axis=1)
    err = np.abs(x - _decode(orc, q) * sc)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, sc * 2.0 ** -10) + np.abs(x) * 2.0 ** -20
    assert np.all(err <= bound)


def test_tile_locality_outlier_columns(orc):
    """The x100 outlier columns change only the tiles that contain them."""
    g = torch.Generator().manual_seed(0)
    base = torch.randn((128, 512), generator=g)
    out = base.clone()
    out[:, 5] *= 100
    out[:, 260] *= 100
    qa, sa = orc.quant_act_1x128(_bits(base.to(torch.bfloat16)))
    qb, sb = orc.quant_act_1x128(_bits(out.to(torch.bfloat16)))
    touched = {0, 2}
    for kb in range(4):
        same = np.array_equal(sa[kb], sb[kb]) and np.array_equal(qa[:, kb * 128:(kb + 1) * 128],
                                                                 qb[:, kb * 128:(kb + 1) * 128])
        assert same == (kb not in touched)


@pytest.mark.parametrize("pow2", [False, True])
def test_128x1_is_1x128_of_transpose(orc, pow2):
    x = _rand_bf16((384, 200), 11)
    qT, s = orc.quant_act_128x1(_bits(x), flags=int(pow2))
    q2, s2 = orc.quant_act_1x128(_bits(x.t().contiguous()), flags=int(pow2))
    assert np.array_equal(qT, q2) and np.array_equal(s, s2)


@pytest.mark.parametrize("pow2", [False, True])
def test_weight_block_scale_is_block_amax(orc, pow2):
    w = _rand_bf16((256, 384), 5, 0.02)
    w[100, 300] = 3.0
    q, s = orc.quant_weight_128x128(_bits(w), flags=int(pow2))
    wf = w.float().numpy()
    for nb in range(2):
        for kb in range(3):
            blk = wf[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            want, _ = orc.tile_scale(float(np.abs(blk).max()), int(pow2))
            assert s[nb, kb] == want
    # the block holding the 3.0 maps it to 448 in default mode
    if not pow2:
        assert q[100, 300] == 0x7E


def test_zero_tile_is_finite(orc):
    x = torch.zeros((2, 256), dtype=torch.bfloat16)
    x[1, 200] = -1.0
    q, s = orc.quant_act_1x128(_bits(x))
    assert np.all(np.isfinite(s)) and s[0, 0] == np.float32(2.0 ** -64 / 448)
    assert np.all(q[0] == 0) and q[1, 200] == 0xFE


def test_weight_quant_of_transpose_is_transpose_of_quant(orc):
    """A 128x128 block's max-abs does not change under transposition, so the
    block quantisation of W^T is the transpose of W's codes and block scales
    (what FP8 Dgrad relies on)."""
    g = np.random.default_rng(21)
    w = (g.standard_normal((384, 256)) * 0.02).astype(np.float32)
    w[7, 200] = 3.0                                   # one block with an outlier
    wb = (w.view(np.uint32) >> 16).astype(np.uint16)  # truncate to bf16 bits
    for flags in (0, 1):
        q, s = orc.quant_weight_128x128(wb, flags)
        qt, st = orc.quant_weight_128x128(np.ascontiguousarray(wb.T), flags)
        assert np.array_equal(qt, q.T)
        assert np.array_equal(st.view(np.uint32), s.T.view(np.uint32))


# ---- the 1x128 tile rule on fp32 values (the quantising GEMM epilogue)
@pytest.mark.parametrize("flags", [0, 1])
def test_f32_tile_quant_equals_bf16_tile_quant_on_bf16_values(orc, flags):
    """On values that bf16 represents exactly the fp32 form must give the
    pinned bf16 quantiser's codes and scales bit for bit."""
    x = _rand_bf16((37, 512), 11, scale=3.0)
    q1, s1 = orc.quant_act_1x128(_bits(x), flags)
    q2, s2 = orc.quant_act_1x128_f32(x.float().numpy(), flags)
    assert np.array_equal(q1, q2)
    assert np.array_equal(s1.view(np.uint32), s2.view(np.uint32))


def _e4m3_table(orc):
    return orc.e4m3_decode(np.arange(256, dtype=np.uint8))


@pytest.mark.parametrize("flags", [0, 1])
def test_f32_tile_quant_follows_the_tile_rule(orc, flags):
    """fp32 values that are not bf16 values, over ~60 binades: (default) each
    tile's max-abs element codes to +-448; (pow2) the scale is a power of two
    with 224*s < amax <= 448*s; every element dequantises within half an E4M3
    step (2^-4 relative for normals, 2^-10 * s absolute for subnormals)."""
    g = np.random.default_rng(3)
    x = (g.standard_t(3, size=(64, 384)) * np.exp(g.uniform(-20, 20, size=(64, 1)))).astype(np.float32)
    q, s = orc.quant_act_1x128_f32(x, flags)
    tab = _e4m3_table(orc)
    st = np.repeat(s.T.astype(np.float64), 128, axis=1)          # [M, K]: the scale of each element's tile
    deq = tab[q] * st
    xt = x.reshape(64, 3, 128)
    amax = np.abs(xt).max(axis=2)                                 # [M, K/128]
    if flags == 0:
        arg = np.abs(xt).argmax(axis=2)
        codes = np.take_along_axis(q.reshape(64, 3, 128), arg[..., None], axis=2)[..., 0]
        assert np.all((codes == 0x7E) | (codes == 0xFE))
    else:
        sm = s.T.astype(np.float64)
        m, e = np.frexp(sm)
        assert np.all(m == 0.5)
        assert np.all(224.0 * sm < amax) and np.all(amax <= 448.0 * sm)
    err = np.abs(deq - x.astype(np.float64))
    bound = 2.0 ** -4 * np.abs(x.astype(np.float64)) * (1 + 1e-6) + 2.0 ** -10 * st
    assert np.all(err <= bound)


def _dequant_bound(x, deq, sc):
    err = np.abs(x - deq)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, sc * 2.0 ** -10) + np.abs(x) * 2.0 ** -20
    return err <= bound


@pytest.mark.parametrize("pow2", [False, True])
def test_weight_dequant_error_bound_every_element(orc, pow2):
    """Every code of the 128x128 quantiser dequantises within half an E4M3
    step with its own block's scale.  The 3 x 2 blocks differ in magnitude by
    up to 10^10, so a code formed with another block's reciprocal (a
    transposed or shifted block index) breaks the bound by orders of
    magnitude; one block is all zero, one holds a lone outlier."""
    g = torch.Generator().manual_seed(17)
    w = torch.randn((384, 256), generator=g)
    mags = [[1e-6, 3e2], [0.02, 0.0], [7.0, 1e4]]
    for nb in range(3):
        for kb in range(2):
            w[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128] *= mags[nb][kb]
    w[200, 30] = 55.0                          # outlier in block (1, 0)
    wb = w.to(torch.bfloat16)
    q, s = orc.quant_weight_128x128(_bits(wb), flags=int(pow2))
    x = wb.double().numpy()
    sc = np.repeat(np.repeat(s.astype(np.float64), 128, axis=0), 128, axis=1)
    assert np.all(_dequant_bound(x, _decode(orc, q) * sc, sc))
    # each block's own amax codes to +-448 in default mode (and only there)
    if not pow2:
        for nb in range(3):
            for kb in range(2):
                blk = x[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
                if np.abs(blk).max() == 0:
                    # zeros keep their sign: +0 -> 0x00, -0 -> 0x80
                    assert np.all((q[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128] & 0x7F) == 0)
                    continue
                i, j = np.unravel_index(np.argmax(np.abs(blk)), blk.shape)
                assert q[nb * 128 + i, kb * 128 + j] in (0x7E, 0xFE)


@pytest.mark.parametrize("pow2", [False, True])
def test_128x1_dequant_error_bound_every_element(orc, pow2):
    """The same bound for the token-direction quantiser, which writes its
    codes transposed: qT[h, t] dequantised with s[t / 128, h] must be within
    half an E4M3 step of x[t, h].  Columns and token blocks differ in
    magnitude (a code scaled by a neighbouring column's or token block's
    scale breaks the bound), and one column is zero in one token block."""
    g = torch.Generator().manual_seed(23)
    T, H = 384, 96
    x = torch.randn((T, H), generator=g)
    x *= torch.logspace(-4, 4, H).reshape(1, H)
    x *= torch.tensor([1.0, 1e-5, 3e3]).repeat_interleave(128).reshape(T, 1)
    x[128:256, 40] = 0.0
    xb = x.to(torch.bfloat16)
    qT, s = orc.quant_act_128x1(_bits(xb), flags=int(pow2))
    xv = xb.double().numpy()
    sc = np.repeat(s.astype(np.float64), 128, axis=0)          # [T, H]: the scale of each element's tile
    deq = _decode(orc, qT).T * sc
    assert np.all(_dequant_bound(xv, deq, sc))
    if not pow2:
        for tb in range(3):
            blk = np.abs(xv[tb * 128:(tb + 1) * 128])
            for h in range(H):
                if blk[:, h].max() > 0:
                    assert qT[h, tb * 128 + int(np.argmax(blk[:, h]))] in (0x7E, 0xFE)
