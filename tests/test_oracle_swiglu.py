"""Pins for the oracle's SwiGLU + 1x128 quantisation (the MoE down-projection
input; the tmdrlife.com page fixes that activation's scales to integral powers of 2).

SwiGLU(g, u) = SiLU(g) * u with SiLU(g) = g / (1 + e^-g).  The oracle forms
it in fp32 steps with its own e^x (Cody-Waite reduction, degree-7 Taylor), so
that a GPU kernel doing the same fp32 steps can be held to identical codes.
These tests pin those fp32 steps to the mathematics: e^x and SwiGLU against
float64 library evaluations, the special values, and the quantiser's tile
rule applied to the pinned fp32 SwiGLU.
"""
import numpy as np
import pytest
import torch

from fp8_fine_grained_16_b300 import synthetic as S


def _ulp32(v):
    v = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -126)))
    return 2.0 ** (e - 23)


def test_exp_matches_float64_exp_within_2_ulp(orc):
    g = np.random.default_rng(1)
    x = np.concatenate([g.uniform(-87.0, 88.0, 40000), g.uniform(-1.0, 1.0, 10000),
                        np.array([0.0, -0.0, 1.0, -1.0, 0.5, 88.0, -87.0, 1e-8, -1e-8])]).astype(np.float32)
    got = orc.exp_cw(x).astype(np.float64)
    want = np.exp(x.astype(np.float64))
    err_ulps = np.abs(got - want) / _ulp32(want)
    print("exp max error %.3f ulp" % err_ulps.max())
    assert err_ulps.max() <= 2.0


def test_exp_special_values(orc):
    assert orc.exp_cw(np.array([0.0], np.float32))[0] == 1.0
    assert np.isinf(orc.exp_cw(np.array([88.5, 1000.0], np.float32))).all()
    assert (orc.exp_cw(np.array([-87.5, -1000.0], np.float32)) == 0.0).all()
    x = np.linspace(-87.0, 88.0, 20001, dtype=np.float32)
    e = orc.exp_cw(x)
    assert np.all(np.diff(e.astype(np.float64)) >= 0.0)           # non-decreasing


def _bf16(shape, seed, scale):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def test_swiglu_matches_float64_definition(orc):
    R, I = 64, 512
    y = _bf16((R, 2 * I), 2, 3.0)
    yb = S.bf16_bits(y)
    h = orc.swiglu_f32(yb, I).astype(np.float64)
    yf = y.float().numpy().astype(np.float64)
    g, u = yf[:, :I], yf[:, I:]
    want = g / (1.0 + np.exp(-g)) * u
    # five fp32 roundings plus the e^x error: a few ulp of each factor
    assert np.all(np.abs(h - want) <= 8.0 * _ulp32(want) + 1e-30)


def test_swiglu_special_values(orc):
    I = 128
    g = np.zeros((4, I), np.float32)
    u = np.full((4, I), 1.5, np.float32)
    g[1] = 100.0            # sigma = 1: SiLU(g) = g
    g[2] = -100.0           # e^100 overflows: sigma = 0, SiLU(g) = -0
    g[3] = 1e-3
    y = torch.from_numpy(np.concatenate([g, u], axis=1)).to(torch.bfloat16)
    h = orc.swiglu_f32(S.bf16_bits(y), I)
    gb = y.float().numpy()[:, :I]
    assert np.all(h[0] == 0.0)
    assert np.all(h[1] == np.float32(gb[1] * np.float32(1.5)))
    assert np.all(h[2] == 0.0) and np.all(np.signbit(h[2]))
    assert np.allclose(h[3], gb[3] * 0.5 * 1.5, rtol=1e-3)


@pytest.mark.parametrize("flags", [0, 1])
def test_swiglu_quant_is_tile_rule_of_swiglu(orc, flags):
    R, I = 33, 384
    y = _bf16((R, 2 * I + 16), 3, 2.0)          # leading dimension wider than 2I
    yb = S.bf16_bits(y)
    q, s = orc.swiglu_quant_1x128(yb, I, flags)
    q2, s2 = orc.quant_act_1x128_f32(orc.swiglu_f32(yb, I), flags)
    assert np.array_equal(q, q2)
    assert np.array_equal(s.view(np.uint32), s2.view(np.uint32))


@pytest.mark.parametrize("flags", [1, 0])
def test_fused_quant_against_fp64_definition(orc, flags):
    """The oracle's fused SwiGLU quantiser (its own fp32 e^x recipe) held to
    the float64 definition with libm's exp followed by the pinned fp32 tile
    rule: equal codes and scales except neighbours at a rounding midpoint or
    a scale boundary, and those few."""
    import torch
    from _checks import check_swiglu_quant_against_fp64
    from fp8_fine_grained_16_b300 import synthetic as S
    y = (torch.randn((256, 2 * 1024), generator=torch.Generator().manual_seed(31)) * 3.0).to(torch.bfloat16)
    q, s = orc.swiglu_quant_1x128(S.bf16_bits(y), 1024, flags)
    n_mid, n_scale = check_swiglu_quant_against_fp64(q, s, y, 1024, flags, orc)
    print("flags%d: %d codes at a midpoint, %d tiles with another scale" % (flags, n_mid, n_scale))
    assert n_mid <= 1e-4 * q.size + 2
    if flags & 1:
        assert n_scale <= 2
