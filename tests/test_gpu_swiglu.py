"""GPU parity of SwiGLU fused with 1x128 quantisation (the MoE down-projection
input; page 2: its scaling factors are integral powers of 2) against the
oracle: codes and scales bit for bit.  Both sides form h = SiLU(g) * u in the
same fp32 steps (e^x by Cody-Waite reduction and a degree-7 Taylor
polynomial, written separately on each side), then apply the 1x128 tile rule.
"""
import numpy as np
import pytest
import torch

from fp8_fine_grained_16_b300 import synthetic as S
from _checks import assert_same_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fb():
    from fp8_fine_grained_16_b300 import build
    build.build()
    from fp8_fine_grained_16_b300 import fp8bs
    return fp8bs


def _bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


@pytest.mark.parametrize("flags", [1, 0])
@pytest.mark.parametrize("R,I,pad", [(1, 128, 0), (7, 384, 0), (300, 2048, 0), (33, 640, 24), (1000, 256, 8)])
def test_swiglu_quant_bit_exact(fb, orc, R, I, pad, flags):
    y = _bf16((R, 2 * I + pad), R + I + pad, 3.0)
    q, s = fb.fp8_swiglu_quant_1x128(y.cuda(), I, flags=flags)
    torch.cuda.synchronize()
    q_ref, s_ref = orc.swiglu_quant_1x128(S.bf16_bits(y), I, flags)
    assert_same_bits(q, q_ref, "codes R%d I%d pad%d flags%d" % (R, I, pad, flags))
    assert_same_bits(s, s_ref, "scales R%d I%d pad%d flags%d" % (R, I, pad, flags))


def test_swiglu_quant_extremes_bit_exact(fb, orc):
    """Gates far past e^x's range (+-100: sigma exactly 1 or 0, the latter giving
    signed zeros), tiny gates, zero tiles and outliers."""
    R, I = 64, 256
    y = _bf16((R, 2 * I), 9, 1.0).float()
    y[0, :I] = 100.0
    y[1, :I] = -100.0
    y[2, :I] = 1e-30
    y[3, :] = 0.0
    y[4, 5] = 60.0
    y[5, I + 7] = -3e4
    y[6, :I] = torch.linspace(-95.0, 95.0, I)
    y = y.to(torch.bfloat16)
    for flags in (0, 1):
        q, s = fb.fp8_swiglu_quant_1x128(y.cuda(), I, flags=flags)
        torch.cuda.synchronize()
        q_ref, s_ref = orc.swiglu_quant_1x128(S.bf16_bits(y), I, flags)
        assert_same_bits(q, q_ref, "extreme codes flags%d" % flags)
        assert_same_bits(s, s_ref, "extreme scales flags%d" % flags)


def test_swiglu_quant_moe_down_full_size_sampled(fb, orc):
    """32768 rows x (2 x 2048): the up-projection output of the MoE workload
    (256 experts, top-8 of 4096 tokens); 512 sampled rows bit for bit."""
    g = torch.Generator().manual_seed(1)
    y = torch.randn((32768, 4096), generator=g).to(torch.bfloat16)
    q, s = fb.fp8_swiglu_quant_1x128(y.cuda(), 2048)
    rows = np.sort(np.random.default_rng(2).choice(32768, 512, replace=False))
    q_ref, s_ref = orc.swiglu_quant_1x128(S.bf16_bits(y[torch.from_numpy(rows)]), 2048, 1)
    assert_same_bits(q[torch.from_numpy(rows).cuda()], q_ref, "full-size codes")
    assert_same_bits(s[:, torch.from_numpy(rows).cuda()].contiguous(), s_ref, "full-size scales")
