"""GPU parity of SwiGLU fused with 1x128 quantisation (the MoE down-projection
input; the DeepSeek-V3 FP8 training pages fix its scaling factors to
integral powers of 2).

Two checks.  The independent one holds the GPU's codes and scales to the
plain definition: h = g / (1 + e^-g) * u in float64 with libm's exp, rounded
once to fp32, then the oracle's pinned fp32 1x128 tile rule; they must match
bit for bit except neighbouring codes (or powers of two) where h sits within
the fp32 slack of a rounding midpoint (or scale boundary), and those must be
few.  The consistency check holds them bit for bit to the oracle's fused
quantiser, which forms h in the same fp32 steps as the kernel (e^x by
Cody-Waite reduction and a degree-7 Taylor polynomial, written separately on
each side).
"""
import numpy as np
import pytest
import torch

from fp8_fine_grained_16_b300 import synthetic as S
from _checks import assert_same_bits, check_swiglu_quant_against_fp64

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


@pytest.mark.parametrize("flags", [1, 0])
@pytest.mark.parametrize("R,I,pad,scale", [(300, 2048, 0, 3.0), (33, 640, 24, 1.0), (2048, 1024, 8, 8.0)])
def test_swiglu_quant_against_fp64_definition(fb, orc, R, I, pad, scale, flags):
    y = _bf16((R, 2 * I + pad), 7 * R + I + pad, scale)
    q, s = fb.fp8_swiglu_quant_1x128(y.cuda(), I, flags=flags)
    torch.cuda.synchronize()
    n_mid, n_scale = check_swiglu_quant_against_fp64(q.cpu().numpy(), s.cpu().numpy(), y, I, flags, orc)
    print("R%d I%d flags%d: %d codes at a midpoint of %d, %d of %d tiles with another scale"
          % (R, I, flags, n_mid, q.numel(), n_scale, s.numel()))
    assert n_mid <= 1e-4 * q.numel() + 2
    if flags & 1:
        assert n_scale <= 1e-3 * s.numel() + 1


def test_swiglu_quant_extremes_against_fp64_definition(fb, orc):
    """Saturated and vanishing gates, zero tiles and outliers against the
    float64 definition (pow-2 and default)."""
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
    for flags in (1, 0):
        q, s = fb.fp8_swiglu_quant_1x128(y.cuda(), I, flags=flags)
        torch.cuda.synchronize()
        n_mid, n_scale = check_swiglu_quant_against_fp64(q.cpu().numpy(), s.cpu().numpy(), y, I, flags, orc)
        assert n_mid <= 2
        if flags & 1:
            assert n_scale <= 1


def test_reciprocal_matches_frcp_rn_for_every_d_from_one(fb):
    """The kernel's sigma = 1/d (Markstein's correction of the hardware
    approximation) equals __frcp_rn bit for bit for every float d >= 1, +inf
    and every NaN pattern: all 2^30 + 2^23 bit patterns from 0x3F800000."""
    assert fb.fp8_selftest_reciprocal(0x3F800000, 0x7FFFFFFF) == 0


def test_swiglu_quant_gates_at_the_range_boundary_bit_exact(fb, orc):
    """Gates at |g| = 87 (the largest value the in-range steps take), the next
    bf16 values past it (87.5, 88, 88.5) and NaN-free extremes, scattered so
    that some lanes' 8 gates are all in range and others hold one gate just
    outside; codes and scales bit for bit against the oracle, both scale
    modes."""
    R, I = 96, 512
    y = _bf16((R, 2 * I), 31, 2.0).float()
    g = torch.Generator().manual_seed(32)
    edge = torch.tensor([87.0, -87.0, 87.5, -87.5, 88.0, -88.0, 88.5, -88.5, 86.5, -86.5])
    for r in range(R):
        n = int(torch.randint(0, 4, (1,), generator=g))        # 0..3 edge gates in this row
        cols = torch.randint(0, I, (n,), generator=g)
        vals = edge[torch.randint(0, len(edge), (n,), generator=g)]
        y[r, cols] = vals
    y[0, :8] = 87.0                                             # a lane all at the boundary
    y[1, 8:16] = -87.0
    y[2, 16:23] = 1.0
    y[2, 23] = 87.5                                             # one gate past it in a lane
    y = y.to(torch.bfloat16)
    for flags in (1, 0):
        q, s = fb.fp8_swiglu_quant_1x128(y.cuda(), I, flags=flags)
        torch.cuda.synchronize()
        q_ref, s_ref = orc.swiglu_quant_1x128(S.bf16_bits(y), I, flags)
        assert_same_bits(q, q_ref, "boundary codes flags%d" % flags)
        assert_same_bits(s, s_ref, "boundary scales flags%d" % flags)
