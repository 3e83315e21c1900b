"""GPU parity of the GEMM whose epilogue quantises D per 1x128 tile along N
(the tmdrlife.com page: the BF16 output of one operator is written to HBM, read back and
quantised, and read again for the next MMA; quantising it where it is formed
removes that round trip).

The codes depend on D's exact fp32 values, and the oracle never takes an
input from the GPU.  So the bit-exact test builds operands whose product is
exactly representable: codes in {0, +-0.5, +-1, +-2, +-3} and power-of-two
scales in [2^-2, 2^2].  Every partial sum is then a multiple of 2^-6 below
2^18, so the tensor core's sum, the fp32 promotion and the oracle's fp64
product all give the same number.  The fused codes and scales must then equal
the oracle's 1x128 tile rule applied to that number, bit for bit.  A second
test on general operands checks every dequantised element against the fp64
product within half an E4M3 step plus the GEMM's fp32 error.
"""
import numpy as np
import pytest
import torch

from fp8_fine_grained_16_b300 import synthetic as S
from _checks import assert_same_bits, rand_codes, rand_scales

pytestmark = pytest.mark.gpu

EXACT_CODES = np.array([0x00, 0x30, 0xB0, 0x38, 0xB8, 0x40, 0xC0, 0x44, 0xC4], dtype=np.uint8)


@pytest.fixture(scope="module")
def fb():
    from fp8_fine_grained_16_b300 import build
    build.build()
    from fp8_fine_grained_16_b300 import fp8bs
    return fp8bs


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _exact_operands(M, N, K, mode, seed):
    g = np.random.default_rng(seed)
    a = g.choice(EXACT_CODES, size=(M, K))
    b = g.choice(EXACT_CODES, size=(N, K))
    sa = np.ldexp(np.float32(1.0), g.integers(-2, 3, size=(K // 128, M))).astype(np.float32)
    sbs = (N // 128, K // 128) if mode == 0 else (K // 128, N)
    sb = np.ldexp(np.float32(1.0), g.integers(-2, 3, size=sbs)).astype(np.float32)
    return a, sa, b, sb


@pytest.mark.parametrize("flags", [0, 1])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (1, 256, 128), (300, 384, 1024), (513, 768, 512),
                                   (300, 384, 2048), (513, 768, 2048)])
def test_q8_epilogue_bit_exact_on_exactly_representable_products(fb, orc, M, N, K, mode, flags):
    # K >= 2048: the few tiles are split along K over the GPU and the fix-up
    # kernel quantises them from the sum of their K ranges
    a, sa, b, sb = _exact_operands(M, N, K, mode, 7 * M + N + K + mode)
    ref = orc.gemm_blockscaled(a, sa, b, sb, mode)
    ref32 = ref.astype(np.float32)
    assert np.array_equal(ref32.astype(np.float64), ref), "operands were meant to give an exact fp32 product"
    q_ref, s_ref = orc.quant_act_1x128_f32(ref32, flags)
    q, s = fb.fp8_gemm_blockscaled_q8(_dev(a), _dev(sa), _dev(b), _dev(sb), mode, flags)
    torch.cuda.synchronize()
    assert_same_bits(q, q_ref, "codes M%d N%d K%d mode%d flags%d" % (M, N, K, mode, flags))
    assert_same_bits(s, s_ref, "scales M%d N%d K%d mode%d flags%d" % (M, N, K, mode, flags))
    assert fb.fp8_get_status() == 0


@pytest.mark.parametrize("flags", [0, 1])
def test_q8_split_tail_bit_exact_rows(fb, orc, flags):
    """4096 x 7168 x 2048: whole tiles quantised in the GEMM's epilogue and the
    last wave's tiles split along K and quantised by the fix-up kernel; every
    7th row's codes and scales against the tile rule on the exact product."""
    M, N, K = 4096, 7168, 2048
    a, sa, b, sb = _exact_operands(M, N, K, 0, 77 + flags)
    rows = np.arange(0, M, 7)
    ref = orc.gemm_blockscaled(a, sa, b, sb, 0, rows=rows, cols=np.arange(N))
    ref32 = ref.astype(np.float32)
    assert np.array_equal(ref32.astype(np.float64), ref), "operands were meant to give an exact fp32 product"
    q_ref, s_ref = orc.quant_act_1x128_f32(ref32, flags)
    q, s = fb.fp8_gemm_blockscaled_q8(_dev(a), _dev(sa), _dev(b), _dev(sb), 0, flags)
    torch.cuda.synchronize()
    assert fb.fp8_get_status() == 0
    assert_same_bits(q[torch.from_numpy(rows).cuda()], q_ref, "codes flags%d" % flags)
    assert_same_bits(s[:, torch.from_numpy(rows).cuda()].contiguous(), s_ref, "scales flags%d" % flags)


@pytest.mark.parametrize("flags", [0, 1])
def test_q8_epilogue_dequantises_within_half_an_e4m3_step(fb, orc, flags):
    M, N, K = 512, 1024, 2048
    a, b = rand_codes((M, K), 51), rand_codes((N, K), 52)
    sa, sb = rand_scales((K // 128, M), 53), rand_scales((N // 128, K // 128), 54)
    q, s = fb.fp8_gemm_blockscaled_q8(_dev(a), _dev(sa), _dev(b), _dev(sb), 0, flags)
    ref = orc.gemm_blockscaled(a, sa, b, sb, 0)
    tab = orc.e4m3_decode(np.arange(256, dtype=np.uint8))
    st = np.repeat(s.cpu().numpy().T.astype(np.float64), 128, axis=1)
    deq = tab[q.cpu().numpy()] * st
    refmax = np.abs(ref).max()
    # half an E4M3 step of the value (normal) or of the scale (subnormal), plus
    # the fp32 GEMM error, which can move a value across a rounding boundary
    bound = 2.0 ** -4 * np.abs(ref) + 2.0 ** -10 * st + 1e-5 * refmax
    err = np.abs(deq - ref)
    print("q8 flags%d: max err/bound %.3f" % (flags, float((err / bound).max())))
    assert np.all(err <= bound)
    # the tile rule holds on the fused scales: 448 * s bounds every tile
    assert np.all(np.abs(ref).reshape(M, N // 128, 128).max(axis=2) <= 448.0 * s.cpu().numpy().T * (1 + 1e-5))
    assert fb.fp8_get_status() == 0


def test_q8_epilogue_dense_linear_sampled(fb, orc):
    """The dense-linear workload through the GPU quantisers and the fused GEMM;
    48 rows x 3 column blocks dequantised against the oracle's fp64 product."""
    d = S.dense_linear()
    x, w = d["x"], d["w"]
    qx, sx = fb.fp8_quant_act_1x128(x.cuda())
    qw, sw = fb.fp8_quant_weight_128x128(w.cuda())
    q, s = fb.fp8_gemm_blockscaled_q8(qx, sx, qw, sw)
    g = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, 4095], g.choice(4096, 46, replace=False)]))
    xb = S.bf16_bits(x)
    qa, sa = orc.quant_act_1x128(xb[rows])
    tab = orc.e4m3_decode(np.arange(256, dtype=np.uint8))
    qn, sn = q.cpu().numpy()[rows], s.cpu().numpy()[:, rows]
    for nb in sorted({0, 55, int(g.integers(1, 55))}):
        wb = S.bf16_bits(w[nb * 128:(nb + 1) * 128])
        qb, sbb = orc.quant_weight_128x128(wb)
        ref = orc.gemm_blockscaled(qa, sa, qb, sbb, 0)
        deq = tab[qn[:, nb * 128:(nb + 1) * 128]] * sn[nb][:, None].astype(np.float64)
        bound = 2.0 ** -4 * np.abs(ref) + 2.0 ** -10 * sn[nb][:, None] + 1e-5 * np.abs(ref).max()
        assert np.all(np.abs(deq - ref) <= bound), "block %d" % nb
    assert fb.fp8_get_status() == 0
