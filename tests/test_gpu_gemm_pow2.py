"""GPU parity of the power-of-two block-scaled GEMM (scales applied by the
tensor core as UE8M0 microscaling factors) against the oracle's fp64 product
of the same E4M3 operands and scales.

The tmdrlife.com page fixes some activation scales to integral powers of 2
and asks for tensor cores that accept the scaling factors; the gnrental.net page
(gnrental.net) ties the fine-grained tiles to the microscaling formats of
Blackwell tensor cores.  With power-of-two scales the block-promoted sum of
the pages and the microscaled sum are the same real number before rounding,
so the tolerance of the other GEMM applies unchanged.  An element-wise bound
holds as well.  How the tensor core orders and rounds the 32 products inside
one MMA is not documented (a probe shows at least 21 bits survive), so the
bound is the one for summing the K products in any order, each addition off
by at most one ulp (2^-23 relative, any rounding mode), followed by the K/32
fp32 additions into the accumulator:
    |D - ref| <= 2 * (K + K/32) * 2^-24 * sum_k |a_k b_k|
plus one bf16 rounding for bf16 outputs.  A K block taken from the wrong
stage, scale slot or accumulator is off by far more.
"""
import numpy as np
import pytest
import torch

from fp8_fine_grained_16_b300 import synthetic as S
from _checks import assert_gemm_close, rand_codes, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fb():
    from fp8_fine_grained_16_b300 import build
    build.build()
    from fp8_fine_grained_16_b300 import fp8bs
    return fp8bs


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def rand_pow2_scales(shape, seed, lo=-12, hi=4):
    g = np.random.default_rng(seed)
    return np.ldexp(np.float32(1.0), g.integers(lo, hi + 1, size=shape)).astype(np.float32)


def _abs_codes(c):
    return (c & 0x7F).astype(np.uint8)


def _elementwise_bound(orc, a, sa, b, sb, mode, K, bf16_out, ref, rows=None, cols=None):
    absref = orc.gemm_blockscaled(_abs_codes(a), sa, _abs_codes(b), sb, mode, rows=rows, cols=cols)
    bound = 2 * (K + K // 32) * 2.0 ** -24 * absref
    if bf16_out:
        bound = bound + np.abs(ref) * 2.0 ** -8
    return bound


def _check_elementwise(got, ref, bound, what):
    err = np.abs(got - ref)
    n_bad = int((err > bound).sum())
    print("%s: max err/bound %.3f" % (what, float((err / np.maximum(bound, 1e-300)).max()) if err.size else 0.0))
    assert n_bad == 0, "%s: %d elements beyond the element-wise bound" % (what, n_bad)


def _run_random(fb, orc, M, N, K, mode, out_dtype, seed):
    a, b = rand_codes((M, K), seed), rand_codes((N, K), seed + 1)
    sa = rand_pow2_scales((K // 128, M), seed + 2)
    sb = rand_pow2_scales((N // 128, K // 128) if mode == 0 else (K // 128, N), seed + 3)
    d = fb.fp8_gemm_blockscaled_pow2(_dev(a), _dev(sa), _dev(b), _dev(sb), mode, out_dtype)
    ref = orc.gemm_blockscaled(a, sa, b, sb, mode)
    bf16 = out_dtype == torch.bfloat16
    what = "pow2 M%d N%d K%d mode%d" % (M, N, K, mode)
    got = to_np(d)
    assert_gemm_close(got, ref, bf16, orc, what)
    _check_elementwise(got, ref, _elementwise_bound(orc, a, sa, b, sb, mode, K, bf16, ref), what)
    assert fb.fp8_get_status() == 0


# N = 384 and 1280 end in a partial 224-column tile; M = 1, 127, 129, 300 end
# in a partial 256-row tile pair.
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (1, 256, 256), (127, 256, 384), (129, 384, 512),
                                   (300, 512, 1024), (256, 896, 2048), (640, 1280, 256)])
def test_pow2_gemm_block128_random(fb, orc, M, N, K, out_dtype):
    _run_random(fb, orc, M, N, K, 0, out_dtype, 3 * M + N + K)


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (200, 384, 512), (1, 128, 128), (384, 896, 1024)])
def test_pow2_gemm_rowscale_random(fb, orc, M, N, K, out_dtype):
    _run_random(fb, orc, M, N, K, 1, out_dtype, 5 * M + N + K)


@pytest.mark.parametrize("mode", [0, 1])
def test_pow2_gemm_many_tiles_full_rows(fb, orc, mode):
    """Every column of every 7th row of a problem where each CTA pair walks
    several tiles and the stage, scale-slot and accumulator rings wrap many
    times, three runs: a race between the scale warps, the MMA and the
    epilogue shows up as scattered elements beyond the element-wise bound."""
    M, N, K = 2048, 7168, 2048
    a, b = rand_codes((M, K), 21), rand_codes((N, K), 22)
    sa = rand_pow2_scales((K // 128, M), 23)
    sb = rand_pow2_scales((N // 128, K // 128) if mode == 0 else (K // 128, N), 24)
    rows = np.arange(0, M, 7)
    cols = np.arange(N)
    ref = orc.gemm_blockscaled(a, sa, b, sb, mode, rows=rows, cols=cols)
    bound = _elementwise_bound(orc, a, sa, b, sb, mode, K, True, ref, rows=rows, cols=cols)
    A, SA, B, SB = _dev(a), _dev(sa), _dev(b), _dev(sb)
    for rep in range(3):
        d = fb.fp8_gemm_blockscaled_pow2(A, SA, B, SB, mode, torch.bfloat16)
        got = to_np(d)[rows]
        what = "pow2 many tiles mode%d rep%d" % (mode, rep)
        assert_gemm_close(got, ref, True, orc, what)
        _check_elementwise(got, ref, bound, what)
    assert fb.fp8_get_status() == 0


def test_pow2_gemm_agrees_with_promoted_gemm(fb, orc):
    """The two GEMMs on the same power-of-two operands: both within the
    element-wise bound of the fp64 product, so within twice it of each other."""
    M, N, K = 512, 896, 1024
    a, b = rand_codes((M, K), 31), rand_codes((N, K), 32)
    sa = rand_pow2_scales((K // 128, M), 33)
    sb = rand_pow2_scales((N // 128, K // 128), 34)
    A, SA, B, SB = _dev(a), _dev(sa), _dev(b), _dev(sb)
    d_mx = to_np(fb.fp8_gemm_blockscaled_pow2(A, SA, B, SB, 0, torch.float32))
    d_pr = to_np(fb.fp8_gemm_blockscaled(A, SA, B, SB, 0, torch.float32))
    ref = orc.gemm_blockscaled(a, sa, b, sb, 0)
    bound = _elementwise_bound(orc, a, sa, b, sb, 0, K, False, ref)
    _check_elementwise(d_mx, ref, bound, "pow2 vs fp64")
    _check_elementwise(d_pr, ref, bound, "promoted vs fp64")
    _check_elementwise(d_mx, d_pr, 2 * bound, "pow2 vs promoted")


def test_pow2_dense_linear_full_sampled(fb, orc):
    """4096 x 7168 x 7168 through the GPU quantisers in power-of-two mode and
    the microscaled GEMM; the oracle recomputes 48 rows x 3 column blocks from
    the bf16 inputs."""
    d = S.dense_linear()
    x, w = d["x"], d["w"]
    P = fb.FP8_SCALE_POW2
    qx, sx = fb.fp8_quant_act_1x128(x.cuda(), flags=P)
    qw, sw = fb.fp8_quant_weight_128x128(w.cuda(), flags=P)
    y = fb.fp8_gemm_blockscaled_pow2(qx, sx, qw, sw)
    g = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, 4095], g.choice(4096, 46, replace=False)]))
    nbs = sorted({0, 55, int(g.integers(1, 55))})
    xb = S.bf16_bits(x)
    qa, sa = orc.quant_act_1x128(xb[rows], P)
    got = to_np(y)[rows]
    for nb in nbs:
        wb = S.bf16_bits(w[nb * 128:(nb + 1) * 128])
        qb, sb = orc.quant_weight_128x128(wb, P)
        ref = orc.gemm_blockscaled(qa, sa, qb, sb, 0)
        what = "pow2 dense nb=%d" % nb
        g_blk = got[:, nb * 128:(nb + 1) * 128]
        assert_gemm_close(g_blk, ref, True, orc, what)
        _check_elementwise(g_blk, ref, _elementwise_bound(orc, qa, sa, qb, sb, 0, 7168, True, ref), what)
    assert fb.fp8_get_status() == 0


def test_pow2_wgrad_full_sampled(fb, orc):
    """dW = dY^T X with power-of-two 128x1 token tiles, fp32 out, K = 8192."""
    d = S.wgrad()
    dy, x = d["dy"], d["x"]
    P = fb.FP8_SCALE_POW2
    qa, sa = fb.fp8_quant_act_128x1(dy.cuda(), flags=P)
    qb, sb = fb.fp8_quant_act_128x1(x.cuda(), flags=P)
    dw = fb.fp8_gemm_blockscaled_pow2(qa, sa, qb, sb, fb.FP8_BSCALE_ROW, torch.float32)
    g = np.random.default_rng(6)
    ii = np.unique(np.concatenate([[0, 7167], g.choice(7168, 30, replace=False)]))
    jj = np.unique(np.concatenate([[0, 7167], g.choice(7168, 200, replace=False)]))
    dyb, xb = S.bf16_bits(dy), S.bf16_bits(x)
    qar, sar = orc.quant_act_128x1(np.ascontiguousarray(dyb[:, ii]), P)
    qbr, sbr = orc.quant_act_128x1(np.ascontiguousarray(xb[:, jj]), P)
    ref = orc.gemm_blockscaled(qar, sar, qbr, sbr, 1)
    got = dw.cpu().numpy()[np.ix_(ii, jj)]
    assert_gemm_close(got, ref, False, orc, "pow2 wgrad")
    _check_elementwise(got, ref, _elementwise_bound(orc, qar, sar, qbr, sbr, 1, 8192, False, ref), "pow2 wgrad")
    assert fb.fp8_get_status() == 0


def test_pow2_gemm_reports_a_scale_that_is_not_a_power_of_two(fb):
    M, N, K = 128, 256, 256
    a, b = rand_codes((M, K), 41), rand_codes((N, K), 42)
    sa = rand_pow2_scales((K // 128, M), 43)
    sb = rand_pow2_scales((N // 128, K // 128), 44)
    sa[1, 17] = 0.75
    assert fb.fp8_get_status() == 0
    fb.fp8_gemm_blockscaled_pow2(_dev(a), _dev(sa), _dev(b), _dev(sb), 0, torch.bfloat16)
    assert fb.fp8_get_status() == fb.FP8_ERR_SCALE
    assert fb.fp8_get_status() == 0
