"""Pins for the oracle's block-scaled GEMM (the tmdrlife.com and gnrental.net pages: each 128-element K
interval is accumulated, multiplied by the scaling factors and added into
FP32; the jp-study.kr page: the interval is 128 elements).  The oracle forms the exact
fp64 product of the dequantised operands, which equals the block-promoted
sum sum_kb sA*sB*P_kb."""
from fractions import Fraction

import numpy as np
import pytest
import torch


def _codes(shape, seed, lo=0, hi=256):
    g = np.random.default_rng(seed)
    c = g.integers(lo, hi, size=shape, dtype=np.int64).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x3C       # no NaN codes
    return c


def _int_values(codes):
    """E4M3 value * 2^9 as an exact integer, via torch's float8 decode."""
    v = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy() * 512.0
    assert np.all(v == np.round(v))
    return v.astype(np.int64)


def _pow2_scales(shape, seed):
    g = np.random.default_rng(seed)
    return (2.0 ** g.integers(-12, 4, size=shape)).astype(np.float32)


def test_exact_block_sums_tiny(orc):
    """D from exact rational arithmetic on integer block partials (b_mode 0)."""
    M, N, K = 5, 128, 256
    a, b = _codes((M, K), 1), _codes((N, K), 2)
    g = np.random.default_rng(3)
    sa = g.uniform(0.01, 2, size=(K // 128, M)).astype(np.float32)
    sb = g.uniform(0.01, 2, size=(N // 128, K // 128)).astype(np.float32)
    ai, bi = _int_values(a), _int_values(b)
    d = orc.gemm_blockscaled(a, sa, b, sb, 0)
    for m in range(M):
        for n in range(0, N, 7):
            exact = Fraction(0)
            mag = Fraction(0)
            for kb in range(K // 128):
                sl = slice(kb * 128, (kb + 1) * 128)
                P = int(np.dot(ai[m, sl], bi[n, sl]))           # exact in int64 (< 2^43)
                mag += abs(Fraction(float(sa[kb, m])) * Fraction(float(sb[n // 128, kb]))) * \
                    int(np.abs(ai[m, sl] * bi[n, sl]).sum())
                exact += Fraction(float(sa[kb, m])) * Fraction(float(sb[n // 128, kb])) * P
            exact /= 2 ** 18
            mag /= 2 ** 18
            # fp64 summation of K exact products: |err| <= K * 2^-53 * sum|terms|
            assert abs(Fraction(d[m, n]) - exact) <= K * Fraction(1, 2 ** 53) * mag


def test_unit_scales_single_block_is_integer_matmul(orc):
    M, N, K = 33, 256, 128
    a, b = _codes((M, K), 4), _codes((N, K), 5)
    ones_a = np.ones((1, M), np.float32)
    ones_b = np.ones((N // 128, 1), np.float32)
    d = orc.gemm_blockscaled(a, ones_a, b, ones_b, 0)
    ref = (_int_values(a) @ _int_values(b).T).astype(np.float64) * 2.0 ** -18
    assert np.array_equal(d, ref)


def test_one_hot_b_selects_dequantised_columns(orc):
    M, K = 17, 256
    N = 128
    a = _codes((M, K), 6)
    sa = _pow2_scales((K // 128, M), 7)
    b = np.zeros((N, K), np.uint8)
    for n in range(N):
        b[n, 2 * n] = 0x38                      # 1.0 at k = 2n
    sb = np.ones((1, K // 128), np.float32)
    d = orc.gemm_blockscaled(a, sa, b, sb, 0)
    table = orc.e4m3_decode(np.arange(256))
    for n in range(N):
        k = 2 * n
        assert np.array_equal(d[:, n], table[a[:, k]] * sa[k // 128, :].astype(np.float64))


def test_mode1_equals_mode0_for_blockwise_constant_scales(orc):
    M, N, K = 9, 256, 384
    a, b = _codes((M, K), 8), _codes((N, K), 9)
    sa = _pow2_scales((K // 128, M), 10)
    sb0 = np.random.default_rng(11).uniform(0.1, 3, size=(N // 128, K // 128)).astype(np.float32)
    sb1 = np.repeat(sb0.T, 128, axis=1)          # [K/128][N]
    d0 = orc.gemm_blockscaled(a, sa, b, sb0, 0)
    d1 = orc.gemm_blockscaled(a, sa, b, sb1, 1)
    assert np.array_equal(d0, d1)


def test_mode1_transpose_symmetry(orc):
    """With per-row scales on both sides, D(A,B) = D(B,A)^T exactly."""
    M, N, K = 12, 20, 256
    a, b = _codes((M, K), 12), _codes((N, K), 13)
    g = np.random.default_rng(14)
    sa = g.uniform(0.1, 3, size=(K // 128, M)).astype(np.float32)
    sb = g.uniform(0.1, 3, size=(K // 128, N)).astype(np.float32)
    assert np.array_equal(orc.gemm_blockscaled(a, sa, b, sb, 1), orc.gemm_blockscaled(b, sb, a, sa, 1).T)


def test_sampled_equals_full(orc):
    M, N, K = 40, 256, 256
    a, b = _codes((M, K), 15), _codes((N, K), 16)
    sa = _pow2_scales((K // 128, M), 17)
    sb = _pow2_scales((N // 128, K // 128), 18)
    full = orc.gemm_blockscaled(a, sa, b, sb, 0)
    rows = np.array([39, 0, 17]); cols = np.array([255, 3, 128, 127])
    assert np.array_equal(orc.gemm_blockscaled(a, sa, b, sb, 0, rows, cols), full[np.ix_(rows, cols)])


def _bf16_value(bits):
    return Fraction(float(np.array([bits << 16], np.uint32).view(np.float32)[0]))


def _nearest_bf16_exact(d):
    """Nearest bf16 by exact rational distance among the neighbours of the
    fp32 cast (ties to the even bit pattern)."""
    if d == 0.0:
        return 0x8000 if np.signbit(d) else 0
    b = int(np.array([d], np.float32).view(np.uint32)[0] >> 16)
    best = None
    for c in (b - 1, b, b + 1, b + 2):
        c &= 0xFFFF
        if (c & 0x7F80) == 0x7F80:
            continue
        v = _bf16_value(c)
        if (v < 0) != (d < 0) and v != 0:
            continue
        dist = abs(v - Fraction(d))
        key = (dist, c & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def test_round_bf16_single_rounding(orc):
    g = np.random.default_rng(19)
    d = np.concatenate([g.standard_normal(20000) * 10.0 ** g.integers(-30, 30, 20000),
                        [1.00390625, 1.01171875, -6.240013213366936e-31, 1e-40, -1e-42,
                         1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -40]])
    ours = orc.round_bf16(d)
    for v, o in zip(d, ours):
        assert o == _nearest_bf16_exact(v), v


def test_round_bf16_matches_torch_on_fp32_inputs(orc):
    """On values that are already fp32 torch's cast rounds once: compare there."""
    g = np.random.default_rng(20)
    d = (g.standard_normal(200000) * 10.0 ** g.integers(-20, 20, 200000)).astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(d).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.round_bf16(d), ref)
