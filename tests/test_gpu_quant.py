"""GPU parity of the E4M3 cast and the three quantisers against the oracle:
codes and scales must match bit for bit (the jp-study.kr page: online max-abs per 1x128
activation tile and per 128x128 weight block; the jp-study.kr page: FP8 Wgrad -> 128x1
tiles along tokens; the tmdrlife.com and gnrental.net pages: power-of-2 scales)."""
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


def _edge_tensor(M, K):
    """Rows that hit the corner cases: zero tiles, bf16 extremes, subnormal
    bf16 inputs, -0, constant tiles, a single non-zero element."""
    x = _bf16((M, K), 99)
    x[0] = 0.0
    x[1] = -0.0
    x[2, :] = 3.3895313892515355e38          # largest bf16
    x[3, ::2] = -3.3895313892515355e38
    x[4] = 9.183549615799121e-41              # a subnormal bf16
    x[5] = 1.0
    x[6] = 0.0
    x[6, 77] = -2.5
    x[7] = torch.arange(K, dtype=torch.float32).to(torch.bfloat16) * 1e-30
    return x


def test_cast_exhaustive_all_fp32(fb, orc):
    """Every fp32 bit pattern (NaNs excluded) casts to the oracle's code."""
    chunk = 1 << 28
    for start in range(0, 1 << 32, chunk):
        bits = torch.arange(start, start + chunk, dtype=torch.int64, device="cuda")
        x = bits.to(torch.int32).view(torch.float32)
        q = fb.fp8_cast_e4m3(x)
        ref = torch.from_numpy(orc.e4m3_encode_bits(start, chunk)).cuda()
        bad = (q != ref) & ~torch.isnan(x)
        n = int(bad.sum())
        assert n == 0, "mismatch at 0x%08x" % (start + int(torch.nonzero(bad)[0]))


def test_cast_tail_lengths(fb, orc):
    for n in [1, 7, 9, 1000003]:
        x = torch.randn(n, generator=torch.Generator().manual_seed(n)) * 100
        q = fb.fp8_cast_e4m3(x.cuda())
        assert_same_bits(q, orc.e4m3_encode(x.numpy()), "cast n=%d" % n)


@pytest.mark.parametrize("pow2", [0, 1])
@pytest.mark.parametrize("M,K", [(1, 128), (127, 384), (129, 256), (300, 1024), (128, 512), (33, 7168)])
def test_quant_act_1x128(fb, orc, M, K, pow2):
    x = _bf16((M, K), M * 7 + K)
    q, s = fb.fp8_quant_act_1x128(x.cuda(), flags=pow2)
    qr, sr = orc.quant_act_1x128(S.bf16_bits(x), flags=pow2)
    assert_same_bits(q, qr, "q")
    assert_same_bits(s, sr, "s")


@pytest.mark.parametrize("pow2", [0, 1])
def test_quant_act_1x128_edges_and_stride(fb, orc, pow2):
    x = _edge_tensor(16, 640)
    big = torch.zeros((16, 1024), dtype=torch.bfloat16)
    big[:, :640] = x
    q, s = fb.fp8_quant_act_1x128(big.cuda()[:, :640], flags=pow2)      # ldx = 1024 > K
    qr, sr = orc.quant_act_1x128(S.bf16_bits(x), flags=pow2)
    assert_same_bits(q, qr, "q")
    assert_same_bits(s, sr, "s")


@pytest.mark.parametrize("pow2", [0, 1])
def test_quant_act_1x128_tiny_dense(fb, orc, pow2):
    x = S.tiny_dense()["x"]
    q, s = fb.fp8_quant_act_1x128(x.cuda(), flags=pow2)
    qr, sr = orc.quant_act_1x128(S.bf16_bits(x), flags=pow2)
    assert_same_bits(q, qr, "q")
    assert_same_bits(s, sr, "s")


def test_quant_act_1x128_dense_linear_full(fb, orc):
    x = S.dense_linear()["x"]
    for pow2 in (0, 1):
        q, s = fb.fp8_quant_act_1x128(x.cuda(), flags=pow2)
        qr, sr = orc.quant_act_1x128(S.bf16_bits(x), flags=pow2)
        assert_same_bits(q, qr, "q")
        assert_same_bits(s, sr, "s")


def test_quant_act_1x128_moe_down_input_full(fb, orc):
    h = S.moe_down(with_weights=False)["h"]
    q, s = fb.fp8_quant_act_1x128(h.cuda(), flags=1)
    qr, sr = orc.quant_act_1x128(S.bf16_bits(h), flags=1)
    assert_same_bits(q, qr, "q")
    assert_same_bits(s, sr, "s")


@pytest.mark.parametrize("pow2", [0, 1])
@pytest.mark.parametrize("N,K", [(128, 128), (256, 512), (384, 640), (128, 7168)])
def test_quant_weight_128x128(fb, orc, N, K, pow2):
    w = _bf16((N, K), N + K, 0.02)
    w[N // 2, K // 3] = 5.0
    q, s = fb.fp8_quant_weight_128x128(w.cuda(), flags=pow2)
    qr, sr = orc.quant_weight_128x128(S.bf16_bits(w), flags=pow2)
    assert_same_bits(q, qr, "q")
    assert_same_bits(s, sr, "s")


def test_quant_weight_edges_and_stack(fb, orc):
    w = _edge_tensor(256, 384)
    q, s = fb.fp8_quant_weight_128x128(w.cuda())
    qr, sr = orc.quant_weight_128x128(S.bf16_bits(w))
    assert_same_bits(q, qr, "q")
    assert_same_bits(s, sr, "s")
    stack = _bf16((3, 256, 384), 5, 0.02)
    q, s = fb.fp8_quant_weight_128x128(stack.cuda())
    assert s.shape == (3, 2, 3)
    for e in range(3):
        qr, sr = orc.quant_weight_128x128(S.bf16_bits(stack[e]))
        assert_same_bits(q[e], qr, "q[%d]" % e)
        assert_same_bits(s[e], sr, "s[%d]" % e)


def test_quant_weight_dense_linear_full(fb, orc):
    w = S.dense_linear()["w"]
    q, s = fb.fp8_quant_weight_128x128(w.cuda())
    qr, sr = orc.quant_weight_128x128(S.bf16_bits(w))
    assert_same_bits(q, qr, "q")
    assert_same_bits(s, sr, "s")


@pytest.mark.parametrize("pow2", [0, 1])
@pytest.mark.parametrize("T,H", [(128, 8), (384, 200), (256, 7168), (128, 72)])
def test_quant_act_128x1(fb, orc, T, H, pow2):
    x = _bf16((T, H), T + H)
    qT, s = fb.fp8_quant_act_128x1(x.cuda(), flags=pow2)
    qr, sr = orc.quant_act_128x1(S.bf16_bits(x), flags=pow2)
    assert_same_bits(qT, qr, "qT")
    assert_same_bits(s, sr, "s")


def test_quant_act_128x1_edges_and_stride(fb, orc):
    xt = _edge_tensor(96, 256).t().contiguous()            # [T=256, H=96]: edge rows become edge columns
    T, H = xt.shape
    store = torch.zeros((T, 104), dtype=torch.bfloat16)    # ldx = 104 > H
    store[:, :H] = xt
    qT, s = fb.fp8_quant_act_128x1(store.cuda()[:, :H])
    qr, sr = orc.quant_act_128x1(S.bf16_bits(xt))
    assert_same_bits(qT, qr, "qT")
    assert_same_bits(s, sr, "s")


def test_quant_act_128x1_wgrad_full(fb, orc):
    d = S.wgrad()
    for name in ("dy", "x"):
        qT, s = fb.fp8_quant_act_128x1(d[name].cuda())
        qr, sr = orc.quant_act_128x1(S.bf16_bits(d[name]))
        assert_same_bits(qT, qr, name + " qT")
        assert_same_bits(s, sr, name + " s")


@pytest.mark.parametrize("flags", [0, 1])
def test_quant_act_weight_one_launch_dense_linear_full(fb, orc, flags):
    """X [4096,7168] and W [7168,7168] quantised in one launch: codes and
    scales of both bit for bit those of the oracle's 1x128 and 128x128 rules."""
    d = S.dense_linear()
    qx, sx, qw, sw = fb.fp8_quant_act_weight(d["x"].cuda(), d["w"].cuda(), flags=flags)
    qxr, sxr = orc.quant_act_1x128(S.bf16_bits(d["x"]), flags)
    qwr, swr = orc.quant_weight_128x128(S.bf16_bits(d["w"]), flags)
    assert_same_bits(qx, qxr, "qx")
    assert_same_bits(sx, sxr, "sx")
    assert_same_bits(qw, qwr, "qw")
    assert_same_bits(sw, swr, "sw")


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (9, 128, 256), (7, 256, 1152), (8, 128, 128)])
def test_quant_act_weight_one_launch_small_shapes(fb, orc, M, N, K):
    """One row, one weight block, and row counts that leave the last X CTA
    partly empty, both scale modes, against the oracle."""
    x = _bf16((M, K), M + K, 2.0)
    w = _bf16((N, K), N + K + 1, 0.05)
    for flags in (0, 1):
        qx, sx, qw, sw = fb.fp8_quant_act_weight(x.cuda(), w.cuda(), flags=flags)
        qxr, sxr = orc.quant_act_1x128(S.bf16_bits(x), flags)
        qwr, swr = orc.quant_weight_128x128(S.bf16_bits(w), flags)
        assert_same_bits(qx, qxr, "qx")
        assert_same_bits(sx, sxr, "sx")
        assert_same_bits(qw, qwr, "qw")
        assert_same_bits(sw, swr, "sw")


def test_quant_act_weight_one_launch_ragged_and_strided(fb, orc):
    """M not a multiple of the 8 rows a CTA takes, padded row strides for both
    operands, the edge rows of the 1x128 tests in X and a zero block in W."""
    M, N, K = 300, 384, 640
    x = torch.zeros((M, K + 24), dtype=torch.bfloat16)
    x[:, :K] = _bf16((M, K), 5)
    x[:8, :K] = _edge_tensor(8, K)
    w = torch.zeros((N, K + 8), dtype=torch.bfloat16)
    w[:, :K] = _bf16((N, K), 6, 0.02)
    w[128:256, 128:256] = 0.0
    for flags in (0, 1):
        qx, sx, qw, sw = fb.fp8_quant_act_weight(x.cuda()[:, :K], w.cuda()[:, :K], flags=flags)
        qxr, sxr = orc.quant_act_1x128(S.bf16_bits(x[:, :K].contiguous()), flags)
        qwr, swr = orc.quant_weight_128x128(S.bf16_bits(w[:, :K].contiguous()), flags)
        assert_same_bits(qx, qxr, "qx flags%d" % flags)
        assert_same_bits(sx, sxr, "sx flags%d" % flags)
        assert_same_bits(qw, qwr, "qw flags%d" % flags)
        assert_same_bits(sw, swr, "sw flags%d" % flags)
