"""GPU parity of the grouped (per-expert) GEMM for power-of-two scales on the
microscaled tensor-core MMA (the jp-study.kr page: 256 routed experts, each processing the
rows dispatched to it; the tmdrlife.com and gnrental.net pages: power-of-two scales, tensor cores that take
the scaling factors) against the oracle's fp64 per-expert product: the GEMM
tolerance plus the element-wise recursive-summation bound of the dense
power-of-two tests (2 * (K + K/32) * 2^-24 * sum|a*b| + one bf16 rounding).
"""
import numpy as np
import pytest
import torch

from fp8_fine_grained_16_b300 import synthetic as S
from _checks import assert_gemm_close, assert_same_bits, rand_codes, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fb():
    from fp8_fine_grained_16_b300 import build
    build.build()
    from fp8_fine_grained_16_b300 import fp8bs
    return fp8bs


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _pow2(shape, seed):
    g = np.random.default_rng(seed)
    return np.ldexp(np.float32(1.0), g.integers(-12, 5, size=shape)).astype(np.float32)


# Ragged experts (empty ones included) and widths that end in a partial
# 224-column tile (256 = 224 + 32, 384 = 224 + 160, 512 = 2 x 224 + 64).
@pytest.mark.parametrize("counts,N,K", [
    ([0, 3, 37, 129, 300, 0], 256, 256),
    ([128, 128], 384, 512),
    ([1], 256, 128),
    ([5, 0, 0, 250, 1, 130, 257], 512, 384),
    ([200] * 12, 896, 1024),
])
def test_grouped_pow2_small(fb, orc, counts, N, K):
    seed = sum(counts) + N + K
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    E, total = len(counts), int(off[-1])
    a = rand_codes((total, K), seed)
    sa = _pow2((K // 128, total), seed + 1)
    b = rand_codes((E, N, K), seed + 2)
    sb = _pow2((E, N // 128, K // 128), seed + 3)
    d = fb.fp8_grouped_gemm_blockscaled_pow2(_dev(a), _dev(sa), _dev(b), _dev(sb), _dev(off))
    assert fb.fp8_get_status() == 0
    ref = orc.grouped_gemm_blockscaled(a, sa, b, sb, off)
    got = to_np(d)
    assert_gemm_close(got, ref, True, orc, "grouped pow2 %s" % (counts,))
    absref = orc.grouped_gemm_blockscaled((a & 0x7F).astype(np.uint8), sa, (b & 0x7F).astype(np.uint8), sb, off)
    bound = 2 * (K + K // 32) * 2.0 ** -24 * absref + np.abs(ref) * 2.0 ** -8
    assert np.all(np.abs(got - ref) <= bound)


def test_grouped_pow2_bad_offsets_record_status(fb):
    E, N, K, total = 3, 256, 128, 40
    a = torch.zeros((total, K), dtype=torch.uint8, device="cuda")
    sa = torch.ones((1, total), dtype=torch.float32, device="cuda")
    b = torch.zeros((E, N, K), dtype=torch.uint8, device="cuda")
    sb = torch.ones((E, 2, 1), dtype=torch.float32, device="cuda")
    off = torch.tensor([0, 30, 20, 40], dtype=torch.int32, device="cuda")   # not monotone
    fb.fp8_grouped_gemm_blockscaled_pow2(a, sa, b, sb, off)
    assert fb.fp8_get_status() == fb.FP8_ERR_OFFSETS


def test_moe_up_pow2_full_sampled(fb, orc):
    """4096 tokens x 7168 -> top-8 of 256 -> power-of-two quantise -> dispatch
    -> grouped GEMM N=4096; five experts checked against the oracle on two
    column blocks each."""
    T, E, k, N, K = 4096, 256, 8, 4096, 7168
    P = fb.FP8_SCALE_POW2
    d = S.moe_up(with_weights=False)
    x, logits = d["x"], d["logits"]
    r = fb.fp8_moe_route_topk(logits.cuda(), k)
    ref_route = orc.route_topk(logits.numpy(), k)
    assert_same_bits(r["off"], ref_route["off"], "off")
    qx, sx = fb.fp8_quant_act_1x128(x.cuda(), flags=P)
    qa, sa = fb.fp8_permute_rows(qx, sx, r["src_row"])
    qxr, sxr = orc.quant_act_1x128(S.bf16_bits(x), P)
    par, spr = orc.permute_rows(qxr, sxr, ref_route["src_row"])
    assert_same_bits(qa, par, "permuted codes")
    assert_same_bits(sa, spr, "permuted scales")
    w = S.expert_weights(0, E, N, K, device="cuda")
    qw, sw = fb.fp8_quant_weight_128x128(w, flags=P)
    del w
    y = fb.fp8_grouped_gemm_blockscaled_pow2(qa, sa, qw, sw, r["off"])
    assert fb.fp8_get_status() == 0
    off = ref_route["off"]
    counts = np.diff(off)
    got = to_np(y)
    for e in sorted({0, 255, int(np.argmax(counts)), int(np.argmin(counts)), 77}):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        wb = S.bf16_bits(S.expert_weight(0, e, N, K, device="cuda"))
        qb, sbb = orc.quant_weight_128x128(wb, P)
        assert_same_bits(qw[e], qb, "expert %d codes" % e)
        for nb in (0, N // 128 - 1):
            cols = np.arange(nb * 128, (nb + 1) * 128)
            ref = orc.gemm_blockscaled(par[lo:hi], np.ascontiguousarray(spr[:, lo:hi]), qb[cols], sbb[nb:nb + 1], 0)
            assert_gemm_close(got[lo:hi, nb * 128:(nb + 1) * 128], ref, True, orc, "moe_up pow2 e=%d nb=%d" % (e, nb))


def test_moe_down_pow2_full_sampled(fb, orc):
    """The down-projection workload (256 experts, top-8 of 4096 tokens,
    K = 2048) with power-of-two scales: h quantised 1x128 to powers of two,
    grouped GEMM N = 7168 on the microscaled MMA; four experts (the first, the
    last, the largest and one in the middle) checked against the oracle on the
    first and last column blocks."""
    T, E, k, N, K = 4096, 256, 8, 7168, 2048
    P = fb.FP8_SCALE_POW2
    d = S.moe_down(with_weights=False)
    h, logits = d["h"], d["logits"]
    r = fb.fp8_moe_route_topk(logits.cuda(), k)
    ref_route = orc.route_topk(logits.numpy(), k)
    assert_same_bits(r["off"], ref_route["off"], "off")
    qh, sh = fb.fp8_quant_act_1x128(h.cuda(), flags=P)
    qhr, shr = orc.quant_act_1x128(S.bf16_bits(h), P)
    assert_same_bits(qh, qhr, "down-projection input codes")
    assert_same_bits(sh, shr, "down-projection input scales")
    w = S.expert_weights(1, E, N, K, device="cuda")
    qw, sw = fb.fp8_quant_weight_128x128(w, flags=P)
    del w
    y = fb.fp8_grouped_gemm_blockscaled_pow2(qh, sh, qw, sw, r["off"])
    assert fb.fp8_get_status() == 0
    off = ref_route["off"]
    counts = np.diff(off)
    got = to_np(y)
    for e in sorted({0, 255, int(np.argmax(counts)), 131}):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        wb = S.bf16_bits(S.expert_weight(1, e, N, K, device="cuda"))
        qb, sbb = orc.quant_weight_128x128(wb, P)
        assert_same_bits(qw[e], qb, "expert %d codes" % e)
        for nb in (0, N // 128 - 1):
            cols = np.arange(nb * 128, (nb + 1) * 128)
            ref = orc.gemm_blockscaled(qhr[lo:hi], np.ascontiguousarray(shr[:, lo:hi]), qb[cols], sbb[nb:nb + 1], 0)
            assert_gemm_close(got[lo:hi, nb * 128:(nb + 1) * 128], ref, True, orc,
                              "moe_down pow2 e=%d nb=%d" % (e, nb))
