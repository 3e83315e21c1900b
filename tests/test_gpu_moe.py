"""GPU parity of routing, dispatch (permute), the grouped GEMM and the BF16
combine (the jp-study.kr page: 256 routed experts, 8 active, activations quantised before
dispatch; the gnrental.net page: combine kept in BF16)."""
import numpy as np
import pytest
import torch

from fp8_fine_grained_16_b300 import synthetic as S
from _checks import assert_gemm_close, assert_same_bits, rand_codes, rand_scales, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fb():
    from fp8_fine_grained_16_b300 import build
    build.build()
    from fp8_fine_grained_16_b300 import fp8bs
    return fp8bs


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _check_route(fb, orc, logits, k):
    r = fb.fp8_moe_route_topk(logits.cuda(), k)
    ref = orc.route_topk(logits.numpy(), k)
    for key in ("idx", "off", "src_row", "pos"):
        assert_same_bits(r[key], ref[key], key)
    g = r["gate"].cpu().numpy()
    assert np.allclose(g, ref["gate"], rtol=2e-6, atol=1e-7)
    return r, ref


def test_route_small_with_ties(fb, orc):
    g = np.random.default_rng(0)
    logits = torch.from_numpy(g.integers(-3, 4, size=(200, 12)).astype(np.float32))
    _check_route(fb, orc, logits, 3)


@pytest.mark.parametrize("T,E,k", [(1, 4, 4), (63, 33, 5), (65, 64, 8), (130, 1024, 32), (4096, 256, 8),
                                   (20000, 256, 8), (65536, 256, 8)])
def test_route_shapes(fb, orc, T, E, k):
    logits = torch.randn((T, E), generator=torch.Generator().manual_seed(T + E))
    _check_route(fb, orc, logits, k)


def test_route_moe_configs(fb, orc):
    _check_route(fb, orc, S.moe_up(with_weights=False)["logits"], 8)
    _check_route(fb, orc, S.moe_down(with_weights=False)["logits"], 8)


def test_permute_rows(fb, orc):
    rows, K = 300, 640
    q = rand_codes((rows, K), 1)
    s = rand_scales((K // 128, rows), 2)
    src = np.random.default_rng(3).integers(0, rows, size=1001).astype(np.int32)
    qo, so = fb.fp8_permute_rows(_dev(q), _dev(s), _dev(src))
    qr, sr = orc.permute_rows(q, s, src)
    assert_same_bits(qo, qr, "q")
    assert_same_bits(so, sr, "s")


def test_permute_bad_index_records_status(fb):
    q = torch.zeros((4, 128), dtype=torch.uint8, device="cuda")
    s = torch.ones((1, 4), dtype=torch.float32, device="cuda")
    src = torch.tensor([0, 7, 1], dtype=torch.int32, device="cuda")
    qo, so = fb.fp8_permute_rows(q, s, src)
    assert fb.fp8_get_status() == fb.FP8_ERR_OFFSETS
    assert float(so[0, 1]) == 0.0 and float(so[0, 2]) == 1.0


def _combine_bound(y, pos, gate, exact):
    """|got - exact| <= one bf16 ulp of exact + fp32 summation slack."""
    yf = y.double().numpy()
    mag = np.einsum("tj,tjn->tn", np.abs(gate.astype(np.float64)), np.abs(yf[pos]))
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(exact), 2.0 ** -126))) - 7)
    return ulp + mag * 2.0 ** -20


@pytest.mark.parametrize("T,k,N,rows", [(50, 8, 96, 400), (7, 1, 8, 7), (300, 3, 1000, 900)])
def test_combine_small(fb, orc, T, k, N, rows):
    g = np.random.default_rng(T)
    y = torch.randn((rows, N), generator=torch.Generator().manual_seed(T)).to(torch.bfloat16)
    pos = g.integers(0, rows, size=(T, k)).astype(np.int32)
    gate = g.dirichlet(np.ones(k), size=T).astype(np.float32)
    out = fb.fp8_moe_combine_bf16(y.cuda(), _dev(pos), _dev(gate))
    ref = orc.moe_combine(S.bf16_bits(y), pos, gate)
    got = to_np(out)
    exact = np.einsum("tj,tjn->tn", gate.astype(np.float64), y.double().numpy()[pos])
    assert np.all(np.abs(got - exact) <= _combine_bound(y, pos, gate, exact))
    # Held to the oracle: the GPU rounds an fp32 slot-order sum once, the
    # oracle an fp64 sum once, so the two bf16 results are at most one bf16
    # ulp apart, plus the fp32 summation error where the sum cancels.
    refv = S.from_bf16_bits(ref).double().numpy()
    assert np.all(np.abs(got - refv) <= _combine_bound(y, pos, gate, refv))
    print("combine: %.4f%% of outputs differ from the oracle's single rounding" % (100 * np.mean(got != refv)))
    assert np.mean(got != refv) < 0.01


def _grouped_case(fb, orc, counts, N, K, seed):
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    E, total = len(counts), int(off[-1])
    a = rand_codes((total, K), seed)
    sa = rand_scales((K // 128, total), seed + 1)
    b = rand_codes((E, N, K), seed + 2)
    sb = rand_scales((E, N // 128, K // 128), seed + 3)
    d = fb.fp8_grouped_gemm_blockscaled(_dev(a), _dev(sa), _dev(b), _dev(sb), _dev(off))
    assert fb.fp8_get_status() == 0
    ref = orc.grouped_gemm_blockscaled(a, sa, b, sb, off)
    assert_gemm_close(to_np(d), ref, True, orc, "grouped %s" % (counts,))


@pytest.mark.parametrize("counts,N,K", [
    ([0, 3, 37, 129, 300, 0], 256, 256),
    ([128, 128], 384, 512),
    ([1], 256, 128),
    ([5, 0, 0, 250, 1, 130, 257], 512, 384),
])
def test_grouped_small(fb, orc, counts, N, K):
    _grouped_case(fb, orc, counts, N, K, sum(counts) + N)


def test_grouped_bad_offsets_record_status(fb):
    E, N, K, total = 3, 256, 128, 40
    a = torch.zeros((total, K), dtype=torch.uint8, device="cuda")
    sa = torch.ones((1, total), dtype=torch.float32, device="cuda")
    b = torch.zeros((E, N, K), dtype=torch.uint8, device="cuda")
    sb = torch.ones((E, 2, 1), dtype=torch.float32, device="cuda")
    off = torch.tensor([0, 30, 20, 40], dtype=torch.int32, device="cuda")   # not monotone
    fb.fp8_grouped_gemm_blockscaled(a, sa, b, sb, off)
    assert fb.fp8_get_status() == fb.FP8_ERR_OFFSETS


def _moe_sample_check(fb, orc, a, sa, qw, sw, off_ref, d, experts, wseed, N, K, what):
    """Oracle on every row of the chosen experts x 2 column blocks.  `a`, `sa`
    and the expert weights' codes are the oracle's own quantisation (the
    GPU's are asserted equal to them first)."""
    got = to_np(d)
    for e in experts:
        lo, hi = int(off_ref[e]), int(off_ref[e + 1])
        if hi == lo:
            continue
        w = S.expert_weight(wseed, e, N, K, device="cuda")
        qb, sb = orc.quant_weight_128x128(S.bf16_bits(w))
        assert_same_bits(qw[e], qb, "expert %d codes" % e)
        assert_same_bits(sw[e], sb, "expert %d scales" % e)
        for nb in (0, N // 128 - 1):
            cols = np.arange(nb * 128, (nb + 1) * 128)
            ref = orc.gemm_blockscaled(a[lo:hi], np.ascontiguousarray(sa[:, lo:hi]), qb[cols], sb[nb:nb + 1], 0)
            assert_gemm_close(got[lo:hi, nb * 128:(nb + 1) * 128], ref, True, orc, "%s e=%d nb=%d" % (what, e, nb))


def test_moe_up_full_sampled(fb, orc):
    """4096 tokens x 7168 -> top-8 of 256 -> quantise -> dispatch -> grouped GEMM N=4096."""
    T, E, k, N, K = 4096, 256, 8, 4096, 7168
    d = S.moe_up(with_weights=False)
    x, logits = d["x"], d["logits"]
    r = fb.fp8_moe_route_topk(logits.cuda(), k)
    ref_route = orc.route_topk(logits.numpy(), k)
    assert_same_bits(r["off"], ref_route["off"], "off")
    assert_same_bits(r["src_row"], ref_route["src_row"], "src_row")
    qx, sx = fb.fp8_quant_act_1x128(x.cuda())
    qa, sa = fb.fp8_permute_rows(qx, sx, r["src_row"])
    qxr, sxr = orc.quant_act_1x128(S.bf16_bits(x))
    par, spr = orc.permute_rows(qxr, sxr, ref_route["src_row"])
    assert_same_bits(qa, par, "permuted codes")
    assert_same_bits(sa, spr, "permuted scales")
    w = S.expert_weights(0, E, N, K, device="cuda")
    qw, sw = fb.fp8_quant_weight_128x128(w)
    del w
    y = fb.fp8_grouped_gemm_blockscaled(qa, sa, qw, sw, r["off"])
    assert fb.fp8_get_status() == 0
    counts = np.diff(ref_route["off"])
    experts = sorted({0, 255, int(np.argmax(counts)), int(np.argmin(counts)), 77})
    _moe_sample_check(fb, orc, par, spr, qw, sw, ref_route["off"], y, experts, 0, N, K, "moe_up")


def test_moe_down_full_sampled(fb, orc):
    """Grouped GEMM N=7168, K=2048 on SiLU(g)*u rows of the down-projection
    workload (256 experts, top-8 of 4096 tokens)."""
    T, E, k, N, K = 4096, 256, 8, 7168, 2048
    d = S.moe_down(with_weights=False)
    h, logits = d["h"], d["logits"]
    r = fb.fp8_moe_route_topk(logits.cuda(), k)
    ref_route = orc.route_topk(logits.numpy(), k)
    assert_same_bits(r["off"], ref_route["off"], "off")
    qh, sh = fb.fp8_quant_act_1x128(h.cuda())
    qhr, shr = orc.quant_act_1x128(S.bf16_bits(h))
    assert_same_bits(qh, qhr, "down-projection input codes")
    assert_same_bits(sh, shr, "down-projection input scales")
    w = S.expert_weights(1, E, N, K, device="cuda")
    qw, sw = fb.fp8_quant_weight_128x128(w)
    del w
    y = fb.fp8_grouped_gemm_blockscaled(qh, sh, qw, sw, r["off"])
    assert fb.fp8_get_status() == 0
    counts = np.diff(ref_route["off"])
    experts = sorted({0, 255, int(np.argmax(counts)), 131})
    _moe_sample_check(fb, orc, qhr, shr, qw, sw, ref_route["off"], y, experts, 1, N, K, "moe_down")


def test_combine_full_size_sampled(fb, orc):
    """The BF16 combine at the down-projection's full size: expert outputs
    [32768, 7168] (seeded, drawn here, not taken from a GPU GEMM), the
    oracle's top-8 positions and gates of 4096 tokens; every 17th token held
    to the oracle's single rounding within one bf16 ulp (+ the fp32
    summation slack), and the GPU's own routing giving the same result."""
    T, E, k, N = 4096, 256, 8, 7168
    logits = S.moe_down(with_weights=False)["logits"]
    ref_route = orc.route_topk(logits.numpy(), k)
    y = torch.randn((T * k, N), generator=torch.Generator().manual_seed(44)).to(torch.bfloat16)
    pos, gate = ref_route["pos"], ref_route["gate"]
    y_dev = y.cuda()
    out = fb.fp8_moe_combine_bf16(y_dev, _dev(pos), _dev(gate))
    rows = np.arange(0, T, 17)
    got = to_np(out)[rows]
    ref = S.from_bf16_bits(orc.moe_combine(S.bf16_bits(y), pos[rows], gate[rows])).double().numpy()
    assert np.all(np.abs(got - ref) <= _combine_bound(y, pos[rows], gate[rows], ref))
    assert np.mean(got != ref) < 0.01
    r = fb.fp8_moe_route_topk(logits.cuda(), k)
    out_gpu_route = fb.fp8_moe_combine_bf16(y_dev, r["pos"], r["gate"])
    assert torch.allclose(out.float(), out_gpu_route.float(), rtol=1e-2, atol=1e-2)
