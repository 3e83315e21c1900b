"""GPU parity of the block-scaled FP8 GEMM against the oracle's fp64 product
of the same E4M3 operands and scales (pages 2/3: per-interval promotion into
FP32 scaled by the two scales; page 4: 128-element interval)."""
import numpy as np
import pytest
import torch

from fp8_fine_grained_16_b300 import synthetic as S
from _checks import assert_gemm_close, rand_codes, rand_scales, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fb():
    from fp8_fine_grained_16_b300 import build
    build.build()
    from fp8_fine_grained_16_b300 import fp8bs
    return fp8bs


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _run_random(fb, orc, M, N, K, mode, out_dtype, seed):
    a, b = rand_codes((M, K), seed), rand_codes((N, K), seed + 1)
    sa = rand_scales((K // 128, M), seed + 2)
    sb = rand_scales((N // 128, K // 128) if mode == 0 else (K // 128, N), seed + 3)
    d = fb.fp8_gemm_blockscaled(_dev(a), _dev(sa), _dev(b), _dev(sb), mode, out_dtype)
    ref = orc.gemm_blockscaled(a, sa, b, sb, mode)
    assert_gemm_close(to_np(d), ref, out_dtype == torch.bfloat16, orc, "M%d N%d K%d mode%d" % (M, N, K, mode))
    return d


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (1, 256, 256), (127, 256, 384), (129, 384, 512),
                                   (300, 512, 1024), (256, 256, 2048), (640, 1280, 256)])
def test_gemm_block128_random(fb, orc, M, N, K, out_dtype):
    _run_random(fb, orc, M, N, K, 0, out_dtype, M + N + K)


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (200, 384, 512), (1, 128, 128)])
def test_gemm_rowscale_random(fb, orc, M, N, K, out_dtype):
    _run_random(fb, orc, M, N, K, 1, out_dtype, 7 * M + N + K)


def test_gemm_deterministic_and_no_overrun(fb, orc):
    M, N, K = 129, 384, 512
    a, b = rand_codes((M, K), 1), rand_codes((N, K), 2)
    sa, sb = rand_scales((K // 128, M), 3), rand_scales((N // 128, K // 128), 4)
    A, B, SA, SB = _dev(a), _dev(b), _dev(sa), _dev(sb)
    canary = torch.full((M * N + 4096,), -7.0, dtype=torch.bfloat16, device="cuda")
    d1 = canary[: M * N].view(M, N)
    fb.fp8_gemm_blockscaled(A, SA, B, SB, 0, torch.bfloat16, d=d1)
    d2 = fb.fp8_gemm_blockscaled(A, SA, B, SB, 0, torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(d1.view(torch.int16), d2.view(torch.int16))
    assert torch.all(canary[M * N:] == -7.0)
    assert fb.fp8_get_status() == 0


def test_gemm_tiny_dense_end_to_end(fb, orc):
    d = S.tiny_dense()
    x, w = d["x"], d["w"]
    qx, sx = fb.fp8_quant_act_1x128(x.cuda())
    qw, sw = fb.fp8_quant_weight_128x128(w.cuda())
    y = fb.fp8_gemm_blockscaled(qx, sx, qw, sw)
    qxr, sxr = orc.quant_act_1x128(S.bf16_bits(x))
    qwr, swr = orc.quant_weight_128x128(S.bf16_bits(w))
    ref = orc.gemm_blockscaled(qxr, sxr, qwr, swr, 0)
    assert_gemm_close(to_np(y), ref, True, orc, "tiny dense")


def test_gemm_dense_linear_full_sampled(fb, orc):
    """4096 x 7168 x 7168 through the GPU quantisers and GEMM; the oracle
    recomputes 48 rows x 3 column blocks from the bf16 inputs."""
    d = S.dense_linear()
    x, w = d["x"], d["w"]
    qx, sx = fb.fp8_quant_act_1x128(x.cuda())
    qw, sw = fb.fp8_quant_weight_128x128(w.cuda())
    y = fb.fp8_gemm_blockscaled(qx, sx, qw, sw)
    g = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, 4095], g.choice(4096, 46, replace=False)]))
    nbs = sorted({0, 55, int(g.integers(1, 55))})
    xb = S.bf16_bits(x)
    qa, sa = orc.quant_act_1x128(xb[rows])
    got = to_np(y)[rows]
    for nb in nbs:
        wb = S.bf16_bits(w[nb * 128:(nb + 1) * 128])
        qb, sb = orc.quant_weight_128x128(wb)
        ref = orc.gemm_blockscaled(qa, sa, qb, sb, 0)
        assert_gemm_close(got[:, nb * 128:(nb + 1) * 128], ref, True, orc, "dense nb=%d" % nb)


def test_wgrad_full_sampled(fb, orc):
    """dW = dY^T X with 128x1 token tiles, fp32 out, K = 8192 tokens."""
    d = S.wgrad()
    dy, x = d["dy"], d["x"]
    qa, sa = fb.fp8_quant_act_128x1(dy.cuda())
    qb, sb = fb.fp8_quant_act_128x1(x.cuda())
    dw = fb.fp8_gemm_blockscaled(qa, sa, qb, sb, fb.FP8_BSCALE_ROW, torch.float32)
    g = np.random.default_rng(1)
    ii = np.unique(np.concatenate([[0, 7167], g.choice(7168, 30, replace=False)]))
    jj = np.unique(np.concatenate([[0, 7167], g.choice(7168, 200, replace=False)]))
    dyb, xb = S.bf16_bits(dy), S.bf16_bits(x)
    qar, sar = orc.quant_act_128x1(np.ascontiguousarray(dyb[:, ii]))
    qbr, sbr = orc.quant_act_128x1(np.ascontiguousarray(xb[:, jj]))
    ref = orc.gemm_blockscaled(qar, sar, qbr, sbr, 1)
    got = dw.cpu().numpy()[np.ix_(ii, jj)]
    assert_gemm_close(got, ref, False, orc, "wgrad")


def test_wait_timeout_selftest_reports_status(fb):
    assert fb.fp8_get_status() == 0
    fb.fp8_selftest_wait_timeout(20_000_000)          # 20 ms
    assert fb.fp8_get_status() == fb.FP8_ERR_TIMEOUT
    assert fb.fp8_get_status() == 0                    # cleared by the read
    x = torch.ones((4, 128), dtype=torch.bfloat16, device="cuda")
    q, s = fb.fp8_quant_act_1x128(x)                   # the context is still usable
    torch.cuda.synchronize()
    assert int(q[0, 0]) == 0x7E


@pytest.mark.parametrize("mode,out_dtype,K", [(0, torch.float32, 2048), (0, torch.bfloat16, 2048),
                                              (1, torch.float32, 2048), (1, torch.float32, 8192)])
def test_gemm_many_tiles_per_cluster_full_rows(fb, orc, mode, out_dtype, K):
    """Every output column of every 7th row, on a problem where each CTA pair
    walks several tiles and the pipeline rings wrap many times, run three times:
    a race between the MMA, the TMA refills and the promotion shows up here as
    scattered wrong elements that a few sampled columns can miss."""
    M, N = 2048, 4096
    a, b = rand_codes((M, K), 11), rand_codes((N, K), 12)
    sa = rand_scales((K // 128, M), 13)
    sb = rand_scales((N // 128, K // 128) if mode == 0 else (K // 128, N), 14)
    rows = np.arange(0, M, 7)
    ref = orc.gemm_blockscaled(a, sa, b, sb, mode, rows=rows, cols=np.arange(N))
    A, SA, B, SB = _dev(a), _dev(sa), _dev(b), _dev(sb)
    refmax = np.abs(ref).max()
    for rep in range(3):
        d = fb.fp8_gemm_blockscaled(A, SA, B, SB, mode, out_dtype)
        got = to_np(d)[rows]
        assert_gemm_close(got, ref, out_dtype == torch.bfloat16, orc, "many tiles mode%d K%d rep%d" % (mode, K, rep))
        # Element-wise, far tighter than the tolerance above: the fp32 sum of
        # at most 64 promoted K blocks is off by ~1e-6 of max|ref|, and a
        # bf16 output by one bf16 rounding on top.  A corrupted element (a
        # K block read from the wrong accumulator or stage) is off by far more.
        err = np.abs(got - ref)
        bound = 1e-5 * refmax + (np.abs(ref) * 2.0 ** -8 if out_dtype == torch.bfloat16 else 0.0)
        n_bad = int((err > bound).sum())
        assert n_bad == 0, "many tiles mode%d K%d rep%d: %d elements beyond the element-wise bound" % (mode, K, rep, n_bad)
