"""GPU parity of fp8_linear_host, the dense FP8 linear layer called with host
buffers (the jp-study.kr page: 1x128 activation tiles and 128x128 weight
blocks; the tmdrlife.com page: per-interval promotion into FP32 with the two
scales): Y copied back to host memory against the oracle quantising the same
bf16 X and W itself and forming the fp64 product of those codes and scales."""
import numpy as np
import pytest
import torch

from fp8_fine_grained_16_b300 import synthetic as S
from _checks import assert_gemm_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fb():
    from fp8_fine_grained_16_b300 import build
    build.build()
    from fp8_fine_grained_16_b300 import fp8bs
    return fp8bs


def _bf16(shape, seed, scale=1.0):
    return (torch.randn(shape, generator=torch.Generator().manual_seed(seed)) * scale).to(torch.bfloat16)


def _oracle_rows(orc, x, w, rows, flags, col_blocks=None):
    """The oracle's Y on the given rows: X rows quantised 1x128, W quantised
    128x128 (only the 128-row blocks of W in col_blocks, if given)."""
    qa, sa = orc.quant_act_1x128(S.bf16_bits(x)[rows], flags)
    wb = S.bf16_bits(w)
    blocks = range(w.shape[0] // 128) if col_blocks is None else col_blocks
    out = {}
    for nb in blocks:
        qb, sb = orc.quant_weight_128x128(np.ascontiguousarray(wb[nb * 128:(nb + 1) * 128]), flags)
        out[nb] = orc.gemm_blockscaled(qa, sa, qb, sb, 0)
    return out


@pytest.mark.parametrize("flags", [0, 1])
@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (129, 640, 384), (256, 1536, 1024), (300, 2560, 512)])
def test_linear_host_matches_oracle(fb, orc, M, N, K, flags):
    """Every element, for one chunk, a chunk plus a ragged last chunk (1536 =
    1024 + 512) and three chunks (2560); pinned inputs, the output allocated
    by the binding (page-locked)."""
    x, w = _bf16((M, K), M + N, 2.0).pin_memory(), _bf16((N, K), K, 0.02).pin_memory()
    y = fb.fp8_linear_host(x, w, flags=flags)
    torch.cuda.synchronize()
    assert fb.fp8_get_status() == 0
    ref = _oracle_rows(orc, x, w, np.arange(M), flags)
    got = y.float().numpy()
    for nb, r in ref.items():
        assert_gemm_close(got[:, nb * 128:(nb + 1) * 128], r, True, orc, "M%d N%d K%d col block %d" % (M, N, K, nb))


def test_linear_host_pageable_buffers_and_reuse(fb, orc):
    """Pageable host tensors work (the copies serialise), and a second call on
    the same workspace with other data gives its own result."""
    M, N, K = 200, 1024, 640
    y = torch.empty((M, N), dtype=torch.bfloat16)
    for seed in (1, 2):
        x, w = _bf16((M, K), seed), _bf16((N, K), seed + 10, 0.02)
        fb.fp8_linear_host(x, w, y)
        torch.cuda.synchronize()
        ref = _oracle_rows(orc, x, w, np.arange(M), 0, col_blocks=[0, 7])
        for nb, r in ref.items():
            assert_gemm_close(y.float().numpy()[:, nb * 128:(nb + 1) * 128], r, True, orc, "seed %d block %d" % (seed, nb))
    assert fb.fp8_get_status() == 0


def test_linear_host_equals_device_path_on_unsplit_chunk(fb):
    """One 1024-column chunk whose GEMM is not split (K below the split's
    minimum): the host-buffer call must give exactly the bits of the same
    three calls on device tensors."""
    M, N, K = 512, 1024, 1024
    x, w = _bf16((M, K), 5).pin_memory(), _bf16((N, K), 6, 0.02).pin_memory()
    y = fb.fp8_linear_host(x, w)
    xd, wd = x.cuda(), w.cuda()
    qx, sx = fb.fp8_quant_act_1x128(xd)
    qw, sw = fb.fp8_quant_weight_128x128(wd)
    yd = fb.fp8_gemm_blockscaled(qx, sx, qw, sw)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), yd.cpu().view(torch.int16))


def test_linear_host_dense_linear_sampled(fb, orc):
    """The dense-linear workload (X [4096,7168] 0.5*t(3), W [7168,7168]) from
    host memory, in the chunking the bench times: sampled rows and column
    blocks against the oracle."""
    d = S.dense_linear()
    x, w = d["x"].pin_memory(), d["w"].pin_memory()
    y = fb.fp8_linear_host(x, w)
    torch.cuda.synchronize()
    assert fb.fp8_get_status() == 0
    g = np.random.default_rng(11)
    rows = np.unique(np.concatenate([[0, 4095], g.choice(4096, 24, replace=False)]))
    ref = _oracle_rows(orc, x, w, rows, 0, col_blocks=[0, 7, 8, 31, 55])
    got = y.float().numpy()[rows]
    for nb, r in ref.items():
        assert_gemm_close(got[:, nb * 128:(nb + 1) * 128], r, True, orc, "dense linear col block %d" % nb)
