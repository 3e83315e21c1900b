"""GPU parity of the block-scaled GEMM when its last tiles are split along K
(the promotion passages of the tmdrlife.com and gnrental.net pages: the output is the sum over 128-element K blocks of the
promoted, scaled tensor-core partial sums; a split only regroups that fp32
sum into per-range sums that a second kernel adds in K order).

Checks: every column of every 7th row of a split problem against the
oracle's fp64 product; split against unsplit on a K = 7168 problem and on
the Wgrad shape (identical bits on the tiles computed whole, fp32
regrouping error on the split ones); small problems split over the whole
GPU, with ragged rows, half-used column tiles, canaries past D and two runs
bit-identical.
"""
import numpy as np
import pytest
import torch

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


def _operands(M, N, K, mode, seed):
    a, b = rand_codes((M, K), seed), rand_codes((N, K), seed + 1)
    sa = rand_scales((K // 128, M), seed + 2)
    sb = rand_scales((N // 128, K // 128) if mode == 0 else (K // 128, N), seed + 3)
    return a, sa, b, sb


def _elementwise_ok(got, ref, bf16_out):
    # fp32 sums of at most a few hundred promoted terms: ~1e-6 of max|ref|;
    # a bf16 output adds one rounding.  A slab added twice, missed, or read
    # from the wrong tile is off by far more.
    bound = 1e-5 * np.abs(ref).max() + (np.abs(ref) * 2.0 ** -8 if bf16_out else 0.0)
    return int((np.abs(got - ref) > bound).sum())


def test_workspace_size_reports_one_slab_per_sm_pair(fb):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert fb.lib.fp8_gemm_blockscaled_workspace_bytes(4096, 7168, 7168) == (sms // 2) * 256 * 256 * 4
    assert fb.lib.fp8_gemm_blockscaled_workspace_bytes(4096, 7168, 1024) == 0     # too short to split


def _split_mask(fb, M, N, K, form=0):
    """Where D comes from split tiles under the library's plan on this GPU."""
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    ws = fb.lib.fp8_gemm_blockscaled_workspace_bytes(M, N, K)
    split, tail0, _ = fb.fp8_gemm_split_plan(M, N, K, pairs, ws, form)
    bn = fb.fp8_gemm_tile_cols(form)
    num_m2 = (M + 255) // 256
    mask = np.zeros((M, N), dtype=bool)
    for w in range(tail0, num_m2 * ((N + bn - 1) // bn)) if split else ():
        r0, c0 = (w % num_m2) * 256, (w // num_m2) * bn
        mask[r0:r0 + 256, c0:c0 + bn] = True
    return split, mask


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_split_tail_full_rows(fb, orc, out_dtype):
    """4096 x 3840 x 2048: 16 x 15 tiles of 256 columns leave a short last
    wave on 74 SM pairs, which is split along K; every column of every 7th
    row is checked."""
    M, N, K = 4096, 3840, 2048
    split, mask = _split_mask(fb, M, N, K)
    assert split > 0 and mask.any()
    a, sa, b, sb = _operands(M, N, K, 0, 21)
    rows = np.arange(0, M, 7)
    ref = orc.gemm_blockscaled(a, sa, b, sb, 0, rows=rows, cols=np.arange(N))
    d = fb.fp8_gemm_blockscaled(_dev(a), _dev(sa), _dev(b), _dev(sb), 0, out_dtype)
    assert fb.fp8_get_status() == 0
    got = to_np(d)[rows]
    bf16 = out_dtype == torch.bfloat16
    assert_gemm_close(got, ref, bf16, orc, "split tail")
    assert _elementwise_ok(got, ref, bf16) == 0


@pytest.mark.parametrize("M,N,K,mode", [(4096, 3840, 7168, 0), (4096, 3840, 8192, 1)])
def test_split_matches_unsplit(fb, M, N, K, mode):
    """K = 7168 (block B scales) and K = 8192 (per-row B scales, the Wgrad
    form) problems whose last wave is split: the tiles computed whole are
    bit-identical with and without the workspace; the split tiles agree
    within fp32 regrouping."""
    split, tail = _split_mask(fb, M, N, K)
    assert split > 0 and tail.any()
    a, sa, b, sb = _operands(M, N, K, mode, 33)
    A, SA, B, SB = _dev(a), _dev(sa), _dev(b), _dev(sb)
    d_split = fb.fp8_gemm_blockscaled(A, SA, B, SB, mode, torch.float32).cpu().numpy()
    d_whole = fb.fp8_gemm_blockscaled(A, SA, B, SB, mode, torch.float32, split=False).cpu().numpy()
    assert fb.fp8_get_status() == 0
    assert np.array_equal(d_split[~tail].view(np.uint32), d_whole[~tail].view(np.uint32))
    diff = np.abs(d_split[tail] - d_whole[tail])
    assert diff.max() <= 1e-5 * np.abs(d_whole).max(), diff.max()


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("M,N,K", [(1, 256, 2048), (129, 384, 2048), (300, 384, 4096), (513, 768, 2048),
                                   (640, 1280, 4096)])
def test_small_problems_split_over_the_gpu(fb, orc, M, N, K, mode, out_dtype):
    a, sa, b, sb = _operands(M, N, K, mode, 5 * M + N + K + mode)
    A, SA, B, SB = _dev(a), _dev(sa), _dev(b), _dev(sb)
    esz = 4 if out_dtype == torch.float32 else 2
    canary = torch.full((M * N + 8192,), -7.0, dtype=out_dtype, device="cuda")
    d1 = canary[: M * N].view(M, N)
    fb.fp8_gemm_blockscaled(A, SA, B, SB, mode, out_dtype, d=d1)
    d2 = fb.fp8_gemm_blockscaled(A, SA, B, SB, mode, out_dtype)
    torch.cuda.synchronize()
    assert fb.fp8_get_status() == 0
    view = torch.int32 if esz == 4 else torch.int16
    assert torch.equal(d1.view(view), d2.view(view)), "two runs differ"
    assert torch.all(canary[M * N:] == -7.0), "write past D"
    ref = orc.gemm_blockscaled(a, sa, b, sb, mode)
    bf16 = out_dtype == torch.bfloat16
    got = to_np(d1)
    assert_gemm_close(got, ref, bf16, orc, "split M%d N%d K%d mode%d" % (M, N, K, mode))
    assert _elementwise_ok(got, ref, bf16) == 0


def test_released_workspaces_are_allocated_again(fb):
    a, sa, b, sb = _operands(256, 256, 2048, 0, 3)
    A, SA, B, SB = _dev(a), _dev(sa), _dev(b), _dev(sb)
    d1 = fb.fp8_gemm_blockscaled(A, SA, B, SB, 0, torch.float32)
    assert fb.release_gemm_workspaces() >= 1
    assert fb.release_gemm_workspaces() == 0
    d2 = fb.fp8_gemm_blockscaled(A, SA, B, SB, 0, torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(d1.view(torch.int32), d2.view(torch.int32))
    assert fb.fp8_get_status() == 0
