"""fp8_moe_route_topk_noalloc: routing for callers that cannot allocate.

Some callers cannot allocate device memory at the point where they route
tokens (a runtime that gave all of HBM to its own pool at start-up, or a
serving loop that bans cudaMalloc after warm-up because allocating can
synchronise the device).  For them the library offers a routing call whose
scratch is a fixed array inside the library.  These tests call it through
the C ABI, with every output buffer allocated up front, and check that it
gives the same routes as fp8_moe_route_topk with a caller-provided `work`
buffer, on two calls in a row: the second call, on a smaller problem, finds
the first call's counts still in the shared array and must not be misled by
them.

This file is named so that pytest collects it after every other test file.
"""
import numpy as np
import pytest
import torch

from fp8_fine_grained_16_b300 import synthetic as S

pytestmark = pytest.mark.gpu

GATE_RTOL, GATE_ATOL = 2e-6, 1e-7      # the gate tolerance of the routing tests


@pytest.fixture(scope="module")
def fb():
    from fp8_fine_grained_16_b300 import build
    build.build()
    from fp8_fine_grained_16_b300 import fp8bs
    return fp8bs


def _outputs(T, E, k, dev):
    return dict(idx=torch.empty((T, k), dtype=torch.int32, device=dev),
                gate=torch.empty((T, k), dtype=torch.float32, device=dev),
                off=torch.empty(E + 1, dtype=torch.int32, device=dev),
                src_row=torch.empty(T * k, dtype=torch.int32, device=dev),
                pos=torch.empty((T, k), dtype=torch.int32, device=dev))


def _same_routes(got, want):
    for key in ("idx", "off", "src_row", "pos"):
        assert torch.equal(got[key], want[key]), key
    assert torch.allclose(got["gate"], want["gate"], rtol=GATE_RTOL, atol=GATE_ATOL)


def test_noalloc_route_matches_route_with_workspace_twice(fb):
    dev = torch.device("cuda", 0)
    cases = [(S.moe_up(with_weights=False)["logits"], 8),           # 4096 tokens, 256 experts, top-8
             (torch.randn((300, 64), generator=torch.Generator().manual_seed(5)), 5)]
    prepared = []
    for logits, k in cases:
        T, E = logits.shape
        lg = logits.to(dev)
        work = torch.empty(fb.fp8_moe_route_workspace_size(T, E) // 4, dtype=torch.int32, device=dev)
        prepared.append((lg, k, _outputs(T, E, k, dev), _outputs(T, E, k, dev), work))
    torch.cuda.synchronize()
    # two no-alloc calls in a row, then the reference calls with their own work buffers
    for lg, k, out_na, _, _ in prepared:
        fb.fp8_moe_route_topk_noalloc(lg, k, out=out_na)
    for lg, k, _, out_ref, work in prepared:
        fb.fp8_moe_route_topk(lg, k, out=out_ref, work=work)
    torch.cuda.synchronize()
    assert fb.fp8_get_status() == 0
    for _, _, out_na, out_ref, _ in prepared:
        _same_routes(out_na, out_ref)
    # the routes are also valid: every token appears k times, offsets end at T*k
    for lg, k, out_na, _, _ in prepared:
        T = lg.shape[0]
        assert int(out_na["off"][-1]) == T * k
        counts = np.bincount(out_na["src_row"].cpu().numpy(), minlength=T)
        assert np.all(counts == k)


def test_noalloc_route_rejects_problems_beyond_its_scratch(fb):
    T, E = 64 * (2 ** 18 // 256) + 1, 256          # one chunk more than the array holds
    lib = fb.lib
    fake = 1 << 40                                  # never dereferenced: the size check comes first
    rc = lib.fp8_moe_route_topk_noalloc(fake, T, E, 8, fake, fake, fake, fake, fake, None)
    assert rc == fb.FP8_ERR_SCRATCH
    assert "static scratch" in fb.fp8_strerror(rc)
