"""The C-ABI library loads without a GPU, exports every entry point the
header declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8bs.h")


@pytest.fixture(scope="module")
def fb():
    from fp8_fine_grained_16_b300 import build
    build.build()
    from fp8_fine_grained_16_b300 import fp8bs
    return fp8bs


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^FP8_API\s+[\w\s\*]+?\b(fp8_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_five_hot_path_calls():
    syms = declared_symbols()
    for name in ["fp8_quant_act_1x128", "fp8_quant_act_128x1", "fp8_quant_weight_128x128",
                 "fp8_gemm_blockscaled", "fp8_grouped_gemm_blockscaled"]:
        assert name in syms


def test_library_exports_every_declared_symbol(fb):
    syms = declared_symbols()
    assert syms == fb.EXPORTED
    lib = ctypes.CDLL(fb.LIB_PATH)
    for s in syms:
        assert hasattr(lib, s), s


def test_version_and_strerror(fb):
    assert fb.fp8_version() == 100
    assert fb.fp8_strerror(0) == "ok"
    assert "timed out" in fb.fp8_strerror(-5)
    assert fb.fp8_strerror(12345) == "unknown status"


def test_workspace_size(fb):
    assert fb.fp8_moe_route_workspace_size(4096, 256) == 64 * 256 * 4
    assert fb.fp8_moe_route_workspace_size(65, 8) == 2 * 8 * 4
    assert fb.fp8_moe_route_workspace_size(0, 8) == 0


# Argument checks run on the host before any CUDA call, so they are testable
# here; a fake but aligned device address stands in for real buffers.
FAKE = 1 << 40


def test_quant_argument_errors(fb):
    L = fb.lib
    assert L.fp8_quant_act_1x128(None, 4, 128, 128, FAKE, FAKE, 0, None) == -1          # null x
    assert L.fp8_quant_act_1x128(FAKE, 0, 128, 128, FAKE, FAKE, 0, None) == -1          # M = 0
    assert L.fp8_quant_act_1x128(FAKE, 4, 100, 100, FAKE, FAKE, 0, None) == -2          # K % 128
    assert L.fp8_quant_act_1x128(FAKE + 2, 4, 128, 128, FAKE, FAKE, 0, None) == -3      # misaligned x
    assert L.fp8_quant_act_1x128(FAKE, 4, 128, 130, FAKE, FAKE, 0, None) == -3          # ldx % 8
    assert L.fp8_quant_act_1x128(FAKE, 4, 128, 128, FAKE, FAKE, 6, None) == -1          # unknown flag
    assert L.fp8_quant_act_128x1(FAKE, 100, 64, 64, FAKE, FAKE, 0, None) == -2          # T % 128
    assert L.fp8_quant_act_128x1(FAKE, 128, 12, 12, FAKE, FAKE, 0, None) == -2          # H % 8
    assert L.fp8_quant_weight_128x128(FAKE, 100, 128, 128, FAKE, FAKE, 0, None) == -2   # N % 128
    aw = L.fp8_quant_act_weight      # x, M, ldx, qx, sx, w, N, ldw, qw, sw, K, flags, stream
    assert aw(FAKE, 4, 128, FAKE, FAKE, None, 128, 128, FAKE, FAKE, 128, 0, None) == -1     # null w
    assert aw(FAKE, 0, 128, FAKE, FAKE, FAKE, 128, 128, FAKE, FAKE, 128, 0, None) == -1     # M = 0
    assert aw(FAKE, 4, 128, FAKE, FAKE, FAKE, 128, 120, FAKE, FAKE, 128, 0, None) == -1     # ldw < K
    assert aw(FAKE, 4, 128, FAKE, FAKE, FAKE, 100, 128, FAKE, FAKE, 128, 0, None) == -2     # N % 128
    assert aw(FAKE, 4, 200, FAKE, FAKE, FAKE, 128, 200, FAKE, FAKE, 200, 0, None) == -2     # K % 128
    assert aw(FAKE, 4, 128, FAKE, FAKE, FAKE + 8, 128, 128, FAKE, FAKE, 128, 0, None) == -3  # misaligned w
    assert aw(FAKE, 4, 128, FAKE, FAKE, FAKE, 128, 132, FAKE, FAKE, 128, 0, None) == -3     # ldw % 8
    assert aw(FAKE, 4, 128, FAKE, FAKE, FAKE, 128, 128, FAKE, FAKE, 128, 4, None) == -1     # unknown flag
    assert L.fp8_cast_e4m3(None, 5, FAKE, None) == -1
    assert L.fp8_cast_e4m3(None, 0, None, None) == 0                                    # empty: no-op


def test_gemm_argument_errors(fb):
    L = fb.lib
    base = dict(a=FAKE, sa=FAKE, b=FAKE, sb=FAKE, mode=0, d=FAKE, dt=0, M=128, N=256, K=256, st=None)

    def call(**kw):
        a = dict(base, **kw)
        return L.fp8_gemm_blockscaled(*a.values())

    assert call(a=None) == -1
    assert call(mode=2) == -1
    assert call(dt=7) == -1
    assert call(K=200) == -2
    assert call(N=200) == -2
    assert call(d=FAKE + 4) == -3
    assert call(M=0) == -1
    w = L.fp8_gemm_blockscaled_ws
    assert w(None, FAKE, FAKE, FAKE, 0, FAKE, 0, 128, 256, 4096, FAKE, 1 << 20, None) == -1  # null a
    assert w(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 0, 128, 256, 4096, None, 1 << 20, None) == -1  # size, no pointer
    assert w(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 0, 128, 256, 4096, FAKE, -1, None) == -1       # negative size
    assert w(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 0, 128, 256, 4096, FAKE + 8, 1 << 20, None) == -3  # misaligned
    assert w(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 0, 128, 256, 200, FAKE, 1 << 20, None) == -2   # K % 128
    assert L.fp8_gemm_blockscaled_workspace_bytes(0, 256, 4096) == -1
    g = fb.lib.fp8_grouped_gemm_blockscaled
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 10, 256, 256, FAKE, None) == -1            # E = 0
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, 2000, 10, 256, 256, FAKE, None) == -1         # E too large
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 10, 256, 200, FAKE, None) == -2            # K % 128
    assert g(None, None, FAKE, FAKE, FAKE, 4, 0, 256, 256, None, None) == 0              # no rows: no-op


def test_moe_argument_errors(fb):
    L = fb.lib
    assert L.fp8_moe_route_topk(FAKE, 16, 8, 9, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None) == -1   # topk > E
    assert L.fp8_moe_route_topk(FAKE, 16, 2048, 8, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None) == -1
    assert L.fp8_moe_route_topk(FAKE + 2, 16, 8, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None) == -3
    assert L.fp8_permute_rows(FAKE, FAKE, 10, 100, FAKE, 5, FAKE, FAKE, None) == -2
    assert L.fp8_permute_rows(None, None, 10, 128, None, 0, None, None, None) == 0
    assert L.fp8_moe_combine_bf16(FAKE, 10, FAKE, FAKE, 4, 2, 12, FAKE, None) == -2
    assert L.fp8_selftest_wait_timeout(0, None) == -1


def test_pow2_and_fused_entry_point_argument_errors(fb):
    L = fb.lib
    # power-of-two GEMM: the argument rules of fp8_gemm_blockscaled
    p = L.fp8_gemm_blockscaled_pow2
    assert p(None, FAKE, FAKE, FAKE, 0, FAKE, 0, 128, 256, 256, None) == -1                  # null a
    assert p(FAKE, FAKE, FAKE, FAKE, 3, FAKE, 0, 128, 256, 256, None) == -1                  # B-scale mode
    assert p(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 0, 128, 200, 256, None) == -2                  # N % 128
    assert p(FAKE, FAKE, FAKE, FAKE, 0, FAKE + 4, 0, 128, 256, 256, None) == -3              # misaligned d
    gp = L.fp8_grouped_gemm_blockscaled_pow2
    assert gp(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 10, 256, 256, FAKE, None) == -1               # E = 0
    assert gp(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 10, 256, 200, FAKE, None) == -2               # K % 128
    assert gp(None, None, FAKE, FAKE, FAKE, 4, 0, 256, 256, None, None) == 0                 # no rows: no-op
    # quantised epilogue
    q = L.fp8_gemm_blockscaled_q8
    assert q(FAKE, FAKE, FAKE, FAKE, 0, None, FAKE, 0, 128, 256, 256, None) == -1            # null q_out
    assert q(FAKE, FAKE, FAKE, FAKE, 0, FAKE, FAKE, 4, 128, 256, 256, None) == -1            # unknown flag
    assert q(FAKE, FAKE, FAKE, FAKE, 0, FAKE, FAKE, 0, 128, 256, 100, None) == -2            # K % 128
    assert q(FAKE, FAKE, FAKE, FAKE, 0, FAKE + 8, FAKE, 0, 128, 256, 256, None) == -3        # misaligned q_out
    assert q(FAKE, FAKE, FAKE, FAKE, 0, FAKE, FAKE + 2, 0, 128, 256, 256, None) == -3        # misaligned s_out
    qw = L.fp8_gemm_blockscaled_q8_ws
    assert qw(FAKE, FAKE, FAKE, FAKE, 0, FAKE, FAKE, 0, 128, 256, 4096, None, 64, None) == -1    # size, no pointer
    assert qw(FAKE, FAKE, FAKE, FAKE, 0, FAKE, FAKE, 0, 128, 256, 4096, FAKE + 4, 64, None) == -3  # misaligned
    assert qw(FAKE, FAKE, FAKE, FAKE, 0, None, FAKE, 0, 128, 256, 4096, FAKE, 64, None) == -1    # null q_out
    # SwiGLU + quantisation
    s = L.fp8_swiglu_quant_1x128
    assert s(FAKE, 4, 128, 255, FAKE, FAKE, 1, None) == -1                                   # ldy < 2I
    assert s(FAKE, 4, 100, 200, FAKE, FAKE, 1, None) == -2                                   # I % 128
    assert s(FAKE, 4, 128, 260, FAKE, FAKE, 1, None) == -3                                   # ldy % 8
    assert s(FAKE, 0, 128, 256, FAKE, FAKE, 1, None) == -1                                   # R = 0
    assert s(FAKE, 4, 128, 256, FAKE, FAKE, 2, None) == -1                                   # unknown flag
    # transposed copy for Dgrad
    t = L.fp8_transpose_128x128
    assert t(FAKE, FAKE, 100, 128, FAKE, FAKE, None) == -2                                   # N % 128
    assert t(FAKE + 4, FAKE, 128, 128, FAKE, FAKE, None) == -3                               # misaligned q
    assert t(None, FAKE, 128, 128, FAKE, FAKE, None) == -1
    assert t(FAKE, FAKE, 1 << 31, 128, FAKE, FAKE, None) == -2                              # N past int32 coordinates
    # reciprocal self-test: d >= 1 only, and an aligned counter
    rs = L.fp8_selftest_reciprocal
    assert rs(0x3F7FFFFF, 0x3F800000, FAKE, None) == -1                                       # d < 1
    assert rs(0x3F800001, 0x3F800000, FAKE, None) == -1                                       # empty range
    assert rs(0x3F800000, 0x3F800001, FAKE + 4, None) == -3                                   # misaligned counter
    # dense linear from host buffers: argument checks come before any device access
    lh = L.fp8_linear_host
    assert lh(None, FAKE, 128, 128, 128, FAKE, 0, FAKE, 1 << 30, None) == -1                 # null x_h
    assert lh(FAKE, FAKE, 128, 128, 128, FAKE, 0, None, 1 << 30, None) == -1                 # no workspace
    assert lh(FAKE, FAKE, 0, 128, 128, FAKE, 0, FAKE, 1 << 30, None) == -1                   # M = 0
    assert lh(FAKE, FAKE, 128, 128, 128, FAKE, 2, FAKE, 1 << 30, None) == -1                 # unknown flag
    assert lh(FAKE, FAKE, 128, 100, 128, FAKE, 0, FAKE, 1 << 30, None) == -2                 # N % 128
    assert lh(FAKE, FAKE, 128, 128, 128, FAKE, 0, FAKE + 16, 1 << 30, None) == -3            # workspace not 256-aligned
    assert L.fp8_linear_host_workspace_bytes(0, 128, 128) == -1
    assert L.fp8_linear_host_workspace_bytes(128, 128, 100) == -2
    assert "power of two" in fb.fp8_strerror(fb.FP8_ERR_SCALE)


def test_releasing_no_gemm_workspaces_needs_no_gpu(fb):
    fb.release_gemm_workspaces()          # whatever earlier tests in this process cached
    assert fb.release_gemm_workspaces() == 0


def test_releasing_workspaces_waits_for_every_device_that_holds_one(fb):
    """The split workspaces are keyed by (device, stream); before any goes
    back to the caching allocator, every device holding one is waited for,
    not only the current device (a GEMM queued on another GPU may still use
    its workspace)."""
    synced = []
    saved = dict(fb._GEMM_WS)
    fb._GEMM_WS.clear()
    try:
        fb._GEMM_WS.update({(0, 11): "ws0", (3, 12): "ws3a", (3, 15): "ws3b", (6, 0): "ws6"})
        assert fb.release_gemm_workspaces(_synchronize=synced.append) == 4
        assert synced == [0, 3, 6]
        assert not fb._GEMM_WS
    finally:
        fb._GEMM_WS.clear()
        fb._GEMM_WS.update(saved)
