"""Shared parity checks for the GPU tests.

GEMM tolerance (stated for this path): against the oracle's fp64 product of
the same E4M3 operands and scales, relative Frobenius error <= 1e-3 and
max |err| <= 2e-2 * max |ref|.  For bf16 outputs the reference is the fp64
result rounded once to bf16: the bf16 rounding alone is ~1.7e-3 relative
Frobenius, which would exceed the bound before any arithmetic error.
"""
import numpy as np
import torch

REL_FRO = 1e-3
MAX_ABS_FRAC = 2e-2


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().to("cpu")
    if t.dtype == torch.bfloat16:
        return t.float().numpy().astype(np.float64)
    return t.numpy()


def gemm_errors(got: np.ndarray, ref64: np.ndarray, bf16_out: bool, orc):
    ref = ref64
    if bf16_out:
        ref = torch.from_numpy(orc.round_bf16(ref64).view(np.int16)).view(torch.bfloat16).double().numpy()
    err = got.astype(np.float64) - ref
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(err) / nref if nref > 0 else np.linalg.norm(err)
    mx = np.abs(err).max() if err.size else 0.0
    return rel, mx, np.abs(ref).max() if ref.size else 0.0


def assert_gemm_close(got, ref64, bf16_out, orc, what=""):
    rel, mx, refmax = gemm_errors(got, ref64, bf16_out, orc)
    print("%s rel_fro=%.3e max_abs=%.3e (max|ref| %.3e)" % (what, rel, mx, refmax))
    assert rel <= REL_FRO, (what, rel)
    assert mx <= MAX_ABS_FRAC * refmax, (what, mx, refmax)


def assert_same_bits(got: torch.Tensor, ref: np.ndarray, what=""):
    g = got.detach().to("cpu").contiguous().numpy()
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    if g.dtype == np.float32:
        g = g.view(np.uint32)
        ref = np.ascontiguousarray(ref).view(np.uint32)
    bad = np.argwhere(g != ref)
    assert bad.size == 0, "%s: %d mismatches, first at %s (got %s want %s)" % (
        what, len(bad), tuple(bad[0]), g[tuple(bad[0])], ref[tuple(bad[0])])


def rand_codes(shape, seed):
    """Random E4M3 codes, NaN codes excluded."""
    g = np.random.default_rng(seed)
    c = g.integers(0, 256, size=shape, dtype=np.int64).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x3C
    return c


def rand_scales(shape, seed, lo=1e-3, hi=4.0):
    g = np.random.default_rng(seed)
    return np.exp(g.uniform(np.log(lo), np.log(hi), size=shape)).astype(np.float32)


# ---------------------------------------------------------------- SwiGLU + 1x128 against float64
def swiglu_fp64(y: torch.Tensor, I: int) -> np.ndarray:
    """h = g / (1 + e^-g) * u in float64 with libm's exp (numpy), g = y[:, :I],
    u = y[:, I:2I]: the plain definition, sharing no step with either fp32
    recipe."""
    yf = y[:, :2 * I].double().numpy()
    g, u = yf[:, :I], yf[:, I:]
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g)) * u


def check_swiglu_quant_against_fp64(q, s, y, I, flags, orc, near=2.0 ** -18):
    """Codes q [R, I] and scales s [I/128, R] of SwiGLU + 1x128 quantisation,
    held to the float64 definition followed by the oracle's pinned fp32 tile
    rule (h rounded once to fp32).  An fp32 SwiGLU differs from that h by a
    few ulps, so an element may take the neighbouring code where h * inv lies
    within `near` (relative) of the midpoint between two codes, and a tile may
    take the neighbouring power-of-two scale where its max-abs lies within
    `near` of 448 * 2^e.  Everything else must match bit for bit.  In default
    mode the scale amax/448 follows the last bits of the tile's max-abs, so a
    tile whose scale differs is held to the scale within `near` and to the
    per-element dequantisation bound instead.  Returns (code mismatches that
    sat at a midpoint, tiles with a different scale)."""
    q = np.asarray(q)
    s = np.asarray(s, dtype=np.float32)
    h64 = swiglu_fp64(y, I)
    R = h64.shape[0]
    q_ref, s_ref = orc.quant_act_1x128_f32(h64.astype(np.float32), flags)
    tab = orc.e4m3_decode(np.arange(256, dtype=np.uint8))
    s_tiles = s.T.reshape(R, I // 128)                      # [R, tiles]
    r_tiles = s_ref.T.reshape(R, I // 128)
    same_scale = s_tiles.view(np.uint32) == r_tiles.view(np.uint32)
    amax = np.abs(h64).reshape(R, I // 128, 128).max(axis=2)
    if flags & 1:
        # a different power of two only where the max-abs sits on 448 * 2^e
        bad = ~same_scale
        if bad.any():
            a = amax[bad]
            e = np.round(np.log2(np.maximum(a, 1e-300) / 448.0))
            assert np.all(np.abs(a / (448.0 * 2.0 ** e) - 1.0) <= near), "pow-2 scale off a boundary"
    else:
        assert np.all(np.abs(s_tiles.astype(np.float64) / r_tiles - 1.0) <= near), "scale beyond the fp32 slack"
    # codes in tiles whose scale matches: equal, or neighbours at a midpoint
    qt, qr = q.reshape(R, I // 128, 128), q_ref.reshape(R, I // 128, 128)
    inv = 1.0 / r_tiles.astype(np.float64)
    x = h64.reshape(R, I // 128, 128) * inv[..., None]
    diff = (qt != qr) & same_scale[..., None]
    n_mid = int(diff.sum())
    if n_mid:
        cg, cr, xv = qt[diff], qr[diff], x[diff]
        vg, vr = tab[cg], tab[cr]
        zero = (vg == 0) & (vr == 0)                         # +0 against -0 of a value that underflows
        assert np.all(zero | ((cg & 0x80) == (cr & 0x80))), "sign differs"
        step = np.abs((cg & 0x7F).astype(np.int64) - (cr & 0x7F).astype(np.int64))
        assert np.all(zero | (step == 1)), "codes are not neighbours"
        mid = 0.5 * (vg + vr)
        assert np.all(zero | (np.abs(xv - mid) <= near * np.abs(mid))), "neighbour code away from a midpoint"
    # tiles with another scale (default mode): each element within half an E4M3 step
    other = ~same_scale
    if other.any():
        st = np.repeat(s_tiles.astype(np.float64), 128, axis=1)
        deq = tab[q] * st
        err = np.abs(deq - h64)
        bound = (np.maximum(np.abs(h64) * 2.0 ** -4, st * 2.0 ** -10)) * (1 + near) + np.abs(h64) * near
        rows_other = np.repeat(other, 128, axis=1)
        assert np.all(err[rows_other] <= bound[rows_other]), "dequantisation bound"
    return n_mid, int(other.sum())
