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
