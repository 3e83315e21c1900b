"""CPU oracle for the fine-grained FP8 path -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never calls it,
and it shares no code with the CUDA kernels: the arithmetic lives in
``fp8_oracle.c`` (plain C, fp64 where the pages fix no precision), and this
module only moves numpy arrays in and out.

bf16 tensors cross this boundary as ``uint16`` arrays holding the raw bits.

Function by function, what pins it (see ``tests/test_oracle_*.py``):
  e4m3_decode / e4m3_encode   all 256 codes against torch's float8_e4m3fn and
                              hand-derived values; all 2^32 fp32 inputs against
                              an independent nearest-value search
  tile_scale                  closed forms (amax -> +-448, exact powers of two)
  quant_*                     hand-worked tiles, amax->448 invariant, the
                              dequantisation error bound, tile locality
  gemm_*                      exact integer block sums, integer matmul special
                              case, one-hot B
  route_topk / permute_rows   brute-force top-k, counting invariants
  moe_combine                 one-hot gates reduce it to a gather
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
          "-fno-fast-math", "-frounding-math", "-fno-builtin"]

FLAG_POW2 = 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/liboracle.so``."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _declare(_lib)
    return _lib


P = ctypes.c_void_p
I64 = ctypes.c_int64
U32 = ctypes.c_uint32
INT = ctypes.c_int


def _declare(L):
    L.orc_e4m3_decode.restype = ctypes.c_double
    L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
    L.orc_e4m3_encode.restype = ctypes.c_uint8
    L.orc_e4m3_encode.argtypes = [ctypes.c_float]
    L.orc_e4m3_encode_array.argtypes = [P, I64, P]
    L.orc_e4m3_encode_bits.argtypes = [ctypes.c_uint64, I64, P]
    L.orc_tile_scale.restype = ctypes.c_float
    L.orc_tile_scale.argtypes = [ctypes.c_float, U32, ctypes.POINTER(ctypes.c_float)]
    L.orc_quant_act_1x128.argtypes = [P, I64, I64, I64, P, P, U32]
    L.orc_quant_act_1x128_f32.argtypes = [P, I64, I64, P, P, U32]
    L.orc_exp_cw.restype = ctypes.c_float
    L.orc_exp_cw.argtypes = [ctypes.c_float]
    L.orc_swiglu_f32.argtypes = [P, I64, I64, I64, P]
    L.orc_swiglu_quant_1x128.argtypes = [P, I64, I64, I64, P, P, U32]
    L.orc_quant_act_128x1.argtypes = [P, I64, I64, I64, P, P, U32]
    L.orc_quant_weight_128x128.argtypes = [P, I64, I64, I64, P, P, U32]
    L.orc_gemm_blockscaled_at.argtypes = [P, P, P, P, INT, I64, I64, I64, P, I64, P, I64, P]
    L.orc_gemm_blockscaled.argtypes = [P, P, P, P, INT, I64, I64, I64, P]
    L.orc_route_topk.argtypes = [P, I64, INT, INT, P, P, P, P, P]
    L.orc_permute_rows.argtypes = [P, P, I64, I64, P, I64, P, P]
    L.orc_grouped_gemm_at.argtypes = [P, P, P, P, P, INT, I64, I64, I64, P, I64, P, I64, P]
    L.orc_moe_combine.argtypes = [P, P, P, I64, INT, I64, P]
    L.orc_round_bf16.argtypes = [P, I64, P]
    L.orc_bf16_to_float.argtypes = [P, I64, P]
    L.orc_max_threads.restype = INT
    L.orc_set_threads.argtypes = [INT]
    L.orc_rounding_is_nearest.restype = INT


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    return lib().orc_max_threads()


def set_threads(n: int) -> None:
    lib().orc_set_threads(n)


# ---------------------------------------------------------------- codec
def e4m3_decode(codes) -> np.ndarray:
    c = _c(codes, np.uint8)
    return np.array([lib().orc_e4m3_decode(int(v)) for v in c.ravel()], dtype=np.float64).reshape(c.shape)


def e4m3_encode(x) -> np.ndarray:
    x = _c(x, np.float32)
    q = np.empty(x.shape, np.uint8)
    lib().orc_e4m3_encode_array(_p(x), x.size, _p(q))
    return q


def e4m3_encode_bits(start: int, n: int) -> np.ndarray:
    q = np.empty(n, np.uint8)
    lib().orc_e4m3_encode_bits(start, n, _p(q))
    return q


def tile_scale(amax: float, flags: int = 0):
    inv = ctypes.c_float()
    s = lib().orc_tile_scale(amax, flags, ctypes.byref(inv))
    return np.float32(s), np.float32(inv.value)


# ---------------------------------------------------------------- bf16
def bf16_to_float(h) -> np.ndarray:
    h = _c(h, np.uint16)
    out = np.empty(h.shape, np.float32)
    lib().orc_bf16_to_float(_p(h), h.size, _p(out))
    return out


def round_bf16(d) -> np.ndarray:
    d = _c(d, np.float64)
    out = np.empty(d.shape, np.uint16)
    lib().orc_round_bf16(_p(d), d.size, _p(out))
    return out


# ---------------------------------------------------------------- quantisers
def quant_act_1x128(x, flags: int = 0):
    """x bf16 bits [M, K] -> (q uint8 [M, K], s float32 [K/128, M])."""
    x = _c(x, np.uint16)
    M, K = x.shape
    assert K % 128 == 0
    q = np.empty((M, K), np.uint8)
    s = np.empty((K // 128, M), np.float32)
    lib().orc_quant_act_1x128(_p(x), M, K, K, _p(q), _p(s), flags)
    return q, s


def quant_act_1x128_f32(x, flags: int = 0):
    """x float32 [M, K] -> (q uint8 [M, K], s float32 [K/128, M]): the 1x128
    tile rule on fp32 values (the quantisation a GEMM epilogue applies)."""
    x = _c(x, np.float32)
    M, K = x.shape
    assert K % 128 == 0
    q = np.empty((M, K), np.uint8)
    s = np.empty((K // 128, M), np.float32)
    lib().orc_quant_act_1x128_f32(_p(x), M, K, _p(q), _p(s), flags)
    return q, s


def exp_cw(x) -> np.ndarray:
    """The oracle's fp32 e^x (Cody-Waite reduction, degree-7 Taylor)."""
    x = _c(x, np.float32)
    return np.array([lib().orc_exp_cw(float(v)) for v in x.ravel()], dtype=np.float32).reshape(x.shape)


def swiglu_f32(y, I: int) -> np.ndarray:
    """y bf16 bits [R, >= 2I] (gate | up) -> h float32 [R, I] = SiLU(gate) * up in fp32 steps."""
    y = _c(y, np.uint16)
    R, ldy = y.shape
    h = np.empty((R, I), np.float32)
    lib().orc_swiglu_f32(_p(y), R, I, ldy, _p(h))
    return h


def swiglu_quant_1x128(y, I: int, flags: int = 0):
    """y bf16 bits [R, >= 2I] -> (q uint8 [R, I], s float32 [I/128, R])."""
    y = _c(y, np.uint16)
    R, ldy = y.shape
    assert I % 128 == 0 and ldy >= 2 * I
    q = np.empty((R, I), np.uint8)
    s = np.empty((I // 128, R), np.float32)
    lib().orc_swiglu_quant_1x128(_p(y), R, I, ldy, _p(q), _p(s), flags)
    return q, s


def quant_act_128x1(x, flags: int = 0):
    """x bf16 bits [T, H] -> (qT uint8 [H, T], s float32 [T/128, H])."""
    x = _c(x, np.uint16)
    T, H = x.shape
    assert T % 128 == 0
    q = np.empty((H, T), np.uint8)
    s = np.empty((T // 128, H), np.float32)
    lib().orc_quant_act_128x1(_p(x), T, H, H, _p(q), _p(s), flags)
    return q, s


def quant_weight_128x128(w, flags: int = 0):
    """w bf16 bits [N, K] -> (q uint8 [N, K], s float32 [N/128, K/128])."""
    w = _c(w, np.uint16)
    N, K = w.shape
    assert N % 128 == 0 and K % 128 == 0
    q = np.empty((N, K), np.uint8)
    s = np.empty((N // 128, K // 128), np.float32)
    lib().orc_quant_weight_128x128(_p(w), N, K, K, _p(q), _p(s), flags)
    return q, s


# ---------------------------------------------------------------- GEMMs
def gemm_blockscaled(a, sa, b, sb, b_mode: int = 0, rows=None, cols=None) -> np.ndarray:
    """fp64 D = dequant(a) @ dequant(b).T, optionally only at rows x cols."""
    a = _c(a, np.uint8); b = _c(b, np.uint8)
    sa = _c(sa, np.float32); sb = _c(sb, np.float32)
    M, K = a.shape
    N = b.shape[0]
    rows = np.arange(M, dtype=np.int64) if rows is None else _c(rows, np.int64)
    cols = np.arange(N, dtype=np.int64) if cols is None else _c(cols, np.int64)
    d = np.empty((rows.size, cols.size), np.float64)
    lib().orc_gemm_blockscaled_at(_p(a), _p(sa), _p(b), _p(sb), b_mode, M, N, K,
                                  _p(rows), rows.size, _p(cols), cols.size, _p(d))
    return d


def grouped_gemm_blockscaled(a, sa, b, sb, off, rows=None, cols=None) -> np.ndarray:
    a = _c(a, np.uint8); b = _c(b, np.uint8)
    sa = _c(sa, np.float32); sb = _c(sb, np.float32)
    off = _c(off, np.int32)
    total, K = a.shape
    E, N, _ = b.shape
    rows = np.arange(total, dtype=np.int64) if rows is None else _c(rows, np.int64)
    cols = np.arange(N, dtype=np.int64) if cols is None else _c(cols, np.int64)
    d = np.empty((rows.size, cols.size), np.float64)
    lib().orc_grouped_gemm_at(_p(a), _p(sa), _p(b), _p(sb), _p(off), E, total, N, K,
                              _p(rows), rows.size, _p(cols), cols.size, _p(d))
    return d


# ---------------------------------------------------------------- MoE
def route_topk(logits, k: int):
    """-> dict(idx [T,k] i32, gate [T,k] f32, off [E+1] i32, src_row [T*k] i32, pos [T,k] i32)."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    idx = np.empty((T, k), np.int32)
    gate = np.empty((T, k), np.float32)
    off = np.empty(E + 1, np.int32)
    src = np.empty(T * k, np.int32)
    pos = np.empty((T, k), np.int32)
    lib().orc_route_topk(_p(logits), T, E, k, _p(idx), _p(gate), _p(off), _p(src), _p(pos))
    return dict(idx=idx, gate=gate, off=off, src_row=src, pos=pos)


def permute_rows(q, s, src_row):
    q = _c(q, np.uint8); s = _c(s, np.float32); src_row = _c(src_row, np.int32)
    rows, K = q.shape
    out_rows = src_row.size
    qo = np.empty((out_rows, K), np.uint8)
    so = np.empty((K // 128, out_rows), np.float32)
    lib().orc_permute_rows(_p(q), _p(s), rows, K, _p(src_row), out_rows, _p(qo), _p(so))
    return qo, so


def moe_combine(y, pos, gate):
    y = _c(y, np.uint16); pos = _c(pos, np.int32); gate = _c(gate, np.float32)
    T, k = pos.shape
    N = y.shape[1]
    out = np.empty((T, N), np.uint16)
    lib().orc_moe_combine(_p(y), _p(pos), _p(gate), T, k, N, _p(out))
    return out
