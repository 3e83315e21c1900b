"""Thin ctypes binding of libfp8bs.so (declared in include/fp8bs.h).

Every function here has the name of the C entry point it calls and only
marshals arguments: it checks the torch tensors' dtype, device and layout,
allocates missing outputs with ``torch.empty`` on the input's device, passes
raw device pointers plus the current CUDA stream, and raises ``FP8Error`` on
a non-zero status.  All arithmetic runs in the library's CUDA kernels; there
is no fallback.  Importing this module fails if the library is not built.

bf16 tensors are ``torch.bfloat16``; E4M3 codes are ``torch.uint8`` (view
them as ``torch.float8_e4m3fn`` if wanted); scales are ``torch.float32``.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp8bs.so")

if not os.path.exists(LIB_PATH):
    raise ImportError("libfp8bs.so is not built: run `python -m fp8_fine_grained_16_b300.build`")

lib = ctypes.CDLL(LIB_PATH)

FP8_OK = 0
FP8_SCALE_POW2 = 1
FP8_BSCALE_BLOCK128 = 0
FP8_BSCALE_ROW = 1
FP8_OUT_BF16 = 0
FP8_OUT_F32 = 1
FP8_GEMM_FORM_DENSE = 0
FP8_GEMM_FORM_Q8 = 1
FP8_GEMM_FORM_GROUPED = 2
FP8_ERR_TIMEOUT = -5
FP8_ERR_OFFSETS = -6
FP8_ERR_SCRATCH = -8
FP8_ERR_SCALE = -9

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int
_U32 = ctypes.c_uint32

_SIGS = {
    "fp8_cast_e4m3": [_P, _I64, _P, _P],
    "fp8_quant_act_1x128": [_P, _I64, _I64, _I64, _P, _P, _U32, _P],
    "fp8_quant_act_128x1": [_P, _I64, _I64, _I64, _P, _P, _U32, _P],
    "fp8_quant_weight_128x128": [_P, _I64, _I64, _I64, _P, _P, _U32, _P],
    "fp8_quant_act_weight": [_P, _I64, _I64, _P, _P, _P, _I64, _I64, _P, _P, _I64, _U32, _P],
    "fp8_gemm_blockscaled": [_P, _P, _P, _P, _I, _P, _I, _I64, _I64, _I64, _P],
    "fp8_gemm_blockscaled_ws": [_P, _P, _P, _P, _I, _P, _I, _I64, _I64, _I64, _P, _I64, _P],
    "fp8_gemm_blockscaled_pow2": [_P, _P, _P, _P, _I, _P, _I, _I64, _I64, _I64, _P],
    "fp8_gemm_blockscaled_q8": [_P, _P, _P, _P, _I, _P, _P, _U32, _I64, _I64, _I64, _P],
    "fp8_gemm_blockscaled_q8_ws": [_P, _P, _P, _P, _I, _P, _P, _U32, _I64, _I64, _I64, _P, _I64, _P],
    "fp8_swiglu_quant_1x128": [_P, _I64, _I64, _I64, _P, _P, _U32, _P],
    "fp8_transpose_128x128": [_P, _P, _I64, _I64, _P, _P, _P],
    "fp8_grouped_gemm_blockscaled": [_P, _P, _P, _P, _P, _I, _I64, _I64, _I64, _P, _P],
    "fp8_grouped_gemm_blockscaled_pow2": [_P, _P, _P, _P, _P, _I, _I64, _I64, _I64, _P, _P],
    "fp8_moe_route_topk": [_P, _I64, _I, _I, _P, _P, _P, _P, _P, _P, _P],
    "fp8_moe_route_topk_noalloc": [_P, _I64, _I, _I, _P, _P, _P, _P, _P, _P],
    "fp8_permute_rows": [_P, _P, _I64, _I64, _P, _I64, _P, _P, _P],
    "fp8_moe_combine_bf16": [_P, _I64, _P, _P, _I64, _I, _I64, _P, _P],
    "fp8_get_status": [_P],
    "fp8_selftest_wait_timeout": [ctypes.c_uint64, _P],
    "fp8_selftest_reciprocal": [_U32, _U32, _P, _P],
    "fp8_linear_host": [_P, _P, _I64, _I64, _I64, _P, _U32, _P, _I64, _P],
}
for _name, _args in _SIGS.items():
    _f = getattr(lib, _name)
    _f.argtypes = _args
    _f.restype = _I
lib.fp8_moe_route_workspace_size.argtypes = [_I64, _I]
lib.fp8_moe_route_workspace_size.restype = _I64
lib.fp8_gemm_blockscaled_workspace_bytes.argtypes = [_I64, _I64, _I64]
lib.fp8_gemm_blockscaled_workspace_bytes.restype = _I64
lib.fp8_gemm_split_plan.argtypes = [_I, _I64, _I64, _I64, _I, _I64, _P, _P, _P]
lib.fp8_gemm_split_plan.restype = _I
lib.fp8_gemm_split_units.argtypes = [_I, _I64, _I64, _I64, _I, _I64, _I64, _P, _I64]
lib.fp8_gemm_split_units.restype = _I64
lib.fp8_linear_host_workspace_bytes.argtypes = [_I64, _I64, _I64]
lib.fp8_linear_host_workspace_bytes.restype = _I64
lib.fp8_gemm_tile_cols.argtypes = [_I]
lib.fp8_gemm_tile_cols.restype = _I
lib.fp8_strerror.argtypes = [_I]
lib.fp8_strerror.restype = ctypes.c_char_p
lib.fp8_version.argtypes = []
lib.fp8_version.restype = _I

#: every symbol include/fp8bs.h declares
EXPORTED = sorted(list(_SIGS) + ["fp8_moe_route_workspace_size", "fp8_gemm_blockscaled_workspace_bytes",
                                  "fp8_gemm_split_plan", "fp8_gemm_split_units", "fp8_gemm_tile_cols",
                                  "fp8_linear_host_workspace_bytes",
                                  "fp8_strerror", "fp8_version"])


class FP8Error(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__("%s failed: %s (%d)" % (fn, lib.fp8_strerror(code).decode(), code))
        self.code = code


def _check(fn: str, code: int) -> None:
    if code != FP8_OK:
        raise FP8Error(fn, code)


def _stream(stream=None) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: torch.Tensor | None, dtype=None, name="tensor") -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def _rows(x: torch.Tensor, name: str):
    if x.dim() != 2:
        raise ValueError("%s must be 2-D" % name)
    if x.stride(1) != 1:
        raise ValueError("%s must have unit column stride" % name)
    return x.shape[0], x.shape[1], x.stride(0)


# ---------------------------------------------------------------- cast
def fp8_cast_e4m3(x: torch.Tensor, q: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    if q is None:
        q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _check("fp8_cast_e4m3", lib.fp8_cast_e4m3(_ptr(x, torch.float32, "x"), x.numel(),
                                              _ptr(q, torch.uint8, "q"), _stream(stream)))
    return q


# ---------------------------------------------------------------- quantisers
def fp8_quant_act_1x128(x: torch.Tensor, q=None, s=None, flags: int = 0, stream=None):
    """x bf16 [M, K] (row stride may exceed K) -> (q u8 [M, K], s f32 [K/128, M])."""
    M, K, ldx = _rows(x, "x")
    if x.dtype != torch.bfloat16 or not x.is_cuda:
        raise TypeError("x must be a CUDA bf16 tensor")
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device) if q is None else q
    s = torch.empty((K // 128, M), dtype=torch.float32, device=x.device) if s is None else s
    _check("fp8_quant_act_1x128", lib.fp8_quant_act_1x128(x.data_ptr(), M, K, ldx, _ptr(q, torch.uint8, "q"),
                                                          _ptr(s, torch.float32, "s"), flags, _stream(stream)))
    return q, s


def fp8_quant_act_128x1(x: torch.Tensor, qT=None, s=None, flags: int = 0, stream=None):
    """x bf16 [T, H] -> (qT u8 [H, T], s f32 [T/128, H])."""
    T, H, ldx = _rows(x, "x")
    if x.dtype != torch.bfloat16 or not x.is_cuda:
        raise TypeError("x must be a CUDA bf16 tensor")
    qT = torch.empty((H, T), dtype=torch.uint8, device=x.device) if qT is None else qT
    s = torch.empty((T // 128, H), dtype=torch.float32, device=x.device) if s is None else s
    _check("fp8_quant_act_128x1", lib.fp8_quant_act_128x1(x.data_ptr(), T, H, ldx, _ptr(qT, torch.uint8, "qT"),
                                                          _ptr(s, torch.float32, "s"), flags, _stream(stream)))
    return qT, s


def fp8_quant_weight_128x128(w: torch.Tensor, q=None, s=None, flags: int = 0, stream=None):
    """w bf16 [N, K] or [E, N, K] -> (q u8 same shape, s f32 [(E,) N/128, K/128])."""
    if w.dtype != torch.bfloat16 or not w.is_cuda:
        raise TypeError("w must be a CUDA bf16 tensor")
    lead = w.shape[:-2]
    w2 = w.reshape(-1, w.shape[-1]) if w.dim() == 3 else w
    N, K, ldw = _rows(w2, "w")
    q = torch.empty(w.shape, dtype=torch.uint8, device=w.device) if q is None else q
    s = torch.empty((*lead, w.shape[-2] // 128, K // 128), dtype=torch.float32, device=w.device) if s is None else s
    _check("fp8_quant_weight_128x128", lib.fp8_quant_weight_128x128(w2.data_ptr(), N, K, ldw,
                                                                    _ptr(q, torch.uint8, "q"),
                                                                    _ptr(s, torch.float32, "s"), flags,
                                                                    _stream(stream)))
    return q, s


def fp8_quant_act_weight(x: torch.Tensor, w: torch.Tensor, qx=None, sx=None, qw=None, sw=None, flags: int = 0,
                         stream=None):
    """x bf16 [M, K], w bf16 [N, K] -> (qx, sx, qw, sw) in one launch, the same
    results as fp8_quant_act_1x128(x) and fp8_quant_weight_128x128(w)."""
    if x.dtype != torch.bfloat16 or w.dtype != torch.bfloat16 or not (x.is_cuda and w.is_cuda):
        raise TypeError("x and w must be CUDA bf16 tensors")
    M, K, ldx = _rows(x, "x")
    N, Kw, ldw = _rows(w, "w")
    if Kw != K:
        raise ValueError("x and w must have the same number of columns")
    qx = torch.empty((M, K), dtype=torch.uint8, device=x.device) if qx is None else qx
    sx = torch.empty((K // 128, M), dtype=torch.float32, device=x.device) if sx is None else sx
    qw = torch.empty((N, K), dtype=torch.uint8, device=w.device) if qw is None else qw
    sw = torch.empty((N // 128, K // 128), dtype=torch.float32, device=w.device) if sw is None else sw
    _check("fp8_quant_act_weight", lib.fp8_quant_act_weight(
        x.data_ptr(), M, ldx, _ptr(qx, torch.uint8, "qx"), _ptr(sx, torch.float32, "sx"),
        w.data_ptr(), N, ldw, _ptr(qw, torch.uint8, "qw"), _ptr(sw, torch.float32, "sw"), K, flags,
        _stream(stream)))
    return qx, sx, qw, sw


# ---------------------------------------------------------------- GEMMs
# One split workspace per (device, stream): calls on one stream run in order,
# so they can share it.  Its size depends only on the device, so an entry is
# allocated once and never replaced (nothing frees memory a queued call uses).
_GEMM_WS: dict = {}


def _gemm_workspace(device: torch.device, stream_handle: int, M: int, N: int, K: int):
    need = lib.fp8_gemm_blockscaled_workspace_bytes(M, N, K)
    if need < 0:
        _check("fp8_gemm_blockscaled_workspace_bytes", int(need))
    if need == 0:
        return None, 0
    key = (device.index, stream_handle)
    ws = _GEMM_WS.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.empty(need, dtype=torch.uint8, device=device)
        _GEMM_WS[key] = ws
    return ws, need


_LINEAR_WS: dict = {}


def _linear_workspace(device: torch.device, stream_handle: int, M: int, N: int, K: int):
    need = lib.fp8_linear_host_workspace_bytes(M, N, K)
    if need < 0:
        _check("fp8_linear_host_workspace_bytes", int(need))
    key = (device.index, stream_handle)
    ws = _LINEAR_WS.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.empty(need, dtype=torch.uint8, device=device)
        _LINEAR_WS[key] = ws
    return ws, need


def _workspace_devices() -> list:
    """The device indices that hold a cached workspace (each must be waited
    for before its workspace goes back to the caching allocator)."""
    return sorted({dev for dev, _ in _GEMM_WS} | {dev for dev, _ in _LINEAR_WS})


def release_gemm_workspaces(_synchronize=torch.cuda.synchronize) -> int:
    """Free the workspaces kept per device and stream: the GEMM split slabs
    (one per SM pair, 18.9 MB on a 148-SM GPU, per stream that ran a split
    GEMM) and the device buffers of fp8_linear_host.  It
    first waits for every device that holds one, so no GEMM queued on any
    of them still reads or writes its workspace.  Returns how many were
    freed; later calls allocate again as needed."""
    n = len(_GEMM_WS) + len(_LINEAR_WS)
    if n:
        for dev in _workspace_devices():
            _synchronize(dev)
        _GEMM_WS.clear()
        _LINEAR_WS.clear()
    return n


def fp8_gemm_tile_cols(form: int = FP8_GEMM_FORM_DENSE) -> int:
    """Columns of one 256-row output tile of a GEMM form (host only)."""
    n = lib.fp8_gemm_tile_cols(form)
    if n < 0:
        _check("fp8_gemm_tile_cols", n)
    return n


def fp8_gemm_split_plan(M: int, N: int, K: int, pairs: int, workspace_bytes: int, form: int = FP8_GEMM_FORM_DENSE):
    """(split, tail0, launched_pairs) of a dense GEMM form's tail split (host only)."""
    out = (ctypes.c_int64 * 3)()
    p = ctypes.addressof(out)
    _check("fp8_gemm_split_plan", lib.fp8_gemm_split_plan(form, M, N, K, pairs, workspace_bytes, p, p + 8, p + 16))
    return int(out[0]), int(out[1]), int(out[2])


def fp8_gemm_split_units(M: int, N: int, K: int, pairs: int, workspace_bytes: int, pair: int,
                         form: int = FP8_GEMM_FORM_DENSE):
    """[(tile, kb0, kb1, slab), ...] that launched pair `pair` runs (host only)."""
    n = lib.fp8_gemm_split_units(form, M, N, K, pairs, workspace_bytes, pair, None, 0)
    if n < 0:
        _check("fp8_gemm_split_units", int(n))
    buf = (ctypes.c_int64 * (4 * max(n, 1)))()
    lib.fp8_gemm_split_units(form, M, N, K, pairs, workspace_bytes, pair, ctypes.addressof(buf), n)
    return [tuple(int(v) for v in buf[4 * i:4 * i + 4]) for i in range(n)]


def fp8_gemm_blockscaled(a, sa, b, sb, b_scale_mode: int = FP8_BSCALE_BLOCK128, out_dtype=torch.bfloat16,
                         d=None, stream=None, split: bool = True) -> torch.Tensor:
    """D[M, N] = block-scaled a[M, K] x b[N, K]^T (bf16 or fp32 out).  With
    ``split`` (the default) it calls fp8_gemm_blockscaled_ws with a workspace
    kept per device and stream, so a short last wave of tiles is split along
    K; ``split=False`` calls fp8_gemm_blockscaled."""
    M, K = a.shape
    N = b.shape[0]
    if b.shape[1] != K:
        raise ValueError("a and b disagree on K")
    d_dtype = FP8_OUT_F32 if out_dtype == torch.float32 else FP8_OUT_BF16
    if d is None:
        d = torch.empty((M, N), dtype=torch.float32 if d_dtype == FP8_OUT_F32 else torch.bfloat16, device=a.device)
    args = (_ptr(a, torch.uint8, "a"), _ptr(sa, torch.float32, "sa"), _ptr(b, torch.uint8, "b"),
            _ptr(sb, torch.float32, "sb"), b_scale_mode, _ptr(d, None, "d"), d_dtype, M, N, K)
    st = _stream(stream)
    if not split:
        _check("fp8_gemm_blockscaled", lib.fp8_gemm_blockscaled(*args, st))
        return d
    ws, nbytes = _gemm_workspace(a.device, st, M, N, K)
    _check("fp8_gemm_blockscaled_ws", lib.fp8_gemm_blockscaled_ws(
        *args, None if ws is None else ws.data_ptr(), nbytes, st))
    return d


def _host_ptr(t: torch.Tensor, name: str) -> int:
    if t.is_cuda:
        raise ValueError("%s must be a host (CPU) tensor" % name)
    if t.dtype != torch.bfloat16:
        raise TypeError("%s must be torch.bfloat16, got %s" % (name, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def fp8_linear_host(x_h: torch.Tensor, w_h: torch.Tensor, y_h: torch.Tensor | None = None, flags: int = 0,
                    device=None, stream=None) -> torch.Tensor:
    """Y = X W^T from HOST tensors x_h bf16 [M, K] and w_h bf16 [N, K] into the
    host tensor y_h bf16 [M, N] (allocated page-locked if not given): the
    copies in and out, the two quantisations and the GEMM, pipelined over
    chunks of W on the GPU `device` (default: the current one).  Asynchronous
    on the stream: y_h holds the result once the stream reaches this call's
    end (torch.cuda.synchronize, or an event)."""
    M, K = x_h.shape
    N = w_h.shape[0]
    if w_h.shape[1] != K:
        raise ValueError("x_h and w_h disagree on K")
    if y_h is None:
        y_h = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    elif tuple(y_h.shape) != (M, N):
        raise ValueError("y_h must be [M, N]")
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else torch.device(device).index)
    with torch.cuda.device(dev):
        st = _stream(stream)
        ws, nbytes = _linear_workspace(dev, st, M, N, K)
        _check("fp8_linear_host", lib.fp8_linear_host(
            _host_ptr(x_h, "x_h"), _host_ptr(w_h, "w_h"), M, N, K, _host_ptr(y_h, "y_h"), flags,
            ws.data_ptr(), nbytes, st))
    return y_h


def fp8_gemm_blockscaled_pow2(a, sa, b, sb, b_scale_mode: int = FP8_BSCALE_BLOCK128, out_dtype=torch.bfloat16,
                              d=None, stream=None) -> torch.Tensor:
    """As fp8_gemm_blockscaled, for power-of-two scales applied by the tensor core."""
    M, K = a.shape
    N = b.shape[0]
    if b.shape[1] != K:
        raise ValueError("a and b disagree on K")
    d_dtype = FP8_OUT_F32 if out_dtype == torch.float32 else FP8_OUT_BF16
    if d is None:
        d = torch.empty((M, N), dtype=torch.float32 if d_dtype == FP8_OUT_F32 else torch.bfloat16, device=a.device)
    _check("fp8_gemm_blockscaled_pow2", lib.fp8_gemm_blockscaled_pow2(
        _ptr(a, torch.uint8, "a"), _ptr(sa, torch.float32, "sa"), _ptr(b, torch.uint8, "b"),
        _ptr(sb, torch.float32, "sb"), b_scale_mode, _ptr(d, None, "d"), d_dtype, M, N, K, _stream(stream)))
    return d


def fp8_swiglu_quant_1x128(y: torch.Tensor, I: int, q=None, s=None, flags: int = FP8_SCALE_POW2, stream=None):
    """y bf16 [R, >= 2I] (gate | up; row stride may exceed the width) -> SwiGLU
    quantised per 1x128 tile: (q u8 [R, I], s f32 [I/128, R]).  Power-of-two
    scales by default."""
    R, _, ldy = _rows(y, "y")
    if y.dtype != torch.bfloat16 or not y.is_cuda:
        raise TypeError("y must be a CUDA bf16 tensor")
    q = torch.empty((R, I), dtype=torch.uint8, device=y.device) if q is None else q
    s = torch.empty((I // 128, R), dtype=torch.float32, device=y.device) if s is None else s
    _check("fp8_swiglu_quant_1x128", lib.fp8_swiglu_quant_1x128(
        y.data_ptr(), R, I, ldy, _ptr(q, torch.uint8, "q"), _ptr(s, torch.float32, "s"), flags, _stream(stream)))
    return q, s


def fp8_gemm_blockscaled_q8(a, sa, b, sb, b_scale_mode: int = FP8_BSCALE_BLOCK128, flags: int = 0,
                            q_out=None, s_out=None, stream=None, split: bool = True):
    """D = block-scaled a x b^T, quantised in the epilogue per 1x128 tile along N:
    (q u8 [M, N], s f32 [N/128, M]), the layout fp8_quant_act_1x128 produces.
    ``split`` as for fp8_gemm_blockscaled (fp8_gemm_blockscaled_q8_ws with the
    per-stream workspace, or fp8_gemm_blockscaled_q8 without)."""
    M, K = a.shape
    N = b.shape[0]
    if b.shape[1] != K:
        raise ValueError("a and b disagree on K")
    q_out = torch.empty((M, N), dtype=torch.uint8, device=a.device) if q_out is None else q_out
    s_out = torch.empty((N // 128, M), dtype=torch.float32, device=a.device) if s_out is None else s_out
    args = (_ptr(a, torch.uint8, "a"), _ptr(sa, torch.float32, "sa"), _ptr(b, torch.uint8, "b"),
            _ptr(sb, torch.float32, "sb"), b_scale_mode, _ptr(q_out, torch.uint8, "q_out"),
            _ptr(s_out, torch.float32, "s_out"), flags, M, N, K)
    st = _stream(stream)
    if not split:
        _check("fp8_gemm_blockscaled_q8", lib.fp8_gemm_blockscaled_q8(*args, st))
        return q_out, s_out
    ws, nbytes = _gemm_workspace(a.device, st, M, N, K)
    _check("fp8_gemm_blockscaled_q8_ws", lib.fp8_gemm_blockscaled_q8_ws(
        *args, None if ws is None else ws.data_ptr(), nbytes, st))
    return q_out, s_out


def fp8_transpose_128x128(q, s, qT=None, sT=None, stream=None):
    """q u8 [N, K], s f32 [N/128, K/128] -> (qT u8 [K, N], sT f32 [K/128, N/128]):
    the 128x128-block quantisation of the transposed matrix (for Dgrad)."""
    N, K = q.shape
    qT = torch.empty((K, N), dtype=torch.uint8, device=q.device) if qT is None else qT
    sT = torch.empty((K // 128, N // 128), dtype=torch.float32, device=q.device) if sT is None else sT
    _check("fp8_transpose_128x128", lib.fp8_transpose_128x128(
        _ptr(q, torch.uint8, "q"), _ptr(s, torch.float32, "s"), N, K, _ptr(qT, torch.uint8, "qT"),
        _ptr(sT, torch.float32, "sT"), _stream(stream)))
    return qT, sT


def fp8_grouped_gemm_blockscaled_pow2(a, sa, b, sb, expert_offsets, d=None, stream=None) -> torch.Tensor:
    """As fp8_grouped_gemm_blockscaled, for power-of-two scales applied by the tensor core."""
    R, K = a.shape
    E, N, Kb = b.shape
    if Kb != K:
        raise ValueError("a and b disagree on K")
    if d is None:
        d = torch.empty((R, N), dtype=torch.bfloat16, device=b.device)
    _check("fp8_grouped_gemm_blockscaled_pow2", lib.fp8_grouped_gemm_blockscaled_pow2(
        _ptr(a, torch.uint8, "a"), _ptr(sa, torch.float32, "sa"), _ptr(b, torch.uint8, "b"),
        _ptr(sb, torch.float32, "sb"), _ptr(expert_offsets, torch.int32, "expert_offsets"), E, R, N, K,
        _ptr(d, torch.bfloat16, "d"), _stream(stream)))
    return d


def fp8_grouped_gemm_blockscaled(a, sa, b, sb, expert_offsets, d=None, stream=None) -> torch.Tensor:
    """Per-expert block-scaled GEMM: a [R, K], b [E, N, K], offsets int32 [E+1] on device -> bf16 [R, N]."""
    R, K = a.shape
    E, N, Kb = b.shape
    if Kb != K:
        raise ValueError("a and b disagree on K")
    if d is None:
        d = torch.empty((R, N), dtype=torch.bfloat16, device=b.device)
    _check("fp8_grouped_gemm_blockscaled", lib.fp8_grouped_gemm_blockscaled(
        _ptr(a, torch.uint8, "a"), _ptr(sa, torch.float32, "sa"), _ptr(b, torch.uint8, "b"),
        _ptr(sb, torch.float32, "sb"), _ptr(expert_offsets, torch.int32, "expert_offsets"), E, R, N, K,
        _ptr(d, torch.bfloat16, "d"), _stream(stream)))
    return d


# ---------------------------------------------------------------- MoE helpers
def fp8_moe_route_workspace_size(T: int, E: int) -> int:
    return lib.fp8_moe_route_workspace_size(T, E)


def fp8_moe_route_topk(logits: torch.Tensor, topk: int, out: dict | None = None, work=None, stream=None) -> dict:
    """logits f32 [T, E] -> dict(idx, gate, off, src_row, pos) on the device."""
    T, E = logits.shape
    dev = logits.device
    o = out or dict(idx=torch.empty((T, topk), dtype=torch.int32, device=dev),
                    gate=torch.empty((T, topk), dtype=torch.float32, device=dev),
                    off=torch.empty(E + 1, dtype=torch.int32, device=dev),
                    src_row=torch.empty(T * topk, dtype=torch.int32, device=dev),
                    pos=torch.empty((T, topk), dtype=torch.int32, device=dev))
    if work is None:
        work = torch.empty(max(1, fp8_moe_route_workspace_size(T, E) // 4), dtype=torch.int32, device=dev)
    _check("fp8_moe_route_topk", lib.fp8_moe_route_topk(
        _ptr(logits, torch.float32, "logits"), T, E, topk, _ptr(o["idx"], torch.int32), _ptr(o["gate"], torch.float32),
        _ptr(o["off"], torch.int32), _ptr(o["src_row"], torch.int32), _ptr(o["pos"], torch.int32),
        _ptr(work, torch.int32, "work"), _stream(stream)))
    return o


def fp8_moe_route_topk_noalloc(logits: torch.Tensor, topk: int, out: dict | None = None, stream=None) -> dict:
    """fp8_moe_route_topk for callers that cannot allocate device scratch:
    the library's own static scratch stands in for `work`.  With `out`
    given, this call allocates nothing on the device."""
    T, E = logits.shape
    dev = logits.device
    o = out or dict(idx=torch.empty((T, topk), dtype=torch.int32, device=dev),
                    gate=torch.empty((T, topk), dtype=torch.float32, device=dev),
                    off=torch.empty(E + 1, dtype=torch.int32, device=dev),
                    src_row=torch.empty(T * topk, dtype=torch.int32, device=dev),
                    pos=torch.empty((T, topk), dtype=torch.int32, device=dev))
    _check("fp8_moe_route_topk_noalloc", lib.fp8_moe_route_topk_noalloc(
        _ptr(logits, torch.float32, "logits"), T, E, topk, _ptr(o["idx"], torch.int32), _ptr(o["gate"], torch.float32),
        _ptr(o["off"], torch.int32), _ptr(o["src_row"], torch.int32), _ptr(o["pos"], torch.int32), _stream(stream)))
    return o


def fp8_permute_rows(q, s, src_row, q_out=None, s_out=None, stream=None):
    """q u8 [rows, K], s f32 [K/128, rows], src_row int32 [R] -> (q_out [R, K], s_out [K/128, R])."""
    rows, K = q.shape
    R = src_row.numel()
    q_out = torch.empty((R, K), dtype=torch.uint8, device=q.device) if q_out is None else q_out
    s_out = torch.empty((K // 128, R), dtype=torch.float32, device=q.device) if s_out is None else s_out
    _check("fp8_permute_rows", lib.fp8_permute_rows(
        _ptr(q, torch.uint8, "q"), _ptr(s, torch.float32, "s"), rows, K, _ptr(src_row, torch.int32, "src_row"), R,
        _ptr(q_out, torch.uint8, "q_out"), _ptr(s_out, torch.float32, "s_out"), _stream(stream)))
    return q_out, s_out


def fp8_moe_combine_bf16(y, pos, gate, out=None, stream=None) -> torch.Tensor:
    """y bf16 [rows, N], pos int32 [T, k], gate f32 [T, k] -> bf16 [T, N]."""
    rows, N = y.shape
    T, k = pos.shape
    out = torch.empty((T, N), dtype=torch.bfloat16, device=y.device) if out is None else out
    _check("fp8_moe_combine_bf16", lib.fp8_moe_combine_bf16(
        _ptr(y, torch.bfloat16, "y"), rows, _ptr(pos, torch.int32, "pos"), _ptr(gate, torch.float32, "gate"), T, k, N,
        _ptr(out, torch.bfloat16, "out"), _stream(stream)))
    return out


def fp8_selftest_reciprocal(first_bits: int = 0x3F800000, last_bits: int = 0x7FFFFFFF, device=None) -> int:
    """How many floats d >= 1 with bits in [first_bits, last_bits] get a
    reciprocal in the SwiGLU kernel that differs from __frcp_rn (synchronises)."""
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else torch.device(device).index)
    bad = torch.zeros(1, dtype=torch.int64, device=dev)
    with torch.cuda.device(dev):
        _check("fp8_selftest_reciprocal", lib.fp8_selftest_reciprocal(first_bits, last_bits, bad.data_ptr(),
                                                                      _stream(None)))
        torch.cuda.synchronize(dev)
    return int(bad.item())


def fp8_get_status(stream=None) -> int:
    """Synchronise the stream; return and clear the device status (0 = ok)."""
    return lib.fp8_get_status(_stream(stream))


def fp8_selftest_wait_timeout(timeout_ns: int, stream=None) -> None:
    _check("fp8_selftest_wait_timeout", lib.fp8_selftest_wait_timeout(timeout_ns, _stream(stream)))


def fp8_strerror(code: int) -> str:
    return lib.fp8_strerror(code).decode()


def fp8_version() -> int:
    return lib.fp8_version()
