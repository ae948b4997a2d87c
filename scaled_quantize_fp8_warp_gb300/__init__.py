"""Python binding of libfp8q.so: scaled FP8 quantisation and FP8 GEMM on GB300.

Argument marshalling only.  Every function here validates tensor placement,
takes raw device pointers from torch tensors, passes the current CUDA stream
and calls one C entry point declared in ``include/fp8q.h``; all arithmetic
runs in the library's CUDA kernels.  There is no CPU or PyTorch fallback: if
the library is missing or the device is not a GB300 the call raises.

The names follow the C ABI: ``fp8_amax``, ``fp8_quantize_tensor``,
``fp8_quantize_delayed``, ``fp8_quantize_tile1x128``,
``fp8_quantize_block128x128``, ``fp8_gemm`` and the role wrappers
``fp8_gemm_fprop`` / ``fp8_gemm_dgrad`` / ``fp8_gemm_wgrad``, and
``fp8_linear_autocast``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

E4M3 = 0
E5M2 = 1
DT_F32 = 0
DT_BF16 = 1
SCALE_TENSOR = 0
SCALE_TILE_1x128 = 1
SCALE_BLOCK_128x128 = 2
SCALE_ROW = 3
SCALE_MX_1x32 = 4
RECIPE_TENSOR_CURRENT = 0
RECIPE_TENSOR_DELAYED = 1
RECIPE_BLOCK = 2
RECIPE_MXFP8 = 3
MX_BLOCK = 32
HISTORY_LEN = 16
HISTORY_BYTES = 80

OK = 0
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "MISALIGNED", 3: "ARCH", 4: "WORKSPACE",
                5: "TIMEOUT", 6: "CUDA", 7: "NOT_IMPLEMENTED"}

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libfp8q.so")

#: every symbol include/fp8q.h declares
EXPORTS = (
    "fp8q_status_string", "fp8q_device_status", "fp8q_device_supported",
    "fp8q_selftest_barrier_timeout", "fp8_amax",
    "fp8_quantize_tensor", "fp8_quantize_tensor_current", "fp8_quantize_delayed",
    "fp8q_history_init",
    "fp8_quantize_tile1x128", "fp8_quantize_rowwise", "fp8_quantize_mxfp8",
    "fp8q_mx_scale_bytes", "fp8_quantize_block128x128", "fp8_gemm",
    "fp8_gemm_amax", "fp8_gemm_fprop",
    "fp8_gemm_dgrad", "fp8_gemm_wgrad", "fp8_gemm_grouped", "fp8q_linear_workspace_size",
    "fp8_linear_autocast",
    "fp8_linear_autocast_noalloc", "fp8q_linear_train_workspace_size", "fp8_linear_train",
    "fp8q_linear_train_host_workspace_size", "fp8_linear_train_host",
)


class Fp8qError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({status})")


class Operand(ctypes.Structure):
    """fp8q_operand: device byte matrix [rows, K] plus its scale description."""
    _fields_ = [("data", ctypes.c_void_p), ("format", ctypes.c_int32),
                ("scaling", ctypes.c_int32), ("scale", ctypes.c_void_p),
                ("scale_stride_row", ctypes.c_int64), ("scale_stride_k", ctypes.c_int64)]


def signatures() -> dict:
    """ctypes (restype, argtypes) of every entry point, as include/fp8q.h
    declares them (tests compare the two)."""
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    OP = ctypes.POINTER(Operand)
    return {
        "fp8q_status_string": (ctypes.c_char_p, [I32]),
        "fp8q_device_status": (I32, []),
        "fp8q_device_supported": (I32, []),
        "fp8q_selftest_barrier_timeout": (I32, [P]),
        "fp8_amax": (I32, [P, I32, I64, P, P]),
        "fp8_quantize_tensor": (I32, [P, I32, I64, I64, I32, P, P, P, P, I32, P]),
        "fp8_quantize_delayed": (I32, [P, I32, I64, I64, I32, P, P, P, P, I32, P]),
        "fp8_quantize_tensor_current": (I32, [P, I32, I64, I64, I32, P, P, P, P, I32, P]),
        "fp8q_history_init": (I32, [P, P, P]),
        "fp8_quantize_tile1x128": (I32, [P, I32, I64, I64, I32, P, P, P, P, I32, P]),
        "fp8_quantize_rowwise": (I32, [P, I32, I64, I64, I32, P, P, P, P, I32, P]),
        "fp8_quantize_block128x128": (I32, [P, I32, I64, I64, I32, P, P, P, I32, P]),
        "fp8_quantize_mxfp8": (I32, [P, I32, I64, I64, I32, P, P, P, P, P]),
        "fp8q_mx_scale_bytes": (SZ, [I64, I64]),
        "fp8_gemm": (I32, [OP, OP, P, I32, I64, I64, I64, P]),
        "fp8_gemm_amax": (I32, [OP, OP, P, I32, I64, I64, I64, P, P]),
        "fp8_gemm_fprop": (I32, [OP, OP, P, I32, I64, I64, I64, P]),
        "fp8_gemm_dgrad": (I32, [OP, OP, P, I32, I64, I64, I64, P]),
        "fp8_gemm_wgrad": (I32, [OP, OP, P, I32, I64, I64, I64, P]),
        "fp8_gemm_grouped": (I32, [P, I32, I32, P]),
        "fp8q_linear_workspace_size": (SZ, [I32, I64, I64, I64]),
        "fp8_linear_autocast": (I32, [P, P, I32, I64, I64, I64, I32, P, P, P, I32, P, SZ,
                                      P]),
        "fp8_linear_autocast_noalloc": (I32, [P, P, I32, I64, I64, I64, I32, P, P, P, I32,
                                              P]),
        "fp8q_linear_train_workspace_size": (SZ, [I32, I64, I64, I64]),
        "fp8_linear_train": (I32, [P, P, P, I32, I64, I64, I64, I32, P, P, P, P, P, P, I32,
                                   P, SZ, P]),
        "fp8q_linear_train_host_workspace_size": (SZ, [I32, I32, I32, I64, I64, I64]),
        "fp8_linear_train_host": (I32, [P, P, P, I32, I64, I64, I64, I32, P, P, P, P, P, P,
                                        I32, P, SZ, P]),
    }


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libfp8q.so (built by ``build_lib``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} not found: build it with `python -m scaled_quantize_fp8_warp_gb300.build_lib`"
                " (the FP8 path has no fallback)")
        lib = ctypes.CDLL(path)
        sig = signatures()
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def lib() -> ctypes.CDLL:
    return _lib if _lib is not None else load_library()


# --------------------------------------------------------------- marshalling

def _check(status: int, what: str):
    if status != OK:
        raise Fp8qError(status, what)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("fp8q needs CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("fp8q needs contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _in_dtype(x: torch.Tensor) -> int:
    if x.dtype == torch.bfloat16:
        return DT_BF16
    if x.dtype == torch.float32:
        return DT_F32
    raise TypeError(f"input must be bfloat16 or float32, got {x.dtype}")


_DT = {torch.bfloat16: DT_BF16, torch.float32: DT_F32}


def _out_dtype(dt) -> int:
    if dt == torch.bfloat16:
        return DT_BF16
    if dt == torch.float32:
        return DT_F32
    raise TypeError(f"output must be bfloat16 or float32, got {dt}")


def _rows_cols(x: torch.Tensor):
    if x.dim() != 2:
        raise ValueError("expected a 2-D matrix")
    return x.shape[0], x.shape[1]


def _empty(shape, dtype, like: torch.Tensor):
    return torch.empty(shape, dtype=dtype, device=like.device)


# ------------------------------------------------------------------ a1 amax

def fp8_amax(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """max |x| into a 1-element fp32 device tensor."""
    out = out if out is not None else _empty((1,), torch.float32, x)
    _check(lib().fp8_amax(_ptr(x), _in_dtype(x), x.numel(), _ptr(out), _stream(stream)),
           "fp8_amax")
    return out


# --------------------------------------------------------- a2/a3 quantize

def fp8_quantize_tensor(x, fmt, amax, want_q=True, want_qt=False, saturate=False,
                        q=None, q_t=None, scale=None, stream=None):
    """Per-tensor current scaling with s from the device scalar ``amax``.
    Returns (q [R,C] uint8 | None, q_t [C,R] uint8 | None, scale [1] fp32)."""
    R, C = _rows_cols(x)
    if want_q and q is None:
        q = _empty((R, C), torch.uint8, x)
    if want_qt and q_t is None:
        q_t = _empty((C, R), torch.uint8, x)
    scale = scale if scale is not None else _empty((1,), torch.float32, x)
    _check(lib().fp8_quantize_tensor(_ptr(x), _in_dtype(x), R, C, fmt, _ptr(amax), _ptr(scale),
                                     _ptr(q if want_q else None), _ptr(q_t if want_qt else None),
                                     int(saturate), _stream(stream)), "fp8_quantize_tensor")
    return (q if want_q else None), (q_t if want_qt else None), scale


def fp8_quantize_tensor_current(x, fmt, want_q=True, want_qt=False, saturate=False, q=None,
                                q_t=None, amax=None, scale=None, stream=None):
    """amax and per-tensor cast in one call (one cooperative launch when x
    holds at most 8 MiB).  Returns (q | None, q_t | None, amax [1], scale [1])."""
    R, C = _rows_cols(x)
    if want_q and q is None:
        q = _empty((R, C), torch.uint8, x)
    if want_qt and q_t is None:
        q_t = _empty((C, R), torch.uint8, x)
    amax = amax if amax is not None else _empty((1,), torch.float32, x)
    scale = scale if scale is not None else _empty((1,), torch.float32, x)
    _check(lib().fp8_quantize_tensor_current(
        _ptr(x), _in_dtype(x), R, C, fmt, _ptr(amax), _ptr(scale), _ptr(q if want_q else None),
        _ptr(q_t if want_qt else None), int(saturate), _stream(stream)),
        "fp8_quantize_tensor_current")
    return (q if want_q else None), (q_t if want_qt else None), amax, scale


class History:
    """Device-resident delayed-scaling state (fp8q_amax_history, 80 bytes)."""

    def __init__(self, device=None, initial=None, stream=None):
        dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.buf = torch.empty(HISTORY_BYTES // 4, dtype=torch.int32, device=dev)
        self.reset(initial, stream)

    def reset(self, initial=None, stream=None):
        arr = None
        if initial is not None:
            vals = [float(v) for v in initial]
            if len(vals) != HISTORY_LEN:
                raise ValueError(f"history needs {HISTORY_LEN} values")
            arr = (ctypes.c_float * HISTORY_LEN)(*vals)
        _check(lib().fp8q_history_init(_ptr(self.buf), arr, _stream(stream)), "fp8q_history_init")

    def state(self):
        """(amax list, next, scale) read back to the host (synchronises)."""
        h = self.buf.cpu()
        f = h.view(torch.float32)
        return f[:HISTORY_LEN].tolist(), int(h[HISTORY_LEN]), float(f[HISTORY_LEN + 1])

    def scratch(self):
        h = self.buf.cpu()
        return int(h[HISTORY_LEN + 2]), int(h[HISTORY_LEN + 3])


def fp8_quantize_delayed(x, fmt, hist: History, want_q=True, want_qt=False, saturate=False,
                         q=None, q_t=None, scale=None, stream=None):
    R, C = _rows_cols(x)
    if want_q and q is None:
        q = _empty((R, C), torch.uint8, x)
    if want_qt and q_t is None:
        q_t = _empty((C, R), torch.uint8, x)
    scale = scale if scale is not None else _empty((1,), torch.float32, x)
    _check(lib().fp8_quantize_delayed(_ptr(x), _in_dtype(x), R, C, fmt, _ptr(hist.buf),
                                      _ptr(scale), _ptr(q if want_q else None),
                                      _ptr(q_t if want_qt else None), int(saturate),
                                      _stream(stream)), "fp8_quantize_delayed")
    return (q if want_q else None), (q_t if want_qt else None), scale


def fp8_quantize_tile1x128(x, fmt, rows=True, cols=False, saturate=False, q=None,
                           q_scales=None, q_t=None, qt_scales=None, stream=None):
    """1x128 row tiles (q [R,C], q_scales [ceil(C/128), R]) and/or 128x1 column
    tiles (q_t [C,R], qt_scales [ceil(R/128), C]) from one read of x."""
    R, C = _rows_cols(x)
    if rows:
        q = q if q is not None else _empty((R, C), torch.uint8, x)
        q_scales = q_scales if q_scales is not None else _empty(((C + 127) // 128, R),
                                                                torch.float32, x)
    if cols:
        q_t = q_t if q_t is not None else _empty((C, R), torch.uint8, x)
        qt_scales = qt_scales if qt_scales is not None else _empty(((R + 127) // 128, C),
                                                                   torch.float32, x)
    _check(lib().fp8_quantize_tile1x128(
        _ptr(x), _in_dtype(x), R, C, fmt, _ptr(q if rows else None),
        _ptr(q_scales if rows else None), _ptr(q_t if cols else None),
        _ptr(qt_scales if cols else None), int(saturate), _stream(stream)),
        "fp8_quantize_tile1x128")
    return ((q, q_scales) if rows else (None, None)) + ((q_t, qt_scales) if cols else (None, None))


def fp8_quantize_rowwise(x, fmt, rows=True, cols=False, saturate=False, q=None, q_scales=None,
                         q_t=None, qt_scales=None, stream=None):
    """Row-wise scaling: q [R,C] with q_scales [R] (one scale per row) and/or
    q_t [C,R] with qt_scales [C] (one scale per column of x)."""
    R, C = _rows_cols(x)
    if rows:
        q = q if q is not None else _empty((R, C), torch.uint8, x)
        q_scales = q_scales if q_scales is not None else _empty((R,), torch.float32, x)
    if cols:
        q_t = q_t if q_t is not None else _empty((C, R), torch.uint8, x)
        qt_scales = qt_scales if qt_scales is not None else _empty((C,), torch.float32, x)
    _check(lib().fp8_quantize_rowwise(
        _ptr(x), _in_dtype(x), R, C, fmt, _ptr(q if rows else None),
        _ptr(q_scales if rows else None), _ptr(q_t if cols else None),
        _ptr(qt_scales if cols else None), int(saturate), _stream(stream)),
        "fp8_quantize_rowwise")
    return ((q, q_scales) if rows else (None, None)) + ((q_t, qt_scales) if cols else (None, None))


def mx_scale_bytes(rows: int, cols: int) -> int:
    """Bytes of one orientation's MXFP8 scale atoms for an [rows, cols] matrix."""
    return int(lib().fp8q_mx_scale_bytes(rows, cols))


def fp8_quantize_mxfp8(x, fmt, rows=True, cols=False, q=None, q_scales=None, q_t=None,
                       qt_scales=None, stream=None):
    """MXFP8 (OCP MX v1.0): q [R,C] with 1x32 row blocks and/or q_t [C,R] with
    32x1 column blocks of x; scales are E8M0 bytes in the library's atom
    layout (uint8 tensors of mx_scale_bytes(R, C) bytes; see include/fp8q.h).
    Returns (q, q_scales, q_t, qt_scales), None for a pair not requested."""
    R, C = _rows_cols(x)
    nbytes = mx_scale_bytes(R, C)
    if rows:
        q = q if q is not None else _empty((R, C), torch.uint8, x)
        q_scales = q_scales if q_scales is not None else _empty((nbytes,), torch.uint8, x)
    if cols:
        q_t = q_t if q_t is not None else _empty((C, R), torch.uint8, x)
        qt_scales = qt_scales if qt_scales is not None else _empty((nbytes,), torch.uint8, x)
    _check(lib().fp8_quantize_mxfp8(
        _ptr(x), _in_dtype(x), R, C, fmt, _ptr(q if rows else None),
        _ptr(q_scales if rows else None), _ptr(q_t if cols else None),
        _ptr(qt_scales if cols else None), _stream(stream)), "fp8_quantize_mxfp8")
    return ((q, q_scales) if rows else (None, None)) + ((q_t, qt_scales) if cols else (None, None))


def fp8_quantize_block128x128(x, fmt, want_q=True, want_qt=False, saturate=False, q=None,
                              q_t=None, scales=None, stream=None):
    R, C = _rows_cols(x)
    if want_q and q is None:
        q = _empty((R, C), torch.uint8, x)
    if want_qt and q_t is None:
        q_t = _empty((C, R), torch.uint8, x)
    scales = scales if scales is not None else _empty(((R + 127) // 128, (C + 127) // 128),
                                                      torch.float32, x)
    _check(lib().fp8_quantize_block128x128(_ptr(x), _in_dtype(x), R, C, fmt,
                                           _ptr(q if want_q else None),
                                           _ptr(q_t if want_qt else None), _ptr(scales),
                                           int(saturate), _stream(stream)),
           "fp8_quantize_block128x128")
    return (q if want_q else None), (q_t if want_qt else None), scales


# ------------------------------------------------------------- a4/a5 GEMM

class GemmOperand:
    """An FP8 operand [rows, K] (uint8 device tensor) with its scales; keeps
    the tensors alive next to the ctypes struct."""

    def __init__(self, data: torch.Tensor, fmt: int, scaling: int, scale: torch.Tensor,
                 stride_row: int = 0, stride_k: int = 0):
        if data.dtype != torch.uint8 or data.dim() != 2:
            raise TypeError("operand data must be a 2-D uint8 tensor")
        self.data, self.scale = data, scale
        self.rows, self.K = data.shape
        self.struct = Operand(data.data_ptr(), fmt, scaling, scale.data_ptr(), stride_row,
                              stride_k)

    @classmethod
    def tensor(cls, q, fmt, scale):
        return cls(q, fmt, SCALE_TENSOR, scale)

    @classmethod
    def tile(cls, q, fmt, scales):
        """scales [ceil(K/128), rows] as written by fp8_quantize_tile1x128."""
        return cls(q, fmt, SCALE_TILE_1x128, scales, 1, q.shape[0])

    @classmethod
    def row(cls, q, fmt, scales):
        """One scale per row over all of K (scales [rows])."""
        return cls(q, fmt, SCALE_ROW, scales, 1, 0)

    @classmethod
    def mx(cls, q, fmt, atoms):
        """MXFP8 operand: atoms as fp8_quantize_mxfp8 writes them for q."""
        return cls(q, fmt, SCALE_MX_1x32, atoms, 0, 0)

    @classmethod
    def block(cls, q, fmt, scales):
        """scales [ceil(rows/128), ceil(K/128)] of this orientation."""
        return cls(q, fmt, SCALE_BLOCK_128x128, scales, scales.shape[1], 1)

    @classmethod
    def block_transposed(cls, q_t, fmt, scales):
        """q_t = q^T of a block-quantised matrix; scales as written for q."""
        return cls(q_t, fmt, SCALE_BLOCK_128x128, scales, 1, scales.shape[1])


class GemmDesc(ctypes.Structure):
    """fp8q_gemm_desc: one GEMM of an fp8_gemm_grouped call."""
    _fields_ = [("A", Operand), ("B", Operand), ("C", ctypes.c_void_p),
                ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


#: most GEMMs one fp8_gemm_grouped call takes (FP8Q_GEMM_GROUP_MAX)
GEMM_GROUP_MAX = 3


def fp8_gemm_grouped(problems, out_dtype=torch.bfloat16, outs=None, stream=None):
    """Up to three independent GEMMs in one call: problems = [(A, B), ...]
    with C_i = A_i . B_i^T as fp8_gemm computes it (one launch when the
    CTA-pair kernel runs them all).  Returns the outputs."""
    problems = list(problems)
    outs = list(outs) if outs is not None else [
        torch.empty((A.rows, B.rows), dtype=out_dtype, device=A.data.device) for A, B in problems]
    if len(outs) != len(problems):
        raise ValueError("one output per problem")
    arr = (GemmDesc * max(1, len(problems)))()
    for i, ((A, B), C) in enumerate(zip(problems, outs)):
        arr[i] = GemmDesc(A.struct, B.struct, _ptr(C), A.rows, B.rows, A.K)
    dt = _out_dtype(outs[0].dtype) if outs else _out_dtype(out_dtype)
    _check(lib().fp8_gemm_grouped(ctypes.cast(arr, ctypes.c_void_p), len(problems), dt,
                                  _stream(stream)), "fp8_gemm_grouped")
    return outs


def _gemm_call(fn_name, A: GemmOperand, B: GemmOperand, out, M, N, K, stream):
    fn = getattr(lib(), fn_name)
    _check(fn(ctypes.byref(A.struct), ctypes.byref(B.struct), _ptr(out), _out_dtype(out.dtype),
              M, N, K, _stream(stream)), fn_name)
    return out


def fp8_gemm(A: GemmOperand, B: GemmOperand, out_dtype=torch.bfloat16, out=None, stream=None):
    """C [M, N] = A [M, K] . B [N, K]^T, dequantised."""
    M, N = A.rows, B.rows
    out = out if out is not None else torch.empty((M, N), dtype=out_dtype, device=A.data.device)
    return _gemm_call("fp8_gemm", A, B, out, M, N, A.K, stream)


def fp8_gemm_amax(A: GemmOperand, B: GemmOperand, out_dtype=torch.bfloat16, out=None,
                  amax=None, stream=None):
    """fp8_gemm plus amax(|C|) over the stored output from the same launch.
    Returns (C, amax) with amax a one-element fp32 device tensor."""
    M, N = A.rows, B.rows
    out = out if out is not None else torch.empty((M, N), dtype=out_dtype, device=A.data.device)
    amax = amax if amax is not None else _empty((1,), torch.float32, A.data)
    _check(lib().fp8_gemm_amax(ctypes.byref(A.struct), ctypes.byref(B.struct), _ptr(out),
                               _out_dtype(out.dtype), M, N, A.K, _ptr(amax), _stream(stream)),
           "fp8_gemm_amax")
    return out, amax


def fp8_gemm_fprop(x: GemmOperand, w: GemmOperand, out_dtype=torch.bfloat16, out=None,
                   stream=None):
    M, K, N = x.rows, x.K, w.rows
    out = out if out is not None else torch.empty((M, N), dtype=out_dtype, device=x.data.device)
    return _gemm_call("fp8_gemm_fprop", x, w, out, M, N, K, stream)


def fp8_gemm_dgrad(g: GemmOperand, w_t: GemmOperand, out_dtype=torch.bfloat16, out=None,
                   stream=None):
    M, N, K = g.rows, g.K, w_t.rows
    out = out if out is not None else torch.empty((M, K), dtype=out_dtype, device=g.data.device)
    return _gemm_call("fp8_gemm_dgrad", g, w_t, out, M, N, K, stream)


def fp8_gemm_wgrad(g_t: GemmOperand, x_t: GemmOperand, out_dtype=torch.bfloat16, out=None,
                   stream=None):
    N, M, K = g_t.rows, g_t.K, x_t.rows
    out = out if out is not None else torch.empty((N, K), dtype=out_dtype, device=g_t.data.device)
    return _gemm_call("fp8_gemm_wgrad", g_t, x_t, out, M, N, K, stream)


# ------------------------------------------------------------ whole forward

def linear_workspace_size(recipe: int, M: int, N: int, K: int) -> int:
    return int(lib().fp8q_linear_workspace_size(recipe, M, N, K))


def fp8_linear_autocast(x, w, recipe=RECIPE_TENSOR_CURRENT, out_dtype=torch.bfloat16,
                        hist_x: History | None = None, hist_w: History | None = None,
                        workspace=None, out=None, stream=None):
    """y = x w^T with dynamic FP8 quantisation of x and w (autocast)."""
    M, K = _rows_cols(x)
    N = w.shape[0]
    need = linear_workspace_size(recipe, M, N, K)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    out = out if out is not None else torch.empty((M, N), dtype=out_dtype, device=x.device)
    _check(lib().fp8_linear_autocast(
        _ptr(x), _ptr(w), _in_dtype(x), M, N, K, recipe,
        _ptr(hist_x.buf) if hist_x else None, _ptr(hist_w.buf) if hist_w else None,
        _ptr(out), _out_dtype(out.dtype), _ptr(workspace), workspace.numel(), _stream(stream)),
        "fp8_linear_autocast")
    return out


def linear_train_workspace_size(recipe: int, M: int, N: int, K: int) -> int:
    return int(lib().fp8q_linear_train_workspace_size(recipe, M, N, K))


def fp8_linear_train(x, w, g, recipe=RECIPE_TENSOR_CURRENT, out_dtype=torch.bfloat16,
                     hist_x: History | None = None, hist_w: History | None = None,
                     hist_g: History | None = None, workspace=None, y=None, dx=None, dw=None,
                     stream=None):
    """One linear layer's Fprop, Dgrad and Wgrad with x, w, grad_out quantized
    on the fly (device tensors).  Returns (y, dx, dw)."""
    M, K = _rows_cols(x)
    N = w.shape[0]
    if workspace is None:
        workspace = torch.empty(linear_train_workspace_size(recipe, M, N, K), dtype=torch.uint8,
                                device=x.device)
    y = y if y is not None else torch.empty((M, N), dtype=out_dtype, device=x.device)
    dx = dx if dx is not None else torch.empty((M, K), dtype=out_dtype, device=x.device)
    dw = dw if dw is not None else torch.empty((N, K), dtype=out_dtype, device=x.device)
    hp = lambda h: _ptr(h.buf) if h else None
    _check(lib().fp8_linear_train(
        _ptr(x), _ptr(w), _ptr(g), _in_dtype(x), M, N, K, recipe, hp(hist_x), hp(hist_w),
        hp(hist_g), _ptr(y), _ptr(dx), _ptr(dw), _out_dtype(y.dtype), _ptr(workspace),
        workspace.numel(), _stream(stream)), "fp8_linear_train")
    return y, dx, dw


def linear_train_host_workspace_size(recipe: int, in_dtype, out_dtype, M: int, N: int,
                                     K: int) -> int:
    return int(lib().fp8q_linear_train_host_workspace_size(
        recipe, _DT[in_dtype], _DT[out_dtype], M, N, K))


def fp8_linear_train_host(x_h, w_h, g_h, y_h, dx_h, dw_h, workspace,
                          recipe=RECIPE_TENSOR_CURRENT, hist_x: History | None = None,
                          hist_w: History | None = None, hist_g: History | None = None,
                          stream=None):
    """fp8_linear_train from and to host tensors (pinned CPU tensors; the
    copies happen inside the call's work on `stream`).  Outputs are filled
    once `stream` has reached this call's end."""
    M, K = x_h.shape
    N = w_h.shape[0]
    for t in (x_h, w_h, g_h, y_h, dx_h, dw_h):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("host buffers must be contiguous CPU tensors")
    hp = lambda h: _ptr(h.buf) if h else None
    _check(lib().fp8_linear_train_host(
        x_h.data_ptr(), w_h.data_ptr(), g_h.data_ptr(), _DT[x_h.dtype], M, N, K, recipe,
        hp(hist_x), hp(hist_w), hp(hist_g), y_h.data_ptr(), dx_h.data_ptr(), dw_h.data_ptr(),
        _DT[y_h.dtype], _ptr(workspace), workspace.numel(), _stream(stream)),
        "fp8_linear_train_host")


#: size of the library's static scratch (FP8Q_NOALLOC_SCRATCH_BYTES)
NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


def fp8_linear_autocast_noalloc(x, w, recipe=RECIPE_TENSOR_CURRENT, out_dtype=torch.bfloat16,
                                hist_x: History | None = None, hist_w: History | None = None,
                                out=None, stream=None):
    """fp8_linear_autocast for callers that cannot allocate device memory:
    the library keeps the FP8 copies and scales in its own fixed 64 MiB
    device array (see include/fp8q.h), so only the output is supplied here.
    Pass ``out`` to make the call allocate nothing at all from Python either."""
    M, K = _rows_cols(x)
    N = w.shape[0]
    out = out if out is not None else torch.empty((M, N), dtype=out_dtype, device=x.device)
    _check(lib().fp8_linear_autocast_noalloc(
        _ptr(x), _ptr(w), _in_dtype(x), M, N, K, recipe,
        _ptr(hist_x.buf) if hist_x else None, _ptr(hist_w.buf) if hist_w else None,
        _ptr(out), _out_dtype(out.dtype), _stream(stream)), "fp8_linear_autocast_noalloc")
    return out


# ------------------------------------------------------------- diagnostics

def device_status() -> int:
    """Synchronise and read (and clear) the device error word."""
    return int(lib().fp8q_device_status())


def selftest_barrier_timeout(stream=None) -> None:
    """Launch the failure-path self-test (see include/fp8q.h)."""
    _check(lib().fp8q_selftest_barrier_timeout(_stream(stream)), "fp8q_selftest_barrier_timeout")


def device_supported() -> bool:
    return bool(lib().fp8q_device_supported())


def status_string(status: int) -> str:
    return lib().fp8q_status_string(status).decode()
