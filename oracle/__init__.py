"""Plain CPU oracle for scaled FP8 quantisation and the FP8 GEMM.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product path
(``scaled_quantize_fp8_warp_gb300``) never does.  The C code in
``fp8_oracle.c`` is the oracle; this module only compiles it with gcc, loads
it with ctypes and marshals numpy arrays.  It shares no code with the CUDA
library.

Definitions follow the "fp8_parity.py" page (``scaled_roundtrip``,
``FP8Matmul``, smoke steps 1-4) and the NVIDIA low-precision-training blog
repost (GEMM roles, delayed scaling); every C function cites its passage.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

E4M3 = 0
E5M2 = 1
IN_F32 = 0
IN_BF16 = 1
SCALE_TENSOR = 0
SCALE_TILE = 1
SCALE_BLOCK = 2
SCALE_ROW = 3
SCALE_MX = 4
MX_BLOCK = 32

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8_oracle.c")
_HDR = os.path.join(_HERE, "fp8_oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc, no FMA
    contraction, no fast-math) if it is missing or older than its sources."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
               "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Operand(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("fmt", ctypes.c_int32),
                ("scaling", ctypes.c_int32), ("scale", ctypes.c_void_p),
                ("stride_row", ctypes.c_int64), ("stride_k", ctypes.c_int64),
                ("mx_scale", ctypes.c_void_p)]


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P, I32, I64, F32, F64 = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                 ctypes.c_float, ctypes.c_double)
        sig = {
            "orc_fmax": (F64, [I32]),
            "orc_load": (F32, [P, I32, I64]),
            "orc_fp8_decode": (F64, [ctypes.c_uint8, I32]),
            "orc_fp8_encode": (ctypes.c_uint8, [F32, I32, I32]),
            "orc_amax": (F32, [P, I32, I64]),
            "orc_scale_from_amax": (F32, [F32, I32]),
            "orc_cast": (None, [P, I32, I64, F32, I32, I32, P]),
            "orc_quantize_tensor": (None, [P, I32, I64, I64, F32, I32, I32, P, P]),
            "orc_quantize_tile_rows": (None, [P, I32, I64, I64, I32, I32, P, P]),
            "orc_quantize_tile_cols": (None, [P, I32, I64, I64, I32, I32, P, P]),
            "orc_quantize_block": (None, [P, I32, I64, I64, I32, I32, P, P, P]),
            "orc_quantize_delayed": (F32, [P, I32, I64, I64, I32, I32, P, I32, P, P, P]),
            "orc_quantize_rowwise": (None, [P, I32, I64, I64, I32, I32, P, P, P, P]),
            "orc_dequantize": (None, [P, I64, I32, F32, P]),
            "orc_operand_scale": (F64, [ctypes.POINTER(Operand), I64, I64]),
            "orc_e8m0_decode": (F64, [ctypes.c_uint8]),
            "orc_mx_scale_code": (ctypes.c_uint8, [F32, I32]),
            "orc_quantize_mx_rows": (None, [P, I32, I64, I64, I32, P, P]),
            "orc_quantize_mx_cols": (None, [P, I32, I64, I64, I32, P, P]),
            "orc_gemm_points": (None, [ctypes.POINTER(Operand), ctypes.POINTER(Operand),
                                       I64, I64, P, P, P, P]),
            "orc_gemm_rows": (None, [ctypes.POINTER(Operand), ctypes.POINTER(Operand),
                                     I64, I64, I64, I64, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


# ------------------------------------------------------------------ helpers

def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _input(x: np.ndarray):
    """Accept an fp32 array or a uint16 array holding bf16 bit patterns."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, IN_F32
    if x.dtype == np.uint16:
        return x, IN_BF16
    raise TypeError(f"oracle input must be float32 or uint16 (bf16 bits), got {x.dtype}")


def fmax(fmt: int) -> float:
    return _load().orc_fmax(fmt)


def widen(x: np.ndarray) -> np.ndarray:
    """Inputs as the oracle sees them (bf16 widened exactly to fp32)."""
    x, dt = _input(x)
    if dt == IN_F32:
        return x.copy()
    return (x.astype(np.uint32) << 16).view(np.float32)


def decode(codes, fmt: int) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.orc_fp8_decode(int(b), fmt) for b in c], dtype=np.float64).reshape(
        np.shape(codes))


def decode_table(fmt: int) -> np.ndarray:
    """All 256 byte values decoded (index = byte)."""
    return decode(np.arange(256, dtype=np.uint8), fmt)


def encode(v, fmt: int, saturate: bool = False) -> np.ndarray:
    """Encode fp32 values; vectorised through orc_cast with scale 1 (x / 1 is
    exact, so this is the plain cast)."""
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float32))
    out = np.empty(v.shape, dtype=np.uint8)
    _load().orc_cast(_ptr(v), IN_F32, v.size, 1.0, fmt, int(saturate), _ptr(out))
    return out


def encode_scalar(v: float, fmt: int, saturate: bool = False) -> int:
    return int(_load().orc_fp8_encode(float(v), fmt, int(saturate)))


def amax(x: np.ndarray) -> np.float32:
    x, dt = _input(x)
    return np.float32(_load().orc_amax(_ptr(x), dt, x.size))


def scale_from_amax(a: float, fmt: int) -> np.float32:
    return np.float32(_load().orc_scale_from_amax(float(a), fmt))


def cast(x: np.ndarray, s: float, fmt: int, saturate: bool = False) -> np.ndarray:
    x, dt = _input(x)
    q = np.empty(x.shape, dtype=np.uint8)
    _load().orc_cast(_ptr(x), dt, x.size, float(s), fmt, int(saturate), _ptr(q))
    return q


def quantize_tensor(x: np.ndarray, fmt: int, s: float | None = None, saturate=False,
                    want_q=True, want_qt=False):
    """Per-tensor current scaling.  Returns (q, q_t, s); s defaults to
    scale_from_amax(amax(x))."""
    x, dt = _input(x)
    if x.ndim == 1:
        q, qt, s = quantize_tensor(x[None, :], fmt, s, saturate, want_q, want_qt)
        return (None if q is None else q[0]), qt, s
    rows, cols = x.shape
    if s is None:
        s = scale_from_amax(amax(x), fmt)
    q = np.empty((rows, cols), np.uint8) if want_q else None
    qt = np.empty((cols, rows), np.uint8) if want_qt else None
    _load().orc_quantize_tensor(_ptr(x), dt, rows, cols, float(s), fmt, int(saturate),
                                _ptr(q), _ptr(qt))
    return q, qt, np.float32(s)


def quantize_tile_rows(x: np.ndarray, fmt: int, saturate=False):
    x, dt = _input(x)
    rows, cols = x.shape
    q = np.empty((rows, cols), np.uint8)
    sc = np.empty(((cols + 127) // 128, rows), np.float32)
    _load().orc_quantize_tile_rows(_ptr(x), dt, rows, cols, fmt, int(saturate), _ptr(q), _ptr(sc))
    return q, sc


def quantize_tile_cols(x: np.ndarray, fmt: int, saturate=False):
    x, dt = _input(x)
    rows, cols = x.shape
    qt = np.empty((cols, rows), np.uint8)
    sc = np.empty(((rows + 127) // 128, cols), np.float32)
    _load().orc_quantize_tile_cols(_ptr(x), dt, rows, cols, fmt, int(saturate), _ptr(qt), _ptr(sc))
    return qt, sc


def quantize_block(x: np.ndarray, fmt: int, saturate=False, want_q=True, want_qt=False):
    x, dt = _input(x)
    rows, cols = x.shape
    q = np.empty((rows, cols), np.uint8) if want_q else None
    qt = np.empty((cols, rows), np.uint8) if want_qt else None
    sc = np.empty(((rows + 127) // 128, (cols + 127) // 128), np.float32)
    _load().orc_quantize_block(_ptr(x), dt, rows, cols, fmt, int(saturate), _ptr(q), _ptr(qt),
                               _ptr(sc))
    return q, qt, sc


def quantize_rowwise(x: np.ndarray, fmt: int, rows=True, cols=False, saturate=False):
    """Row-wise scaling.  Returns (q [R,C], q_scales [R], q_t [C,R], qt_scales [C]),
    with None for the pair not requested."""
    x, dt = _input(x)
    R, C = x.shape
    q = np.empty((R, C), np.uint8) if rows else None
    qs = np.empty(R, np.float32) if rows else None
    qt = np.empty((C, R), np.uint8) if cols else None
    qts = np.empty(C, np.float32) if cols else None
    _load().orc_quantize_rowwise(_ptr(x), dt, R, C, fmt, int(saturate), _ptr(q), _ptr(qs),
                                 _ptr(qt), _ptr(qts))
    return q, qs, qt, qts


def quantize_delayed(x: np.ndarray, fmt: int, history: np.ndarray, next_slot: int,
                     saturate=False, want_q=True, want_qt=False):
    """Returns (q, q_t, s, new_history, new_next)."""
    x, dt = _input(x)
    rows, cols = x.shape
    h = np.ascontiguousarray(np.array(history, dtype=np.float32))
    nxt = ctypes.c_int32(int(next_slot))
    q = np.empty((rows, cols), np.uint8) if want_q else None
    qt = np.empty((cols, rows), np.uint8) if want_qt else None
    s = _load().orc_quantize_delayed(_ptr(x), dt, rows, cols, fmt, int(saturate), _ptr(h),
                                     h.size, ctypes.addressof(nxt), _ptr(q), _ptr(qt))
    return q, qt, np.float32(s), h, nxt.value


# ------------------------------------------------------------------ MXFP8

def e8m0_decode(codes) -> np.ndarray:
    """E8M0 scale bytes -> 2^(code - 127) (NaN for 0xFF)."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.orc_e8m0_decode(int(b)) for b in c.ravel()],
                    dtype=np.float64).reshape(c.shape)


def mx_scale_code(amax: float, fmt: int) -> int:
    return int(_load().orc_mx_scale_code(float(amax), fmt))


def quantize_mx_rows(x: np.ndarray, fmt: int):
    """MXFP8 1x32 blocks along each row: (q [R, C], scales [R, ceil(C/32)] E8M0)."""
    x, dt = _input(x)
    rows, cols = x.shape
    q = np.empty((rows, cols), np.uint8)
    sc = np.empty((rows, (cols + MX_BLOCK - 1) // MX_BLOCK), np.uint8)
    _load().orc_quantize_mx_rows(_ptr(x), dt, rows, cols, fmt, _ptr(q), _ptr(sc))
    return q, sc


def quantize_mx_cols(x: np.ndarray, fmt: int):
    """MXFP8 32x1 blocks down each column, written transposed:
    (q_t [C, R], scales [C, ceil(R/32)] E8M0)."""
    x, dt = _input(x)
    rows, cols = x.shape
    qt = np.empty((cols, rows), np.uint8)
    sc = np.empty((cols, (rows + MX_BLOCK - 1) // MX_BLOCK), np.uint8)
    _load().orc_quantize_mx_cols(_ptr(x), dt, rows, cols, fmt, _ptr(qt), _ptr(sc))
    return qt, sc


def dequantize(q: np.ndarray, fmt: int, s: float) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    d = np.empty(q.shape, np.float32)
    _load().orc_dequantize(_ptr(q), q.size, fmt, float(s), _ptr(d))
    return d


def scaled_roundtrip(x: np.ndarray, fmt: int, s: float | None = None):
    """Dequantised per-tensor round trip and its scale (the page's
    ``scaled_roundtrip``), on the oracle."""
    q, _, s = quantize_tensor(x, fmt, s)
    return dequantize(q, fmt, s), s


class GemmOperand:
    """Keeps the numpy buffers alive alongside the ctypes struct."""

    def __init__(self, data: np.ndarray, fmt: int, scaling: int = SCALE_TENSOR,
                 scale=None, stride_row: int = 0, stride_k: int = 0):
        self.data = np.ascontiguousarray(data, dtype=np.uint8)
        self.rows, self.K = self.data.shape
        if scaling == SCALE_MX:
            self.mx = np.ascontiguousarray(np.asarray(scale, dtype=np.uint8))
            self.scale = np.zeros(1, np.float32)
            mx_ptr = self.mx.ctypes.data
        else:
            self.scale = np.ascontiguousarray(np.atleast_1d(np.asarray(scale, dtype=np.float32)))
            mx_ptr = None
        self.struct = Operand(self.data.ctypes.data, fmt, scaling, self.scale.ctypes.data,
                              stride_row, stride_k, mx_ptr)

    @classmethod
    def tensor(cls, q, fmt, s):
        return cls(q, fmt, SCALE_TENSOR, np.float32(s))

    @classmethod
    def tile(cls, q, fmt, scales):
        """1x128 tiles with scales laid out [ceil(K/128), rows]."""
        return cls(q, fmt, SCALE_TILE, scales, stride_row=1, stride_k=q.shape[0])

    @classmethod
    def row(cls, q, fmt, scales):
        """One scale per row over all of K (scales [rows])."""
        return cls(q, fmt, SCALE_ROW, scales, stride_row=1, stride_k=0)

    @classmethod
    def mx(cls, q, fmt, scales):
        """MXFP8: E8M0 codes [rows, ceil(K/32)] row-major (as quantize_mx_rows
        and quantize_mx_cols return them)."""
        sc = np.asarray(scales, dtype=np.uint8)
        return cls(q, fmt, SCALE_MX, sc, stride_row=sc.shape[1], stride_k=1)

    @classmethod
    def block(cls, q, fmt, scales, transposed=False):
        """128x128 blocks; scales [ceil(rows/128), ceil(K/128)] row-major, or
        the transpose of such an array when ``transposed``."""
        sc = np.asarray(scales, dtype=np.float32)
        if transposed:  # scales given as [kb][rb]
            return cls(q, fmt, SCALE_BLOCK, sc, stride_row=1, stride_k=sc.shape[1])
        return cls(q, fmt, SCALE_BLOCK, sc, stride_row=sc.shape[1], stride_k=1)


def gemm_points(A: GemmOperand, B: GemmOperand, ms, ns):
    """Reference outputs y[i] = C[ms[i], ns[i]] and sum_k |a_k b_k|."""
    assert A.K == B.K
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    y = np.empty(ms.size, np.float64)
    ab = np.empty(ms.size, np.float64)
    _load().orc_gemm_points(ctypes.byref(A.struct), ctypes.byref(B.struct), A.K, ms.size,
                            _ptr(ms), _ptr(ns), _ptr(y), _ptr(ab))
    return y, ab


def gemm_rows(A: GemmOperand, B: GemmOperand, m0: int = 0, m1: int | None = None):
    """Dense reference block C[m0:m1, :] and its sum_k |a_k b_k|."""
    assert A.K == B.K
    m1 = A.rows if m1 is None else m1
    N = B.rows
    y = np.empty((m1 - m0, N), np.float64)
    ab = np.empty((m1 - m0, N), np.float64)
    _load().orc_gemm_rows(ctypes.byref(A.struct), ctypes.byref(B.struct), N, A.K, m0, m1,
                          _ptr(y), _ptr(ab))
    return y, ab


def gemm_bound(y_ref: np.ndarray, absum: np.ndarray, out_bf16: bool) -> np.ndarray:
    """Per-element tolerance: 2e-6 * sum|a b| + 1e-6, plus one bf16 ulp of
    y_ref when the output is bf16."""
    tol = 2e-6 * absum + 1e-6
    if out_bf16:
        tol = tol + bf16_ulp(y_ref)
    return tol


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (8 significant bits)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 7).astype(np.int64))
