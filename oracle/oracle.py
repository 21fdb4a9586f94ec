"""Python face of the CPU oracle (``oracle_gemm.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / reference leg are the only callers.  Nothing
here imports the product package, and the product package never imports
this module.

The oracle computes ``D = alpha * op(A) @ op(B) + beta * C`` by the plain
definition in binary64 (TVM TIRx "gemm" page, opening paragraph and the
"What it accepts" table; Phobos "@tensorcore" page, the
gemm_fp16tc_fp32acc.ph epilogue), and the per-element error bound
``|alpha| * sum_k |a_ik * b_kj| + |beta| * |c_ij|``.

With ``sfa`` / ``sfb`` given, the 8-bit operands are MX block-scaled: every
32 consecutive K elements of a row of op(A) share the UE8M0 scale
``2^(sfa[i, k // 32] - 127)``, and of a column of op(B) the scale
``2^(sfb[j, k // 32] - 127)`` (``sfa`` is [M, ceil(K/32)], ``sfb`` is
[N, ceil(K/32)], uint8; 255 is NaN) -- the OCP Microscaling reading of the
"block scaling (SFA / SFB)" the TIRx gemm guide lists in section 七.

E2M1 (the OCP 4-bit format; fp4 in the guide's list of precisions) is
stored packed, two elements per byte, element e of a row-major array
(e = row * ld + col) in the low nibble of byte e // 2 when e is even and in
the high nibble when it is odd; its leading dimensions count elements.

Inputs are numpy arrays or torch CPU tensors: A and B hold fp16 / bf16
bits, or E4M3 / E5M2 bits (one byte each; the 8-bit precisions of the
tcgen05 path the TIRx gemm guide lists in section 七); C holds fp32 (or
fp16 / bf16 bits when the output is 16-bit).  Row-major with explicit
leading dimensions.
"""
from __future__ import annotations

import concurrent.futures as _cf
import ctypes
import os
import subprocess
import threading

import numpy as np

F16, BF16, F32, E4M3, E5M2, E2M1 = 0, 1, 2, 3, 4, 5
FP8 = (E4M3, E5M2)
PACKED = (E2M1,)   # two elements per byte, even elements in the low nibble

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle_gemm.c")
LIBRARY = os.path.join(_HERE, "liboracle_gemm.so")
CFLAGS = ["-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC"]


def compile_library(src: str, out: str) -> str:
    """gcc ``src`` into the shared library ``out`` (atomically replaced)."""
    tmp = out + ".tmp.%d" % os.getpid()
    subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, src, "-lm", "-lpthread"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``oracle_gemm.c`` into ``liboracle_gemm.so`` beside it."""
    if force or not os.path.exists(LIBRARY) or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE):
        compile_library(SOURCE, LIBRARY)
    return LIBRARY


def _bits16(x):
    """A 2-D uint16 array of fp16 / bf16 bit patterns."""
    if x is None:
        return None
    if hasattr(x, "detach"):                      # torch tensor
        import torch
        x = x.detach().cpu().contiguous().view(torch.int16).numpy()
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        x = x.view(np.uint16)
    if x.dtype not in (np.uint16, np.int16):
        raise TypeError("16-bit operand expected, got %s" % x.dtype)
    return x.view(np.uint16)


def _bits8(x):
    """A 2-D uint8 array of E4M3 / E5M2 bit patterns."""
    if x is None:
        return None
    if hasattr(x, "detach"):                      # torch tensor (float8 or uint8)
        import torch
        x = x.detach().cpu().contiguous().view(torch.uint8).numpy()
    x = np.ascontiguousarray(x)
    if x.dtype not in (np.uint8, np.int8):
        raise TypeError("8-bit operand expected, got %s" % x.dtype)
    return x.view(np.uint8)


def _operand(x, in_dtype):
    return _bits8(x) if (in_dtype in FP8 or in_dtype in PACKED) else _bits16(x)


def _ld_operand(arr, default, in_dtype):
    """Leading dimension in elements (a packed byte row holds two)."""
    if arr is not None and arr.ndim == 2 and in_dtype in PACKED:
        return 2 * arr.shape[1]
    return _ld(arr, default)


def _c_array(c, c_dtype):
    if c is None:
        return None
    if hasattr(c, "detach"):
        import torch
        c = c.detach().cpu().contiguous()
        c = c.numpy() if c.dtype == torch.float32 else c.view(torch.int16).numpy()
    c = np.ascontiguousarray(c)
    if c_dtype == F32:
        if c.dtype != np.float32:
            raise TypeError("fp32 C expected, got %s" % c.dtype)
        return c
    return _bits16(c)


def _scales(x):
    """A 2-D uint8 array of UE8M0 scale bytes."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        import torch
        x = x.detach().cpu().contiguous().view(torch.uint8).numpy()
    x = np.ascontiguousarray(x)
    if x.dtype not in (np.uint8, np.int8):
        raise TypeError("uint8 scales expected, got %s" % x.dtype)
    return x.view(np.uint8)


def _ptr(a):
    return None if a is None else a.ctypes.data


def _ld(arr, default):
    return arr.shape[1] if arr is not None and arr.ndim == 2 else default


class Oracle:
    """One loaded build of the oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        lib.oracle_decode_f16.restype = dbl
        lib.oracle_decode_f16.argtypes = [ctypes.c_uint16]
        lib.oracle_decode_bf16.restype = dbl
        lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
        lib.oracle_decode_e4m3.restype = dbl
        lib.oracle_decode_e4m3.argtypes = [ctypes.c_uint8]
        lib.oracle_decode_e5m2.restype = dbl
        lib.oracle_decode_e5m2.argtypes = [ctypes.c_uint8]
        lib.oracle_gemm.restype = i32
        lib.oracle_gemm.argtypes = [vp, vp, i64, vp, vp, vp, i64, i64, i64, i64, i64, i64,
                                    i32, i32, dbl, dbl, i32, i32, i64, i64]
        lib.oracle_gemm_entries.restype = i32
        lib.oracle_gemm_entries.argtypes = [vp, vp, vp, vp, i64, vp, vp, vp, i64, i64, i64,
                                            i64, i64, i64, i32, i32, dbl, dbl, i32, i32]
        lib.oracle_decode_e2m1.restype = dbl
        lib.oracle_decode_e2m1.argtypes = [ctypes.c_uint8]
        lib.oracle_decode_ue8m0.restype = dbl
        lib.oracle_decode_ue8m0.argtypes = [ctypes.c_uint8]
        lib.oracle_gemm_mx.restype = i32
        lib.oracle_gemm_mx.argtypes = [vp, vp, i64, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64,
                                       i64, i64, i64, i32, i32, dbl, dbl, i32, i32, i64, i64]
        lib.oracle_gemm_mx_entries.restype = i32
        lib.oracle_gemm_mx_entries.argtypes = [vp, vp, vp, vp, i64, vp, vp, vp, vp, vp, i64, i64,
                                               i64, i64, i64, i64, i64, i64, i32, i32, dbl, dbl,
                                               i32, i32]
        self.lib = lib
        self.path = path

    def decode_f16(self, bits: int) -> float:
        return self.lib.oracle_decode_f16(int(bits))

    def decode_bf16(self, bits: int) -> float:
        return self.lib.oracle_decode_bf16(int(bits))

    def decode_e4m3(self, bits: int) -> float:
        return self.lib.oracle_decode_e4m3(int(bits))

    def decode_e5m2(self, bits: int) -> float:
        return self.lib.oracle_decode_e5m2(int(bits))

    def decode_e2m1(self, bits: int) -> float:
        return self.lib.oracle_decode_e2m1(int(bits))

    def decode_ue8m0(self, bits: int) -> float:
        return self.lib.oracle_decode_ue8m0(int(bits))

    def gemm(self, A, B, C, M, N, K, *, transA=0, transB=0, alpha=1.0, beta=0.0,
             in_dtype=F16, c_dtype=F32, lda=None, ldb=None, ldc=None,
             rows=None, threads=1, sfa=None, sfb=None, ld_sfa=None, ld_sfb=None):
        """Full rows of D (all rows unless ``rows=(begin, end)``).

        Returns ``(D, bound)``: float64 arrays of shape [M, N]; rows outside
        the requested range stay NaN.  ``threads > 1`` runs disjoint row
        blocks of the same single-threaded C loop concurrently.  ``sfa`` and
        ``sfb`` (both or neither) make the 8-bit operands MX block-scaled.
        """
        mx = _mx_args(sfa, sfb, ld_sfa, ld_sfb, K)
        Ab, Bb = _operand(A, in_dtype), _operand(B, in_dtype)
        C_ = _c_array(C, c_dtype) if beta != 0.0 else None
        lda = lda if lda is not None else _ld_operand(Ab, M if transA else K, in_dtype)
        ldb = ldb if ldb is not None else _ld_operand(Bb, K if transB else N, in_dtype)
        ldc = ldc if ldc is not None else _ld(C_, N)
        D = np.full((M, N), np.nan)
        bound = np.full((M, N), np.nan)
        r0, r1 = rows if rows is not None else (0, M)
        lib = self.lib

        def run(a, b):
            if mx is None:
                rc = lib.oracle_gemm(D.ctypes.data, bound.ctypes.data, N, _ptr(Ab), _ptr(Bb),
                                     _ptr(C_), M, N, K, lda, ldb, ldc, int(transA), int(transB),
                                     float(alpha), float(beta), int(in_dtype), int(c_dtype), a, b)
            else:
                sa, sb, la, lb = mx
                rc = lib.oracle_gemm_mx(D.ctypes.data, bound.ctypes.data, N, _ptr(Ab), _ptr(Bb),
                                        _ptr(C_), _ptr(sa), _ptr(sb), M, N, K, lda, ldb, ldc, la, lb,
                                        int(transA), int(transB), float(alpha), float(beta),
                                        int(in_dtype), int(c_dtype), a, b)
            if rc != 0:
                raise ValueError("oracle_gemm rejected its arguments")

        if threads <= 1 or r1 - r0 < 2:
            run(r0, r1)
        else:
            step = max(1, (r1 - r0 + threads * 4 - 1) // (threads * 4))
            with _cf.ThreadPoolExecutor(threads) as ex:
                list(ex.map(lambda a: run(a, min(a + step, r1)), range(r0, r1, step)))
        return D, bound

    def gemm_entries(self, A, B, C, M, N, K, rows, cols, *, transA=0, transB=0, alpha=1.0,
                     beta=0.0, in_dtype=F16, c_dtype=F32, lda=None, ldb=None, ldc=None,
                     threads=1, sfa=None, sfb=None, ld_sfa=None, ld_sfb=None):
        """D and bound at the listed (rows[e], cols[e]) positions only."""
        mx = _mx_args(sfa, sfb, ld_sfa, ld_sfb, K)
        Ab, Bb = _operand(A, in_dtype), _operand(B, in_dtype)
        C_ = _c_array(C, c_dtype) if beta != 0.0 else None
        lda = lda if lda is not None else _ld_operand(Ab, M if transA else K, in_dtype)
        ldb = ldb if ldb is not None else _ld_operand(Bb, K if transB else N, in_dtype)
        ldc = ldc if ldc is not None else _ld(C_, N)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        cols = np.ascontiguousarray(cols, dtype=np.int64)
        n = rows.shape[0]
        D = np.empty(n)
        bound = np.empty(n)
        lib = self.lib

        def run(a, b):
            if mx is None:
                rc = lib.oracle_gemm_entries(D[a:].ctypes.data, bound[a:].ctypes.data,
                                             rows[a:].ctypes.data, cols[a:].ctypes.data, b - a,
                                             _ptr(Ab), _ptr(Bb), _ptr(C_), M, N, K, lda, ldb, ldc,
                                             int(transA), int(transB), float(alpha), float(beta),
                                             int(in_dtype), int(c_dtype))
            else:
                sa, sb, la, lb = mx
                rc = lib.oracle_gemm_mx_entries(D[a:].ctypes.data, bound[a:].ctypes.data,
                                                rows[a:].ctypes.data, cols[a:].ctypes.data, b - a,
                                                _ptr(Ab), _ptr(Bb), _ptr(C_), _ptr(sa), _ptr(sb),
                                                M, N, K, lda, ldb, ldc, la, lb,
                                                int(transA), int(transB), float(alpha),
                                                float(beta), int(in_dtype), int(c_dtype))
            if rc != 0:
                raise ValueError("oracle_gemm_entries rejected its arguments")

        if n == 0:
            return D, bound
        if threads <= 1 or n < 2:
            run(0, n)
        else:
            step = max(1, (n + threads * 4 - 1) // (threads * 4))
            with _cf.ThreadPoolExecutor(threads) as ex:
                list(ex.map(lambda a: run(a, min(a + step, n)), range(0, n, step)))
        return D, bound


def _mx_args(sfa, sfb, ld_sfa, ld_sfb, K):
    """(sfa, sfb, ld_sfa, ld_sfb) as the C oracle takes them, or None."""
    if sfa is None and sfb is None:
        return None
    if sfa is None or sfb is None:
        raise ValueError("block scaling needs both sfa and sfb")
    sa, sb = _scales(sfa), _scales(sfb)
    kb = (K + 31) // 32
    return (sa, sb, ld_sfa if ld_sfa is not None else _ld(sa, kb),
            ld_sfb if ld_sfb is not None else _ld(sb, kb))


_default = None
_default_lock = threading.Lock()


def default() -> Oracle:
    """The oracle built from ``oracle_gemm.c`` (compiled on first use)."""
    global _default
    with _default_lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def gemm(*args, **kwargs):
    return default().gemm(*args, **kwargs)


def gemm_entries(*args, **kwargs):
    return default().gemm_entries(*args, **kwargs)


def decode_f16(bits):
    return default().decode_f16(bits)


def decode_bf16(bits):
    return default().decode_bf16(bits)


def decode_e4m3(bits):
    return default().decode_e4m3(bits)


def decode_e5m2(bits):
    return default().decode_e5m2(bits)


def decode_ue8m0(bits):
    return default().decode_ue8m0(bits)


def decode_e2m1(bits):
    return default().decode_e2m1(bits)
