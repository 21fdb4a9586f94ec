"""ctypes binding of libgemm_gb300.so (the C ABI in include/gemm_gb300.h).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  Buffers may be given as torch tensors (their
``data_ptr()`` is passed) or as raw integer addresses; the stream as a
``torch.cuda.Stream``, a raw ``cudaStream_t`` integer, or ``None`` for
torch's current stream.  There is no fallback: if the library has not been
built, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

F16, BF16, F32, E4M3, E5M2, E2M1 = 0, 1, 2, 3, 4, 5
GEMM_OK = 0
GEMM_ERR_DEVICE_TIMEOUT = -8
GEMM_ERR_UNSUPPORTED_LAYOUT = -10

LIBRARY_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgemm_gb300.so")

_lock = threading.Lock()
_lib = None


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str = "gemm"):
        self.status = status
        super().__init__("%s failed: %s (%d)" % (what, gemm_status_string(status), status))


def load_library():
    """Load libgemm_gb300.so (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIBRARY_PATH):
                raise RuntimeError(
                    "libgemm_gb300.so is not built (%s); build it with "
                    "`python -m dense_tensor_core_02_gb300.build` or __graft_entry__.build()" % LIBRARY_PATH)
            lib = ctypes.CDLL(LIBRARY_PATH)
            i64, i32, vp, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_float
            lib.gemm.restype = i32
            lib.gemm.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64, i32, i32, f32, f32,
                                 i32, i32, vp]
            lib.gemm_status_string.restype = ctypes.c_char_p
            lib.gemm_status_string.argtypes = [i32]
            lib.gemm_poll_device_error.restype = i32
            lib.gemm_poll_device_error.argtypes = [vp, ctypes.POINTER(i32)]
            lib.gemm_tile_coords.restype = i32
            lib.gemm_tile_coords.argtypes = [i32, i32, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]
            lib.gemm_plan.restype = i32
            lib.gemm_plan.argtypes = [i64, i64, i64, i32, ctypes.POINTER(i64)]
            lib.gemm_plan_layout.restype = i32
            lib.gemm_plan_layout.argtypes = [i64, i64, i64, i32, i32, i32, i32, ctypes.POINTER(i64)]
            lib.gemm_noalloc.restype = i32
            lib.gemm_noalloc.argtypes = list(lib.gemm.argtypes)
            lib.gemm_host.restype = i32
            lib.gemm_host.argtypes = list(lib.gemm.argtypes)
            lib.gemm_mx.restype = i32
            lib.gemm_mx.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64, i64, i64,
                                    i32, i32, f32, f32, i32, i32, vp]
            lib.gemm_schedule_units.restype = i32
            lib.gemm_schedule_units.argtypes = [i32, i32, i32, i32, i32, ctypes.POINTER(i32), i32]
            _lib = lib
    return _lib


def library():
    return load_library()


def _addr(x):
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return int(x)


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return int(stream)


def gemm(D, A, B, C, M, N, K, lda, ldb, ldc, ldd, transA, transB, alpha, beta,
         in_dtype, out_dtype, stream=None) -> int:
    """The C entry point ``gemm`` with the same arguments; returns its status."""
    lib = load_library()
    return lib.gemm(_addr(D), _addr(A), _addr(B), _addr(C), int(M), int(N), int(K), int(lda), int(ldb),
                    int(ldc), int(ldd), int(transA), int(transB), float(alpha), float(beta),
                    int(in_dtype), int(out_dtype), _stream(stream))


def gemm_noalloc(D, A, B, C, M, N, K, lda, ldb, ldc, ldd, transA, transB, alpha, beta,
                 in_dtype, out_dtype, stream=None) -> int:
    """The C entry point ``gemm_noalloc``: what ``gemm`` computes, for callers
    that cannot allocate device memory (the library then uses a fixed static
    scratch record instead of a cudaMalloc'd one).  Returns its status."""
    lib = load_library()
    return lib.gemm_noalloc(_addr(D), _addr(A), _addr(B), _addr(C), int(M), int(N), int(K), int(lda),
                            int(ldb), int(ldc), int(ldd), int(transA), int(transB), float(alpha),
                            float(beta), int(in_dtype), int(out_dtype), _stream(stream))


def gemm_host(D, A, B, C, M, N, K, lda, ldb, ldc, ldd, transA, transB, alpha, beta,
              in_dtype, out_dtype, stream=None) -> int:
    """The C entry point ``gemm_host``: what ``gemm`` computes, with A, B, C
    and D in host memory (pinned for asynchronous copies); D is complete
    once ``stream`` has completed the call.  Returns its status."""
    lib = load_library()
    return lib.gemm_host(_addr(D), _addr(A), _addr(B), _addr(C), int(M), int(N), int(K), int(lda), int(ldb),
                         int(ldc), int(ldd), int(transA), int(transB), float(alpha), float(beta), int(in_dtype),
                         int(out_dtype), _stream(stream))


def gemm_mx(D, A, B, C, SFA, SFB, M, N, K, lda, ldb, ldc, ldd, ld_sfa, ld_sfb, transA, transB, alpha, beta,
            in_dtype, out_dtype, stream=None) -> int:
    """The C entry point ``gemm_mx``: ``gemm`` with MX block-scaled E4M3 /
    E5M2 / packed E2M1 operands (one UE8M0 scale byte per 32 K elements of
    each row of op(A), SFA [M, ceil(K/32)], and of each column of op(B),
    SFB [N, ceil(K/32)]).  Returns its status."""
    lib = load_library()
    return lib.gemm_mx(_addr(D), _addr(A), _addr(B), _addr(C), _addr(SFA), _addr(SFB), int(M), int(N), int(K),
                       int(lda), int(ldb), int(ldc), int(ldd), int(ld_sfa), int(ld_sfb), int(transA), int(transB),
                       float(alpha), float(beta), int(in_dtype), int(out_dtype), _stream(stream))


def gemm_status_string(status: int) -> str:
    return load_library().gemm_status_string(int(status)).decode()


def gemm_poll_device_error(stream=None):
    """Synchronise ``stream``; read and clear one status record of the
    current device (gemm()'s or gemm_noalloc()'s, whichever holds an error;
    nothing is created or allocated); return (status, [code, block, site,
    detail])."""
    info = (ctypes.c_int * 4)()
    rc = load_library().gemm_poll_device_error(_stream(stream), info)
    return rc, list(info)


def gemm_tile_coords(tile, num_m, num_n, group_m):
    m = ctypes.c_int()
    n = ctypes.c_int()
    rc = load_library().gemm_tile_coords(int(tile), int(num_m), int(num_n), int(group_m),
                                         ctypes.byref(m), ctypes.byref(n))
    if rc != GEMM_OK:
        raise GemmError(rc, "gemm_tile_coords")
    return m.value, n.value


_PLAN_KEYS = ("cta_pair", "tile_m", "tile_n", "num_tiles", "grid", "smem_bytes", "epi_warps", "stages",
              "sk_tiles", "workspace_bytes")


def gemm_plan(M, N, K, num_sms):
    out = (ctypes.c_int64 * 10)()
    rc = load_library().gemm_plan(int(M), int(N), int(K), int(num_sms), out)
    if rc != GEMM_OK:
        raise GemmError(rc, "gemm_plan")
    return dict(zip(_PLAN_KEYS, list(out)))


def gemm_plan_layout(M, N, K, transB, in_dtype, out_dtype, num_sms):
    """The configuration gemm() would choose for this layout and these types."""
    out = (ctypes.c_int64 * 10)()
    rc = load_library().gemm_plan_layout(int(M), int(N), int(K), int(transB), int(in_dtype), int(out_dtype),
                                         int(num_sms), out)
    if rc != GEMM_OK:
        raise GemmError(rc, "gemm_plan_layout")
    return dict(zip(_PLAN_KEYS, list(out)))


def gemm_schedule_units(num_tiles, iters, workers, sk_tiles, worker):
    """The work units of one worker: list of (tile, kb, ke, sk, ci, nc)."""
    lib = load_library()
    n = lib.gemm_schedule_units(int(num_tiles), int(iters), int(workers), int(sk_tiles), int(worker), None, 0)
    if n < 0:
        raise GemmError(n, "gemm_schedule_units")
    buf = (ctypes.c_int * (6 * max(n, 1)))()
    lib.gemm_schedule_units(int(num_tiles), int(iters), int(workers), int(sk_tiles), int(worker), buf, n)
    return [tuple(buf[6 * i:6 * i + 6]) for i in range(n)]


_DT = {}


def _dtype_code(t):
    import torch
    if not _DT:
        _DT.update({torch.float16: F16, torch.bfloat16: BF16, torch.float32: F32})
    return _DT[t.dtype]


def gemm_tensors(A, B, C=None, *, transA=0, transB=0, alpha=1.0, beta=0.0, out=None,
                 out_dtype=None, stream=None):
    """Tensor front end: reads sizes, strides and dtypes off torch tensors.

    A, B are 2-D row-major (stride(1) == 1) CUDA tensors of one 16-bit
    dtype; C (when beta != 0) and ``out`` are [M, N] row-major.  ``out`` is
    allocated with torch when not given.  Raises GemmError on a non-zero
    status.
    """
    import torch
    M = A.shape[1] if transA else A.shape[0]
    K = A.shape[0] if transA else A.shape[1]
    N = B.shape[0] if transB else B.shape[1]
    for name, t in (("A", A), ("B", B), ("C", C), ("out", out)):
        if t is not None and t.dim() == 2 and t.stride(1) != 1 and t.shape[1] > 1:
            raise ValueError("%s must be row-major (stride(1) == 1)" % name)
    if out is None:
        odt = out_dtype if out_dtype is not None else (C.dtype if C is not None else torch.float32)
        out = torch.empty((M, N), dtype=odt, device=A.device)
    rc = gemm(out, A, B, C if beta != 0 else None, M, N, K, A.stride(0), B.stride(0),
              C.stride(0) if (C is not None and beta != 0) else N, out.stride(0), transA, transB,
              alpha, beta, _dtype_code(A), _dtype_code(out), stream)
    if rc != GEMM_OK:
        raise GemmError(rc)
    return out
