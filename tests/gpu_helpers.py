"""Shared helpers of the GPU parity tests: run the C ABI on seeded inputs,
run the oracle on the same inputs, compare element by element.

Tolerance (per element, fp32 output):
    |D_gpu - D_ref| <= 1e-3 * (|alpha| * (|A| @ |B|)_ij + |beta| * |C_ij|) + 1e-6
with D_ref and the bound from the oracle (binary64).  For 16-bit outputs
half a unit in the last place of the output format at |D_ref| is added
(the final rounding).  Integer-valued inputs must match bit for bit.
"""
from __future__ import annotations

import contextlib
import os

import numpy as np
import torch

import oracle.oracle as oracle
from dense_tensor_core_02_gb300 import binding

CODE = {"f16": 0, "bf16": 1, "f32": 2, "e4m3": 3, "e5m2": 4, "e2m1": 5}
TORCH = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32, "e4m3": torch.float8_e4m3fn,
         "e5m2": torch.float8_e5m2}
ORACLE_THREADS = max(1, min(16, len(os.sched_getaffinity(0))))


@contextlib.contextmanager
def env(**kw):
    old = {k: os.environ.get(k) for k in kw}
    try:
        for k, v in kw.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = str(v)
        yield
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def run_gemm(A, B, C, M, N, K, *, transA=0, transB=0, alpha=1.0, beta=0.0, in_dtype="f16",
             out_dtype="f32", d_fill=float("nan"), stream=None):
    """Copy CPU inputs to cuda:0, call the C ABI, return (D on CPU, status)."""
    dev = torch.device("cuda", 0)
    Ad = A.to(dev) if A is not None else None
    Bd = B.to(dev) if B is not None else None
    Cd = C.to(dev) if C is not None else None
    D = torch.full((M, N), d_fill, dtype=TORCH[out_dtype], device=dev)
    lda = Ad.stride(0) if Ad is not None and Ad.dim() == 2 else 0
    ldb = Bd.stride(0) if Bd is not None and Bd.dim() == 2 else 0
    ldc = Cd.stride(0) if Cd is not None else N
    rc = binding.gemm(D, Ad, Bd, Cd, M, N, K, lda, ldb, ldc, D.stride(0), transA, transB, alpha, beta,
                      CODE[in_dtype], CODE[out_dtype], stream)
    torch.cuda.synchronize()
    return D.cpu(), rc


def poll():
    rc, info = binding.gemm_poll_device_error()
    return rc, info


def oracle_full(A, B, C, M, N, K, *, transA=0, transB=0, alpha=1.0, beta=0.0, in_dtype="f16",
                out_dtype="f32"):
    return oracle.gemm(A, B, C, M, N, K, transA=transA, transB=transB, alpha=alpha, beta=beta,
                       in_dtype=CODE[in_dtype], c_dtype=CODE[out_dtype], threads=ORACLE_THREADS)


def oracle_at(A, B, C, M, N, K, rows, cols, *, transA=0, transB=0, alpha=1.0, beta=0.0,
              in_dtype="f16", out_dtype="f32"):
    """Oracle at sampled positions.  The operands are handed over in
    K-contiguous storage (a pure copy: same values, flags flipped), so each
    sampled dot product walks memory in order."""
    Ak = A.t().contiguous() if transA else A
    Bk = B if transB else B.t().contiguous()
    return oracle.gemm_entries(Ak, Bk, C, M, N, K, rows, cols, transA=0, transB=1, alpha=alpha,
                               beta=beta, in_dtype=CODE[in_dtype], c_dtype=CODE[out_dtype],
                               threads=ORACLE_THREADS)


def sample_positions(M, N, *, block=128, per_block=8, seed=0):
    """Positions touching every block x block output block: its four corners
    and `per_block` random interior points, plus the last row and column."""
    rng = np.random.default_rng(seed)
    rows, cols = [], []
    for bi in range(0, M, block):
        r1 = min(bi + block, M) - 1
        for bj in range(0, N, block):
            c1 = min(bj + block, N) - 1
            rows += [bi, bi, r1, r1]
            cols += [bj, c1, bj, c1]
            rows += list(rng.integers(bi, r1 + 1, size=per_block))
            cols += list(rng.integers(bj, c1 + 1, size=per_block))
    step_c = max(1, N // 512)
    step_r = max(1, M // 512)
    rows += [M - 1] * len(range(0, N, step_c))
    cols += list(range(0, N, step_c))
    rows += list(range(0, M, step_r))
    cols += [N - 1] * len(range(0, M, step_r))
    return np.array(rows, dtype=np.int64), np.array(cols, dtype=np.int64)


def _half_ulp(x, out_dtype):
    if out_dtype == "f32":
        return np.zeros_like(x)
    mant, emin = (10, -14) if out_dtype == "f16" else (7, -126)
    ax = np.maximum(np.abs(x), 2.0 ** emin)
    e = np.floor(np.log2(ax))
    return 0.5 * np.exp2(e - mant)


def assert_close(d_gpu, d_ref, bound, out_dtype="f32", what=""):
    d = np.asarray(d_gpu, dtype=np.float64)
    tol = 1e-3 * bound + 1e-6 + _half_ulp(d_ref, out_dtype)
    err = np.abs(d - d_ref)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:8]
        detail = ["%s: gpu=%r ref=%r tol=%r" % (tuple(i), d[tuple(i)], d_ref[tuple(i)], tol[tuple(i)])
                  for i in idx]
        raise AssertionError("%s: %d of %d elements outside tolerance\n  %s" % (
            what, int(bad.sum()), bad.size, "\n  ".join(detail)))


def assert_exact(d_gpu, d_ref, what=""):
    d = np.asarray(d_gpu, dtype=np.float64)
    bad = d != d_ref
    if bad.any():
        idx = np.argwhere(bad)[:8]
        detail = ["%s: gpu=%r ref=%r" % (tuple(i), d[tuple(i)], d_ref[tuple(i)]) for i in idx]
        raise AssertionError("%s: %d of %d elements differ\n  %s" % (
            what, int(bad.sum()), bad.size, "\n  ".join(detail)))


def int_matrix(shape, lo, hi, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, shape, generator=g, dtype=torch.int32).float().to(TORCH[dtype])


def normal_matrix(shape, dtype, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(TORCH[dtype])


def strided(host, offset, ld, dtype, fill=float("nan")):
    """Copy a CPU matrix [rows, cols] into a device buffer at element
    `offset` with row stride `ld`; return (flat buffer, view)."""
    rows, cols = host.shape
    dev = torch.device("cuda", 0)
    n = offset + (rows - 1) * ld + cols + 8 if rows else offset + 8
    buf = torch.full((n,), fill, dtype=TORCH[dtype], device=dev)
    view = buf.as_strided((rows, cols), (ld, 1), offset)
    view.copy_(host.to(dev))
    return buf, view


def run_layout(A, B, C, M, N, K, *, offs=(0, 0, 0, 0), lds=None, transA=0, transB=0, alpha=1.0, beta=0.0,
               in_dtype="f16", out_dtype="f32", fn=None):
    """Call the C ABI (gemm, or `fn`) with A, B, C, D placed at element
    offsets `offs` and row strides `lds` (default: the densest legal
    strides); return D on the CPU, the whole D buffer (for canary checks)
    and the status."""
    fn = fn or binding.gemm
    ra, ca = (K, M) if transA else (M, K)
    rb, cb = (N, K) if transB else (K, N)
    lda, ldb, ldc, ldd = lds or (ca, cb, N, N)
    _, Av = strided(A, offs[0], lda, in_dtype)
    _, Bv = strided(B, offs[1], ldb, in_dtype)
    Cv = strided(C, offs[2], ldc, out_dtype)[1] if C is not None else None
    Dbuf, Dv = strided(torch.full((M, N), float("nan")), offs[3], ldd, out_dtype)
    rc = fn(Dv, Av, Bv, Cv, M, N, K, lda, ldb, ldc if C is not None else N, ldd, transA, transB, alpha, beta,
            CODE[in_dtype], CODE[out_dtype], None)
    torch.cuda.synchronize()
    return Dv.cpu(), Dbuf.cpu(), rc


def check_canaries(Dbuf, M, N, off, ldd):
    """Everything in the D buffer outside the M x N view is still NaN."""
    flat = Dbuf.double().numpy()
    mask = np.ones(flat.shape, dtype=bool)
    for r in range(M):
        mask[off + r * ldd: off + r * ldd + N] = False
    assert np.isnan(flat[mask]).all(), "elements outside D written"


def tflops(M, N, K, ms):
    return 2.0 * M * N * K / (ms * 1e-3) / 1e12


def ceil_div(a, b):
    return -(-a // b)

