"""The C ABI on the CPU: symbols, status strings, host-side validation,
the persistent tile order and the launch plan.  No call here reaches a GPU:
every rejection below happens before the library touches the device.
"""
import ctypes
import glob
import os
import re

import pytest

from dense_tensor_core_02_gb300 import binding
from dense_tensor_core_02_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return binding.load_library()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"GEMM_API\s+[\w\s\*]+?\b(\w+)\s*\(", text):
            names.add(m.group(1))
    return names


def test_header_declares_the_abi():
    assert {"gemm", "gemm_status_string", "gemm_poll_device_error", "gemm_tile_coords",
            "gemm_plan"} <= _declared_functions()


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    names = {0: "GEMM_OK", -1: "GEMM_ERR_INVALID_ARG", -2: "GEMM_ERR_UNSUPPORTED_DTYPE",
             -3: "GEMM_ERR_MISALIGNED", -4: "GEMM_ERR_ALIAS", -5: "GEMM_ERR_ARCH",
             -6: "GEMM_ERR_LAUNCH", -7: "GEMM_ERR_CUDA", -8: "GEMM_ERR_DEVICE_TIMEOUT",
             -9: "GEMM_ERR_TOO_LARGE"}
    for code, name in names.items():
        assert binding.gemm_status_string(code) == name
    assert binding.gemm_status_string(12345) == "GEMM_ERR_UNKNOWN"


# Fake, 16-byte-aligned, non-overlapping device addresses: validation never
# dereferences them, and every case below is rejected before any CUDA call.
A_ = 0x10000000
B_ = 0x20000000
C_ = 0x30000000
D_ = 0x40000000
OK_ARGS = dict(D=D_, A=A_, B=B_, C=C_, M=64, N=64, K=64, lda=64, ldb=64, ldc=64, ldd=64,
               transA=0, transB=0, alpha=1.0, beta=1.0, in_dtype=0, out_dtype=2)


def _call(**kw):
    a = dict(OK_ARGS)
    a.update(kw)
    return binding.gemm(a["D"], a["A"], a["B"], a["C"], a["M"], a["N"], a["K"], a["lda"], a["ldb"],
                        a["ldc"], a["ldd"], a["transA"], a["transB"], a["alpha"], a["beta"],
                        a["in_dtype"], a["out_dtype"], 0)


REJECTIONS = [
    (dict(in_dtype=2), -2),                 # fp32 operands
    (dict(in_dtype=7), -2),
    (dict(out_dtype=9), -2),
    (dict(M=-1), -1),
    (dict(K=-3), -1),
    (dict(transA=2), -1),
    (dict(transB=-1), -1),
    (dict(D=0), -1),
    (dict(C=0), -1),                        # beta != 0 needs C
    (dict(A=0), -1),
    (dict(ldd=63), -1),
    (dict(ldc=63), -1),
    (dict(lda=63), -1),                     # A stored [M, K]: lda >= K
    (dict(transA=1, M=80, lda=64), -1),     # A stored [K, M]: lda >= M
    (dict(ldb=63), -1),                     # B stored [K, N]: ldb >= N
    (dict(transB=1, K=80, ldb=64, lda=80), -1),
    (dict(A=A_ + 2), -3),                   # not 16-byte aligned
    (dict(D=D_ + 8), -3),
    (dict(C=C_ + 4), -3),
    (dict(K=60, lda=60), -3),               # 60 * 2 bytes is not a multiple of 16
    (dict(N=62, ldd=62, ldc=64, ldb=64), -3),   # 62 * 4 bytes
    (dict(out_dtype=0, N=60, ldd=60, ldc=64), -3),    # 60 * 2 bytes
    (dict(D=A_), -4),                       # D overlaps A
    (dict(D=B_ + 256), -4),                 # D overlaps B
    (dict(C=D_ + 4096), -4),                # C overlaps D without being D
    (dict(C=D_, ldc=72), -4),               # C == D but different strides
    (dict(M=1 << 31, lda=64), -9),
]


@pytest.mark.parametrize("kw,code", REJECTIONS, ids=[str(r[0]) for r in REJECTIONS])
def test_rejected_before_any_device_work(lib, kw, code):
    assert _call(**kw) == code


def test_empty_problems_are_no_ops(lib):
    assert _call(M=0) == 0
    assert _call(N=0, D=0) == 0


def test_beta_zero_needs_no_c(lib):
    # C is ignored when beta == 0: NULL, misaligned or overlapping C are all
    # fine; the call then proceeds to the device and fails on a CPU-only box.
    for c in (0, C_ + 4, D_):
        rc = _call(C=c, beta=0.0)
        assert rc in (0, -7, -5), rc


def test_k0_needs_no_operands(lib):
    rc = _call(K=0, A=0, B=0, lda=0, ldb=0)
    assert rc in (0, -7, -5), rc


@pytest.mark.parametrize("num_m,num_n,group", [(1, 1, 8), (32, 32, 8), (7, 5, 3), (13, 1, 16),
                                               (1, 9, 4), (33, 17, 8), (128, 1, 8)])
def test_tile_order_covers_every_tile_once(lib, num_m, num_n, group):
    seen = set()
    for t in range(num_m * num_n):
        m, n = binding.gemm_tile_coords(t, num_m, num_n, group)
        assert 0 <= m < num_m and 0 <= n < num_n
        seen.add((m, n))
    assert len(seen) == num_m * num_n


def test_tile_order_groups_rows(lib):
    # within a full group the order runs down group_m tile rows, then moves right
    coords = [binding.gemm_tile_coords(t, 32, 32, 8) for t in range(16)]
    assert coords[:8] == [(m, 0) for m in range(8)]
    assert coords[8:16] == [(m, 1) for m in range(8)]


def test_tile_coords_rejects_out_of_range(lib):
    with pytest.raises(binding.GemmError):
        binding.gemm_tile_coords(16, 4, 4, 2)


@pytest.mark.parametrize("M,N,K", [(8192, 8192, 8192), (16, 8, 16), (1000, 1000, 1000),
                                   (32768, 256, 4096), (512, 512, 512)])
def test_plan(lib, M, N, K):
    sms = 148
    p = binding.gemm_plan(M, N, K, sms)
    assert p["tile_m"] * ((M + p["tile_m"] - 1) // p["tile_m"]) >= M
    assert p["num_tiles"] == ((M + p["tile_m"] - 1) // p["tile_m"]) * ((N + p["tile_n"] - 1) // p["tile_n"])
    assert p["grid"] <= sms
    if p["cta_pair"]:
        assert p["grid"] % 2 == 0 and p["tile_m"] == 256
        assert p["grid"] == 2 * min(p["num_tiles"], sms // 2)
    else:
        assert p["grid"] == min(p["num_tiles"], sms)
    assert p["smem_bytes"] <= 232448
