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
            "gemm_plan", "gemm_plan_layout"} <= _declared_functions()


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    names = {0: "GEMM_OK", -1: "GEMM_ERR_INVALID_ARG", -2: "GEMM_ERR_UNSUPPORTED_DTYPE",
             -3: "GEMM_ERR_MISALIGNED", -4: "GEMM_ERR_ALIAS", -5: "GEMM_ERR_ARCH",
             -6: "GEMM_ERR_LAUNCH", -7: "GEMM_ERR_CUDA", -8: "GEMM_ERR_DEVICE_TIMEOUT",
             -9: "GEMM_ERR_TOO_LARGE", -10: "GEMM_ERR_UNSUPPORTED_LAYOUT"}
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
    (dict(in_dtype=5), -2),
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
    (dict(A=A_ + 1), -3),                   # not aligned to the element size
    (dict(B=B_ + 3), -3),
    (dict(D=D_ + 2), -3),                   # f32 D
    (dict(C=C_ + 2), -3),
    (dict(out_dtype=0, D=D_ + 1), -3),      # f16 D
    (dict(out_dtype=1, C=C_ + 1), -3),
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


@pytest.mark.parametrize("kw", [dict(A=A_ + 2), dict(D=D_ + 4), dict(C=C_ + 8), dict(K=60, lda=60),
                                dict(N=62, ldd=62, ldc=64, ldb=64), dict(out_dtype=0, N=60, ldd=60, ldc=64),
                                dict(out_dtype=1, D=D_ + 2, C=D_ + 2)])
def test_element_aligned_layouts_pass_validation(lib, kw):
    # Layouts TMA cannot describe (addresses or row strides that are not
    # 16-byte multiples) are accepted and go to the mma.sync kernel: the
    # call proceeds to the device and fails on a CPU-only box.
    rc = _call(**kw)
    assert rc in (0, -7, -5), rc


@pytest.mark.parametrize("kw", [dict(in_dtype=3, A=A_ + 1, lda=65), dict(in_dtype=4, transB=0, ldb=64),
                                dict(in_dtype=3, transA=1, B=B_ + 7)])
def test_fp8_layouts_pass_validation(lib, kw):
    # 8-bit operands need only byte alignment: gemm() repacks what the
    # tcgen05 kernel cannot read in place, so these reach the device.
    rc = _call(**kw)
    assert rc in (0, -7, -5), rc


def _call_noalloc(**kw):
    a = dict(OK_ARGS)
    a.update(kw)
    return binding.gemm_noalloc(a["D"], a["A"], a["B"], a["C"], a["M"], a["N"], a["K"], a["lda"], a["ldb"],
                                a["ldc"], a["ldd"], a["transA"], a["transB"], a["alpha"], a["beta"],
                                a["in_dtype"], a["out_dtype"], 0)


@pytest.mark.parametrize("kw", [dict(in_dtype=3, transB=0), dict(in_dtype=4, transA=1, transB=1),
                                dict(in_dtype=3, transB=1, A=A_ + 8), dict(in_dtype=4, transB=1, lda=72)])
def test_noalloc_fp8_needs_k_major_aligned_operands(lib, kw):
    """Without workspace nothing can be repacked: rejected on the host."""
    assert _call_noalloc(**kw) == -10


def _call_host(**kw):
    a = dict(OK_ARGS)
    a.update(kw)
    return binding.gemm_host(a["D"], a["A"], a["B"], a["C"], a["M"], a["N"], a["K"], a["lda"], a["ldb"],
                             a["ldc"], a["ldd"], a["transA"], a["transB"], a["alpha"], a["beta"],
                             a["in_dtype"], a["out_dtype"], 0)


@pytest.mark.parametrize("kw,code", [(dict(in_dtype=2), -2), (dict(out_dtype=3), -2), (dict(M=-1), -1),
                                     (dict(ldd=63), -1), (dict(C=0), -1), (dict(lda=63), -1),
                                     (dict(A=A_ + 1), -3), (dict(D=A_), -4), (dict(C=D_ + 4), -4),
                                     (dict(C=D_, ldc=72), -4), (dict(transB=3), -1)])
def test_host_entry_rejects_before_any_copy(lib, kw, code):
    assert _call_host(**kw) == code


def test_host_entry_empty_is_a_no_op(lib):
    assert _call_host(M=0) == 0 and _call_host(N=0, D=0) == 0


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
    units = sms // 2 if p["cta_pair"] else sms
    workers = p["grid"] // 2 if p["cta_pair"] else p["grid"]
    if p["cta_pair"]:
        assert p["grid"] % 2 == 0 and p["tile_m"] == 256
    if p["sk_tiles"] == 0:
        assert workers == min(p["num_tiles"], units)
    else:
        assert workers <= units and p["workspace_bytes"] > 0
    assert p["smem_bytes"] <= 232448


SCHEDULES = [
    # (num_tiles, iters, workers, sk_tiles)
    (1024, 64, 76, 36),      # 8192^3 on 76 clusters: 13 whole rounds + 36 split tiles
    (256, 32, 76, 28),       # 4096^3
    (128, 32, 76, 52),       # 32768 x 256 x 4096
    (16, 8, 32, 16),         # 1000^3: every tile split, 2 contributors each
    (16, 8, 76, 16),         # more workers than stages per tile: empty ranges
    (4, 4, 8, 4),
    (7, 3, 5, 2),
    (10, 1, 4, 10),
    (300, 17, 76, 0),        # data-parallel only
    (1, 1, 1, 1),
]


@pytest.mark.parametrize("num_tiles,iters,workers,sk_tiles", SCHEDULES)
def test_schedule_covers_every_stage_once(lib, num_tiles, iters, workers, sk_tiles):
    """Every (tile, stage) is done by exactly one worker; a split tile's
    contributors are numbered 0..nc-1 in K order with one agreed nc."""
    seen = {}
    per_worker = []
    contrib = {}
    for w in range(workers):
        units = binding.gemm_schedule_units(num_tiles, iters, workers, sk_tiles, w)
        total = 0
        for (tile, kb, ke, sk, ci, nc) in units:
            assert 0 <= tile < num_tiles and 0 <= kb < ke <= iters
            assert (sk >= 0) == (tile >= num_tiles - sk_tiles)
            if sk >= 0:
                assert tile == num_tiles - sk_tiles + sk
            if nc == 1:
                assert (kb, ke, ci) == (0, iters, 0)
            for k in range(kb, ke):
                assert (tile, k) not in seen
                seen[(tile, k)] = w
            contrib.setdefault(tile, []).append((kb, ci, nc, w))
            total += ke - kb
        per_worker.append(total)
    assert len(seen) == num_tiles * iters
    for tile, lst in contrib.items():
        lst.sort()
        ncs = {c[2] for c in lst}
        assert ncs == {len(lst)}, (tile, lst)
        assert [c[1] for c in lst] == list(range(len(lst)))          # K order = contributor order
        assert [c[3] for c in lst] == sorted(c[3] for c in lst)      # consecutive workers
    if sk_tiles:
        # stream-K balances the work: every worker within one tile's stages of the mean
        assert max(per_worker) - min(per_worker) <= iters + 1


def test_plan_streamk_choices(lib):
    p = binding.gemm_plan(8192, 8192, 8192, 152)
    assert p["sk_tiles"] == 1024 % 76 and p["grid"] == 152 and p["workspace_bytes"] > 0
    p = binding.gemm_plan(8192, 8192, 256, 152)          # 2 stages per tile: too short to split
    assert p["sk_tiles"] == 0 and p["workspace_bytes"] == 0
    p = binding.gemm_plan(1000, 1000, 1000, 152)         # 16 wide tiles: narrow ones instead, whole
    assert p["sk_tiles"] == 0 and p["tile_n"] == 64 and p["cta_pair"] == 0 and p["grid"] == 128
    p = binding.gemm_plan(4096, 4096, 4096, 152)         # ~12 stages per worker: not split
    assert p["sk_tiles"] == 0
    p = binding.gemm_plan(8192, 8192, 16384, 152)        # ~60 stages per worker
    assert p["sk_tiles"] == 1024 % 76


@pytest.mark.parametrize("M,N,K,tile_n", [(512, 512, 512, 64), (16, 8, 16, 64), (8192, 64, 4096, 64),
                                          (2048, 2048, 2048, 256), (32768, 256, 4096, 256),
                                          (1024, 1024, 4096, 64), (8192, 8192, 256, 256)])
def test_plan_tile_width(lib, M, N, K, tile_n):
    """Narrow 128 x 64 tiles exactly when the wide tiles would occupy at
    most a quarter of the SMs, or N fits one narrow tile."""
    p = binding.gemm_plan(M, N, K, 152)
    assert p["tile_n"] == tile_n
    if tile_n == 64:
        assert p["cta_pair"] == 0 and p["tile_m"] == 128 and p["epi_warps"] == 4


@pytest.mark.parametrize("M,N,K,transB,in_dtype,out_dtype,tile_n,num_tiles", [
    (4096, 4096, 4096, 1, binding.BF16, binding.F32, 224, 16 * 19),   # 3.4 waves of 256 -> 4.0 of 224
    (4096, 4096, 4096, 1, binding.E5M2, binding.F32, 224, 16 * 19),
    (4096, 4096, 4096, 0, binding.E4M3, binding.F32, 224, 16 * 19),   # 8-bit: planned K-major
    (4096, 4096, 4096, 0, binding.BF16, binding.F32, 256, 256),       # MN-major B: 64-wide boxes
    (4096, 4096, 4096, 1, binding.BF16, binding.BF16, 256, 256),      # 16-bit D: 64-column chunks
    (8192, 8192, 8192, 1, binding.F16, binding.F32, 256, 1024),       # stream-K fills the last wave
    (8192, 8192, 4096, 1, binding.F16, binding.F32, 256, 1024),       # 14 waves of 256 = 16 of 224
    (8192, 8192, 256, 1, binding.F16, binding.F32, 256, 1024),        # store-bound: 8 epilogue warps
    (32768, 256, 4096, 1, binding.F16, binding.F32, 256, 128),        # N = 256: one column of tiles
])
def test_plan_wave_fitted_tiles(lib, M, N, K, transB, in_dtype, out_dtype, tile_n, num_tiles):
    """224-wide CTA-pair tiles exactly where they fill the waves better
    (f32 D and K-major B only)."""
    p = binding.gemm_plan_layout(M, N, K, transB, in_dtype, out_dtype, 152)
    assert (p["tile_n"], p["num_tiles"]) == (tile_n, num_tiles)
    if tile_n == 224:
        assert p["cta_pair"] == 1 and p["epi_warps"] == 4 and p["sk_tiles"] == 0 and p["grid"] == 152


def test_plan_layout_defaults_and_rejections(lib):
    for M, N, K in [(512, 512, 512), (4096, 4096, 4096), (8192, 8192, 8192), (1000, 1000, 1000)]:
        assert binding.gemm_plan(M, N, K, 152) == binding.gemm_plan_layout(M, N, K, 0, binding.F16, binding.F32, 152)
    for args, code in [((64, 64, 64, 2, binding.F16, binding.F32, 152), -1),
                       ((64, 64, 64, 0, binding.F32, binding.F32, 152), -2),
                       ((64, 64, 64, 0, binding.F16, binding.E4M3, 152), -2),
                       ((0, 64, 64, 0, binding.F16, binding.F32, 152), -1)]:
        with pytest.raises(binding.GemmError) as e:
            binding.gemm_plan_layout(*args)
        assert e.value.status == code


def test_plan_wave_fitted_tiles_switch(lib, monkeypatch):
    monkeypatch.setenv("GEMM_FIT_TILES", "0")
    assert binding.gemm_plan_layout(4096, 4096, 4096, 1, binding.BF16, binding.F32, 152)["tile_n"] == 256
    monkeypatch.setenv("GEMM_FIT_TILES", "1")
    assert binding.gemm_plan_layout(8192, 8192, 8192, 1, binding.F16, binding.F32, 152)["tile_n"] == 224
    assert binding.gemm_plan_layout(8192, 8192, 8192, 0, binding.F16, binding.F32, 152)["tile_n"] == 256


def test_schedule_rejects_bad_arguments(lib):
    for args in [(0, 1, 1, 0, 0), (4, 0, 1, 0, 0), (4, 4, 2, 5, 0), (4, 4, 2, 1, 2)]:
        with pytest.raises(binding.GemmError):
            binding.gemm_schedule_units(*args)


# ---- gemm_mx: MX block-scaled 8-bit operands --------------------------------

SA_ = 0x50000000
SB_ = 0x60000000
MX_OK = dict(OK_ARGS, in_dtype=3, transB=1, SFA=SA_, SFB=SB_, ld_sfa=2, ld_sfb=2)


def _call_mx(**kw):
    a = dict(MX_OK)
    a.update(kw)
    return binding.gemm_mx(a["D"], a["A"], a["B"], a["C"], a["SFA"], a["SFB"], a["M"], a["N"], a["K"],
                           a["lda"], a["ldb"], a["ldc"], a["ldd"], a["ld_sfa"], a["ld_sfb"], a["transA"],
                           a["transB"], a["alpha"], a["beta"], a["in_dtype"], a["out_dtype"], 0)


MX_REJECTIONS = [
    (dict(in_dtype=0), -2),                 # block scaling is for 8-bit operands
    (dict(in_dtype=1), -2),
    (dict(in_dtype=2), -2),
    (dict(SFA=0), -1),
    (dict(SFB=0), -1),
    (dict(ld_sfa=1), -1),                   # K = 64: two scales per row
    (dict(ld_sfb=1), -1),
    (dict(K=65, lda=80, ldb=80), -1),       # K = 65: three scales per row
    (dict(D=SA_), -4),                      # D overlaps SFA
    (dict(SFB=D_ + 100), -4),               # SFB inside D
    (dict(lda=63), -1),                     # the operand rules of gemm() still apply
    (dict(C=D_ + 4096), -4),
]


@pytest.mark.parametrize("kw,code", MX_REJECTIONS, ids=[str(r[0]) for r in MX_REJECTIONS])
def test_mx_rejected_before_any_device_work(lib, kw, code):
    assert _call_mx(**kw) == code


def test_mx_valid_calls_reach_the_device(lib):
    # unaligned scales, padded scale rows, K = 0 with NULL scales, every
    # transpose form: all pass validation and fail only on a CPU-only box.
    for kw in (dict(), dict(SFA=SA_ + 3, SFB=SB_ + 1), dict(ld_sfa=7, ld_sfb=3), dict(K=0, SFA=0, SFB=0),
               dict(transA=1, transB=0), dict(in_dtype=4, out_dtype=1)):
        rc = _call_mx(**kw)
        assert rc in (0, -7, -5), (kw, rc)
    assert _call_mx(M=0) == 0 and _call_mx(N=0) == 0


def test_fp4_only_through_gemm_mx(lib):
    assert _call(in_dtype=5) == -2                        # gemm() has no 4-bit operands
    assert _call_mx(in_dtype=5, transA=1) == -10          # packed fp4 is K-major only
    assert _call_mx(in_dtype=5, transB=0) == -10
    assert _call_mx(in_dtype=5, K=63, lda=64, ldb=64) == -1   # whole bytes per row
    assert _call_mx(in_dtype=5, lda=65, ldb=66) == -1
    assert _call_mx(in_dtype=5, lda=62) == -1             # lda >= K
    assert _call_mx(in_dtype=5, D=A_ + 16) == -4          # D overlaps A's bytes ([64, 32] bytes from A_)
    assert _call_mx(in_dtype=5, D=A_ + 64 * 32) in (0, -7, -5)   # just past A's last byte: no overlap
    for kw in (dict(), dict(A=A_ + 3, lda=70), dict(K=2, lda=2, ldb=2)):
        rc = _call_mx(in_dtype=5, **kw)
        assert rc in (0, -7, -5), (kw, rc)


def test_plan_layout_invariants(lib):
    """Every plan, over a seeded spread of shapes, layouts and types: the tile
    count covers the output, the grid fits the GPU, 224-wide tiles appear only
    for f32 D with K-major B on CTA pairs, and a workspace exists exactly when
    tiles are split along K."""
    import numpy as np
    rng = np.random.default_rng(2024)
    sms = 152
    for _ in range(3000):
        M, N = (int(x) for x in np.exp(rng.uniform(0, np.log(40000), 2)).astype(int) + 1)
        K = int(np.exp(rng.uniform(0, np.log(70000)))) if rng.random() > 0.05 else 0
        tb = int(rng.integers(0, 2))
        it = int(rng.choice([binding.F16, binding.BF16, binding.E4M3, binding.E5M2]))
        ot = int(rng.choice([binding.F32, binding.F16, binding.BF16]))
        p = binding.gemm_plan_layout(M, N, K, tb, it, ot, sms)
        tm, tn = p["tile_m"], p["tile_n"]
        assert tn in (64, 224, 256) and tm in (128, 256), p
        assert p["num_tiles"] == -(-M // tm) * -(-N // tn), (M, N, K, p)
        assert 1 <= p["grid"] <= sms and (p["grid"] % 2 == 0 or not p["cta_pair"]), p
        if tn == 224:
            assert p["cta_pair"] and ot == binding.F32 and p["epi_warps"] == 4, (M, N, K, tb, it, ot, p)
            assert tb == 1 or it in (binding.E4M3, binding.E5M2), (M, N, K, tb, it, p)
        assert 0 <= p["sk_tiles"] <= p["num_tiles"]
        assert (p["workspace_bytes"] > 0) == (p["sk_tiles"] > 0), p
        assert p["stages"] >= 2 and p["smem_bytes"] <= 232448, p
