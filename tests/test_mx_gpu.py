"""GPU parity of MX block-scaled 8-bit operands (gemm_mx) against the CPU
oracle.

The TIRx gemm guide lists block scaling with separate A and B scale factors
(SFA / SFB) among the tcgen05 path's modes (section 七); the reading taken
is the OCP Microscaling one: one UE8M0 scale byte per 32 K elements of each
row of op(A) (SFA [M, ceil(K/32)]) and of each column of op(B) (SFB
[N, ceil(K/32)]).  The kernel is tcgen05.mma kind::mxf8f6f4 with the scales
copied into tensor memory, 256 x 192 tiles on a CTA pair or 128 x 192 on
one SM.

Integer operands in [-8, 8] with scales within 2^+-1 keep every fp32
partial sum exact, so those cases are compared bit for bit; wider scale
ranges and random operands are compared within the tolerance.
"""
import numpy as np
import pytest
import torch

import oracle.oracle as oracle
from dense_tensor_core_02_gb300 import binding
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

FP8 = ["e4m3", "e5m2"]


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    yield
    rc, info = H.poll()
    assert rc == 0, ("device status after the module", rc, info)


@pytest.fixture(params=["pair", "single"])
def variant(request):
    """256 x 192 tiles on a CTA pair (the default when M > 128) or 128 x 192
    tiles on one SM."""
    with H.env(GEMM_VARIANT=request.param, GEMM_PATH=None):
        yield request.param


def scales(rows, K, lo, hi, seed, pad=0):
    """UE8M0 bytes in [lo, hi], [rows, ceil(K/32) + pad]; the padding holds
    NaN scales (255), which must never be read."""
    kb = (K + 31) // 32
    g = torch.Generator().manual_seed(seed)
    s = torch.full((rows, kb + pad), 255, dtype=torch.uint8)
    s[:, :kb] = torch.randint(lo, hi + 1, (rows, kb), generator=g, dtype=torch.int32).to(torch.uint8)
    return s


def run_mx(A, B, C, SFA, SFB, M, N, K, *, transA=0, transB=1, alpha=1.0, beta=0.0, in_dtype="e4m3",
           out_dtype="f32", sf_offsets=(0, 0)):
    """Copy to cuda:0, call gemm_mx, return (D on the CPU, status).  The
    scale arrays may be placed at byte offsets (any alignment is legal)."""
    dev = torch.device("cuda", 0)
    Ad = A.to(dev) if A is not None else None
    Bd = B.to(dev) if B is not None else None
    Cd = C.to(dev) if C is not None else None
    sf = []
    for S, off in zip((SFA, SFB), sf_offsets):
        if S is None:
            sf.append((None, 0))
            continue
        buf = torch.full((S.numel() + off + 16,), 255, dtype=torch.uint8, device=dev)
        view = buf[off:off + S.numel()].view(S.shape)
        view.copy_(S.to(dev))
        sf.append((view, S.stride(0)))
    D = torch.full((M, N), float("nan"), dtype=H.TORCH[out_dtype], device=dev)
    epu = 2 if in_dtype == "e2m1" else 1   # packed fp4: leading dimensions count elements
    lda = Ad.stride(0) * epu if Ad is not None else 0
    ldb = Bd.stride(0) * epu if Bd is not None else 0
    ldc = Cd.stride(0) if Cd is not None else N
    rc = binding.gemm_mx(D, Ad, Bd, Cd, sf[0][0], sf[1][0], M, N, K, lda, ldb, ldc, D.stride(0), sf[0][1],
                         sf[1][1], transA, transB, alpha, beta, H.CODE[in_dtype], H.CODE[out_dtype], None)
    torch.cuda.synchronize()
    return D.cpu(), rc


def oracle_mx(A, B, C, SFA, SFB, M, N, K, *, transA=0, transB=1, alpha=1.0, beta=0.0, in_dtype="e4m3",
              out_dtype="f32"):
    return oracle.gemm(A, B, C, M, N, K, transA=transA, transB=transB, alpha=alpha, beta=beta,
                       in_dtype=H.CODE[in_dtype], c_dtype=H.CODE[out_dtype], threads=H.ORACLE_THREADS,
                       sfa=SFA.numpy(), sfb=SFB.numpy())


SHAPES = [(128, 192, 128), (16, 8, 32), (1, 1, 1), (257, 200, 160), (300, 400, 544), (640, 520, 1040),
          (129, 385, 48)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", FP8)
@pytest.mark.parametrize("beta", [0.0, 1.0])
def test_integers_exact(variant, shape, dtype, beta):
    M, N, K = shape
    seed = 5 * M + 3 * N + K + (dtype == "e5m2") + 2 * int(beta)
    A = H.int_matrix((M, K), -8, 8, dtype, seed)
    B = H.int_matrix((N, K), -8, 8, dtype, seed + 1)
    C = H.int_matrix((M, N), -100, 100, "f32", seed + 2) if beta else None
    SFA = scales(M, K, 126, 128, seed + 3, pad=2)
    SFB = scales(N, K, 126, 128, seed + 4, pad=1)
    kw = dict(beta=beta, in_dtype=dtype)
    D, rc = run_mx(A, B, C, SFA, SFB, M, N, K, **kw)
    assert rc == 0
    ref, _ = oracle_mx(A, B, C, SFA, SFB, M, N, K, **kw)
    H.assert_exact(D.numpy(), ref, "mx %s %s beta=%s" % (dtype, shape, beta))


@pytest.mark.parametrize("dtype", FP8)
def test_each_block_takes_its_own_scale(variant, dtype):
    """One distinct power of two per (row, block) and (column, block): a
    scale applied to the wrong block, row or column shows at once."""
    M, N, K = 256, 384, 256
    A = H.int_matrix((M, K), 1, 1, dtype, 0)
    B = H.int_matrix((N, K), 1, 1, dtype, 0)
    kb = K // 32
    # exponents within 2^-8 .. 2^7: every fp32 partial sum stays exact
    SFA = torch.tensor([[124 + (i + 3 * b) % 8 for b in range(kb)] for i in range(M)], dtype=torch.uint8)
    SFB = torch.tensor([[124 + (j * 5 + b) % 7 for b in range(kb)] for j in range(N)], dtype=torch.uint8)
    D, rc = run_mx(A, B, None, SFA, SFB, M, N, K, in_dtype=dtype)
    assert rc == 0
    ref, _ = oracle_mx(A, B, None, SFA, SFB, M, N, K, in_dtype=dtype)
    H.assert_exact(D.numpy(), ref, "per-block scales")


@pytest.mark.parametrize("dtype", FP8)
@pytest.mark.parametrize("out_dtype", ["f32", "f16", "bf16"])
def test_random_wide_scales(variant, dtype, out_dtype):
    M, N, K = 520, 392, 776
    seed = 41 + (dtype == "e5m2") + 2 * ["f32", "f16", "bf16"].index(out_dtype)
    A = H.normal_matrix((M, K), dtype, seed)
    B = H.normal_matrix((N, K), dtype, seed + 1)
    C = H.normal_matrix((M, N), out_dtype, seed + 2)
    SFA = scales(M, K, 117, 133, seed + 3)
    SFB = scales(N, K, 119, 131, seed + 4)
    kw = dict(alpha=0.375, beta=-1.25, in_dtype=dtype, out_dtype=out_dtype)
    D, rc = run_mx(A, B, C, SFA, SFB, M, N, K, **kw)
    assert rc == 0
    ref, bound = oracle_mx(A, B, C, SFA, SFB, M, N, K, **kw)
    H.assert_close(D.double().numpy(), ref, bound, out_dtype, "mx random %s -> %s" % (dtype, out_dtype))


@pytest.mark.parametrize("transA", [0, 1])
@pytest.mark.parametrize("transB", [0, 1])
@pytest.mark.parametrize("dtype", FP8)
def test_transpose_forms(transA, transB, dtype):
    """MN-major operands are transposed to K-major in workspace; the scales
    follow op(A)'s rows and op(B)'s columns whatever the storage."""
    M, N, K = 392, 264, 328
    seed = 17 + 4 * transA + 2 * transB + (dtype == "e5m2")
    A = H.int_matrix((K, M) if transA else (M, K), -8, 8, dtype, seed)
    B = H.int_matrix((N, K) if transB else (K, N), -8, 8, dtype, seed + 1)
    C = H.int_matrix((M, N), -50, 50, "f32", seed + 2)
    SFA = scales(M, K, 126, 128, seed + 3)
    SFB = scales(N, K, 126, 128, seed + 4)
    kw = dict(transA=transA, transB=transB, beta=1.0, in_dtype=dtype)
    D, rc = run_mx(A, B, C, SFA, SFB, M, N, K, **kw)
    assert rc == 0
    ref, _ = oracle_mx(A, B, C, SFA, SFB, M, N, K, **kw)
    H.assert_exact(D.numpy(), ref, "mx transpose %d%d %s" % (transA, transB, dtype))


def test_unaligned_scales_and_operands():
    """Scale arrays at odd byte offsets with padded rows; operands and D off
    the 16-byte grid (repacked)."""
    M, N, K = 200, 136, 101
    A = H.int_matrix((M, K), -8, 8, "e4m3", 81)
    B = H.int_matrix((N, K), -8, 8, "e4m3", 82)
    C = H.int_matrix((M, N), -50, 50, "f32", 83)
    SFA = scales(M, K, 126, 128, 84, pad=5)
    SFB = scales(N, K, 126, 128, 85, pad=3)
    D, rc = run_mx(A, B, C, SFA, SFB, M, N, K, beta=1.0, sf_offsets=(3, 1))
    assert rc == 0
    ref, _ = oracle_mx(A, B, C, SFA, SFB, M, N, K, beta=1.0)
    H.assert_exact(D.numpy(), ref, "mx unaligned scales")

    def fn(D_, A_, B_, C_, M_, N_, K_, lda, ldb, ldc, ldd, tA, tB, al, be, idt, odt, st):
        sa, sb = SFA.cuda(), SFB.cuda()
        return binding.gemm_mx(D_, A_, B_, C_, sa, sb, M_, N_, K_, lda, ldb, ldc, ldd, sa.stride(0), sb.stride(0),
                               tA, tB, al, be, idt, odt, st)

    D2, Dbuf, rc = H.run_layout(A, B, C, M, N, K, offs=(1, 3, 1, 1), lds=(K + 2, K + 5, N + 1, N + 3), transB=1,
                                beta=1.0, in_dtype="e4m3", fn=fn)
    assert rc == 0
    H.assert_exact(D2.numpy(), ref, "mx misaligned operands")
    H.check_canaries(Dbuf, M, N, 1, N + 3)


@pytest.mark.parametrize("dtype", FP8)
def test_streamk_split(variant, dtype):
    M, N, K = 1024, 768, 2080
    A = H.int_matrix((M, K), -4, 4, dtype, 91)
    B = H.int_matrix((N, K), -4, 4, dtype, 92)
    SFA = scales(M, K, 126, 128, 93)
    SFB = scales(N, K, 126, 128, 94)
    with H.env(GEMM_SK_MIN_ITERS="1"):
        D, rc = run_mx(A, B, None, SFA, SFB, M, N, K, in_dtype=dtype)
    assert rc == 0
    rows, cols = H.sample_positions(M, N, per_block=8, seed=19)
    ref, _ = oracle.gemm_entries(A, B, None, M, N, K, rows, cols, transB=1, in_dtype=H.CODE[dtype],
                                 threads=H.ORACLE_THREADS, sfa=SFA.numpy(), sfb=SFB.numpy())
    H.assert_exact(D.numpy()[rows, cols], ref, "mx stream-K")


def test_nan_scale_poisons_its_block_only():
    M, N, K = 130, 200, 96
    A = H.int_matrix((M, K), -8, 8, "e4m3", 101)
    B = H.int_matrix((N, K), -8, 8, "e4m3", 102)
    SFA = scales(M, K, 126, 128, 103)
    SFB = scales(N, K, 126, 128, 104)
    SFA[7, 1] = 255
    SFB[150, 2] = 255
    D, rc = run_mx(A, B, None, SFA, SFB, M, N, K)
    assert rc == 0
    ref, _ = oracle_mx(A, B, None, SFA, SFB, M, N, K)
    got = D.numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref)), "NaN pattern differs"
    fin = ~np.isnan(ref)
    H.assert_exact(got[fin], ref[fin], "mx NaN scales, finite part")


def test_k_zero_and_tiny():
    M, N = 70, 88
    C = H.int_matrix((M, N), -50, 50, "f32", 111)
    D, rc = run_mx(None, None, C, None, None, M, N, 0, alpha=3.0, beta=2.0)
    assert rc == 0
    H.assert_exact(D.numpy(), 2.0 * C.double().numpy(), "mx K = 0")


def test_unit_scales_equal_unscaled_fp8():
    """Scale 1 everywhere: the block-scaled kernel and the plain 8-bit
    kernel must both equal the oracle's unscaled product."""
    M, N, K = 512, 576, 1024
    A = H.normal_matrix((M, K), "e4m3", 121)
    B = H.normal_matrix((N, K), "e4m3", 122)
    ones_a = torch.full((M, K // 32), 127, dtype=torch.uint8)
    ones_b = torch.full((N, K // 32), 127, dtype=torch.uint8)
    D, rc = run_mx(A, B, None, ones_a, ones_b, M, N, K)
    assert rc == 0
    ref, bound = H.oracle_full(A, B, None, M, N, K, transB=1, in_dtype="e4m3")
    H.assert_close(D.double().numpy(), ref, bound, "f32", "mx unit scales")
    D8, rc = H.run_gemm(A, B, None, M, N, K, transB=1, in_dtype="e4m3")
    assert rc == 0
    H.assert_close(D8.double().numpy(), ref, bound, "f32", "fp8 unscaled")


from dense_tensor_core_02_gb300 import inputs  # noqa: E402

MX_CASES = [c for c in inputs.CASES if c.mx]


@pytest.mark.parametrize("case", MX_CASES, ids=lambda c: c.name)
def test_workload_sampled(case):
    """The block-scaled workloads at full size, in the benchmark's launch
    configuration, on sampled outputs that touch every 128 x 128 block."""
    A, B, C = inputs.make_inputs(case)
    SFA, SFB = inputs.make_scales(case)
    kw = dict(transA=case.transA, transB=case.transB, alpha=case.alpha, beta=case.beta,
              in_dtype=case.in_dtype, out_dtype=case.out_dtype)
    D, rc = run_mx(A, B, C, SFA, SFB, case.M, case.N, case.K, **kw)
    assert rc == 0
    assert not torch.isnan(D).any(), "unwritten (NaN-filled) output elements"
    rows, cols = H.sample_positions(case.M, case.N, per_block=4, seed=case.seed)
    ref, bound = oracle.gemm_entries(A, B, C, case.M, case.N, case.K, rows, cols, threads=H.ORACLE_THREADS,
                                     sfa=SFA.numpy(), sfb=SFB.numpy(), transA=case.transA, transB=case.transB,
                                     alpha=case.alpha, beta=case.beta, in_dtype=H.CODE[case.in_dtype],
                                     c_dtype=H.CODE[case.out_dtype])
    H.assert_close(D.double().numpy()[rows, cols], ref, bound, case.out_dtype, case.name)


# ---- packed E2M1 (fp4) operands ----------------------------------------------


def fp4_matrix(rows, K, seed, lo_code=0, hi_code=15, pad=0):
    """Random E2M1 codes in [lo_code, hi_code], packed two per byte (even
    columns low): uint8 [rows, (K + pad) / 2], the padding all-ones codes."""
    g = torch.Generator().manual_seed(seed)
    codes = torch.full((rows, K + pad), 0xF, dtype=torch.int32)
    codes[:, :K] = torch.randint(lo_code, hi_code + 1, (rows, K), generator=g, dtype=torch.int32)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).to(torch.uint8)


FP4_SHAPES = [(128, 192, 256), (16, 8, 64), (1, 1, 2), (257, 200, 160), (300, 400, 544), (640, 520, 1040),
              (129, 385, 48)]


@pytest.mark.parametrize("shape", FP4_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("beta", [0.0, 1.0])
def test_fp4_exact(variant, shape, beta):
    """E2M1 products are multiples of 1/4 and the scales stay within 2^+-1,
    so every fp32 partial sum is exact: bit for bit."""
    M, N, K = shape
    seed = 7 * M + 5 * N + K + 2 * int(beta)
    A = fp4_matrix(M, K, seed)
    B = fp4_matrix(N, K, seed + 1)
    C = H.int_matrix((M, N), -100, 100, "f32", seed + 2) if beta else None
    SFA = scales(M, K, 126, 128, seed + 3, pad=1)
    SFB = scales(N, K, 126, 128, seed + 4, pad=2)
    kw = dict(beta=beta, in_dtype="e2m1")
    D, rc = run_mx(A, B, C, SFA, SFB, M, N, K, **kw)
    assert rc == 0
    ref, _ = oracle_mx(A, B, C, SFA, SFB, M, N, K, **kw)
    H.assert_exact(D.numpy(), ref, "fp4 %s beta=%s" % (shape, beta))


def test_fp4_each_block_takes_its_own_scale(variant):
    M, N, K = 256, 384, 512
    A = fp4_matrix(M, K, 131, 2, 2)      # all 1.0
    B = fp4_matrix(N, K, 132, 2, 2)
    kb = K // 32
    SFA = torch.tensor([[124 + (i + 3 * b) % 8 for b in range(kb)] for i in range(M)], dtype=torch.uint8)
    SFB = torch.tensor([[124 + (j * 5 + b) % 7 for b in range(kb)] for j in range(N)], dtype=torch.uint8)
    D, rc = run_mx(A, B, None, SFA, SFB, M, N, K, in_dtype="e2m1")
    assert rc == 0
    ref, _ = oracle_mx(A, B, None, SFA, SFB, M, N, K, in_dtype="e2m1")
    H.assert_exact(D.numpy(), ref, "fp4 per-block scales")


@pytest.mark.parametrize("out_dtype", ["f32", "f16", "bf16"])
def test_fp4_random_wide_scales(variant, out_dtype):
    M, N, K = 520, 392, 776
    seed = 141 + ["f32", "f16", "bf16"].index(out_dtype)
    A = fp4_matrix(M, K, seed)
    B = fp4_matrix(N, K, seed + 1)
    C = H.normal_matrix((M, N), out_dtype, seed + 2)
    # (for f16 D the scales stay small enough that |D| < 65504: an overflow
    # would round to infinity, correctly, and say nothing about the product)
    hi = 129 if out_dtype == "f16" else 135
    SFA = scales(M, K, 115, hi, seed + 3)
    SFB = scales(N, K, 118, hi - 4, seed + 4)
    kw = dict(alpha=-0.625, beta=0.75, in_dtype="e2m1", out_dtype=out_dtype)
    D, rc = run_mx(A, B, C, SFA, SFB, M, N, K, **kw)
    assert rc == 0
    ref, bound = oracle_mx(A, B, C, SFA, SFB, M, N, K, **kw)
    H.assert_close(D.double().numpy(), ref, bound, out_dtype, "fp4 random -> %s" % out_dtype)


def test_fp4_padded_and_offset_rows():
    """Leading dimensions off the 16-byte grid and an odd byte offset: the
    rows are copied into aligned workspace first; the padding (all-ones
    codes, -6.0) must never be read."""
    M, N, K = 200, 136, 102
    A = fp4_matrix(M, K, 151, pad=6)     # lda = 108 elements = 54 bytes
    B = fp4_matrix(N, K, 152, pad=2)     # ldb = 104 = 52 bytes
    SFA = scales(M, K, 126, 128, 153)
    SFB = scales(N, K, 126, 128, 154)
    D, rc = run_mx(A, B, None, SFA, SFB, M, N, K, in_dtype="e2m1")
    assert rc == 0
    ref, _ = oracle.gemm(A, B, None, M, N, K, transB=1, in_dtype=H.CODE["e2m1"], lda=K + 6, ldb=K + 2,
                         threads=H.ORACLE_THREADS, sfa=SFA.numpy(), sfb=SFB.numpy())
    H.assert_exact(D.numpy(), ref, "fp4 padded rows")
    dev = torch.device("cuda", 0)
    buf = torch.zeros(A.numel() + 1 + 64, dtype=torch.uint8, device=dev)
    Av = buf[1:1 + A.numel()].view(A.shape)   # odd byte offset
    Av.copy_(A.to(dev))
    Bd, sa, sb = B.to(dev), SFA.to(dev), SFB.to(dev)
    Dd = torch.full((M, N), float("nan"), device=dev)
    rc = binding.gemm_mx(Dd, Av, Bd, None, sa, sb, M, N, K, K + 6, K + 2, N, N, sa.stride(0), sb.stride(0), 0, 1,
                         1.0, 0.0, H.CODE["e2m1"], H.CODE["f32"], None)
    torch.cuda.synchronize()
    assert rc == 0
    H.assert_exact(Dd.cpu().numpy(), ref, "fp4 odd byte offset")


def test_fp4_streamk_split(variant):
    M, N, K = 1024, 768, 4160
    A = fp4_matrix(M, K, 161)
    B = fp4_matrix(N, K, 162)
    SFA = scales(M, K, 126, 128, 163)
    SFB = scales(N, K, 126, 128, 164)
    with H.env(GEMM_SK_MIN_ITERS="1"):
        D, rc = run_mx(A, B, None, SFA, SFB, M, N, K, in_dtype="e2m1")
    assert rc == 0
    rows, cols = H.sample_positions(M, N, per_block=8, seed=29)
    ref, _ = oracle.gemm_entries(A, B, None, M, N, K, rows, cols, transB=1, in_dtype=H.CODE["e2m1"],
                                 threads=H.ORACLE_THREADS, sfa=SFA.numpy(), sfb=SFB.numpy())
    H.assert_exact(D.numpy()[rows, cols], ref, "fp4 stream-K")


# ---- seeded sweep over gemm_mx's argument space ------------------------------


def _mx_case(seed):
    rng = np.random.default_rng(seed)
    pick = lambda xs: xs[int(rng.integers(len(xs)))]
    dtype = pick(["e4m3", "e5m2", "e2m1"])
    dims = [1, 7, 16, 33, 128, 129, 192, 255, 300, 513]
    kdims = [0, 2, 16, 32, 64, 100, 128, 256, 300, 640] + ([] if dtype == "e2m1" else [1, 7, 33, 129])
    c = dict(M=pick(dims), N=pick(dims), K=pick(kdims), dtype=dtype, out=pick(["f32", "f16", "bf16"]),
             transA=0 if dtype == "e2m1" else int(rng.integers(2)),
             transB=1 if dtype == "e2m1" else int(rng.integers(2)),
             beta=pick([0.0, 1.0, -0.5]), alpha=pick([1.0, 2.0, -0.75]),
             pad=pick([0, 0, 2, 6]), off=pick([0, 0, 1, 3]), sf_pad=pick([0, 1, 5]), sf_off=pick([0, 1]),
             variant=pick([None, None, "single"]))
    c["exact"] = c["out"] == "f32" and c["alpha"] in (1.0, 2.0) and c["beta"] in (0.0, 1.0)
    return c


def _place(host_u8, off, dev):
    """A uint8 [rows, cols] matrix at byte offset `off` of a device buffer."""
    buf = torch.full((host_u8.numel() + off + 64,), 0xFF, dtype=torch.uint8, device=dev)
    v = buf[off:off + host_u8.numel()].view(host_u8.shape)
    v.copy_(host_u8.to(dev))
    return v


@pytest.mark.parametrize("seed", range(60))
def test_mx_fuzz(seed):
    c = _mx_case(3000 + seed)
    M, N, K, dt = c["M"], c["N"], c["K"], c["dtype"]
    dev = torch.device("cuda", 0)
    epu = 2 if dt == "e2m1" else 1
    pad = c["pad"] if dt != "e2m1" else 2 * (c["pad"] // 2)
    # operands as stored (padded rows), then viewed as bytes
    ra, ca = (K, M) if c["transA"] else (M, K)
    rb, cb = (N, K) if c["transB"] else (K, N)
    if dt == "e2m1":
        A = fp4_matrix(ra, ca, seed, pad=pad)
        B = fp4_matrix(rb, cb, seed + 1, pad=pad)
    else:
        A = H.int_matrix((ra, ca + pad), -8, 8, dt, seed).view(torch.uint8)
        B = H.int_matrix((rb, cb + pad), -8, 8, dt, seed + 1).view(torch.uint8)
    lda, ldb = (ca + pad), (cb + pad)
    C = H.int_matrix((M, N), -50, 50, c["out"], seed + 2) if c["beta"] else None
    # (f16 D: scales small enough that |D| stays below the f16 maximum)
    lo, hi = (126, 128) if c["exact"] else (118, 126) if c["out"] == "f16" else (118, 134)
    SFA = scales(M, K, lo, hi, seed + 3, pad=c["sf_pad"])
    SFB = scales(N, K, lo, hi, seed + 4, pad=c["sf_pad"])
    Av, Bv = _place(A, c["off"], dev), _place(B, c["off"] * 2, dev)
    sav, sbv = _place(SFA, c["sf_off"], dev), _place(SFB, c["sf_off"], dev)
    Cd = C.to(dev) if C is not None else None
    D = torch.full((M, N), float("nan"), dtype=H.TORCH[c["out"]], device=dev)
    with H.env(GEMM_VARIANT=c["variant"]):
        rc = binding.gemm_mx(D, Av if K else None, Bv if K else None, Cd, sav if K else None, sbv if K else None,
                             M, N, K, lda, ldb, N, N, SFA.shape[1], SFB.shape[1], c["transA"], c["transB"],
                             c["alpha"], c["beta"], H.CODE[dt], H.CODE[c["out"]], None)
    torch.cuda.synchronize()
    assert rc == 0, (c, binding.gemm_status_string(rc))
    Ao = A if dt == "e2m1" else A.view(H.TORCH[dt])
    Bo = B if dt == "e2m1" else B.view(H.TORCH[dt])
    ref, bound = oracle.gemm(Ao, Bo, C, M, N, K, transA=c["transA"], transB=c["transB"], alpha=c["alpha"],
                             beta=c["beta"], in_dtype=H.CODE[dt], c_dtype=H.CODE[c["out"]], lda=lda, ldb=ldb,
                             threads=H.ORACLE_THREADS, sfa=SFA.numpy(), sfb=SFB.numpy())
    got = D.cpu().double().numpy()
    if c["exact"]:
        H.assert_exact(got, ref, "mx fuzz %s" % c)
    else:
        H.assert_close(got, ref, bound, c["out"], "mx fuzz %s" % c)


@pytest.mark.parametrize("dtype", ["e4m3", "e2m1"])
def test_bounded_wait_reports_and_recovers(variant, dtype):
    """Failure detection without a fault: the test hook leaves the first
    stage of the first tile unfilled, so the MMA issuer's and the scale
    warp's waits on it run out (bounded), the kernel unwinds and records
    GEMM_ERR_DEVICE_TIMEOUT; the next call on the same context is correct."""
    M, N, K = 384, 448, 512
    if dtype == "e2m1":
        A, B = fp4_matrix(M, K, 171), fp4_matrix(N, K, 172)
    else:
        A, B = H.int_matrix((M, K), -8, 8, dtype, 171), H.int_matrix((N, K), -8, 8, dtype, 172)
    SFA, SFB = scales(M, K, 126, 128, 173), scales(N, K, 126, 128, 174)
    with H.env(GEMM_TEST_SKIP_FIRST_STAGE="1", GEMM_WAIT_TIMEOUT_NS="300000000"):
        _, rc = run_mx(A, B, None, SFA, SFB, M, N, K, in_dtype=dtype)
    assert rc == 0
    status, info = H.poll()
    assert status == binding.GEMM_ERR_DEVICE_TIMEOUT, (status, info)
    assert H.poll()[0] == 0
    D, rc = run_mx(A, B, None, SFA, SFB, M, N, K, in_dtype=dtype)
    assert rc == 0 and H.poll()[0] == 0
    ref, _ = oracle_mx(A, B, None, SFA, SFB, M, N, K, in_dtype=dtype)
    H.assert_exact(D.numpy(), ref, "after recovery (%s)" % dtype)


def test_in_place_and_alpha_zero():
    """D = C in place (beta = 1), and alpha = 0 (D = beta * C exactly)."""
    dev = torch.device("cuda", 0)
    M, N, K = 300, 280, 192
    A = H.int_matrix((M, K), -8, 8, "e4m3", 181).to(dev)
    B = H.int_matrix((N, K), -8, 8, "e4m3", 182).to(dev)
    SFA, SFB = scales(M, K, 126, 128, 183), scales(N, K, 126, 128, 184)
    sa, sb = SFA.to(dev), SFB.to(dev)
    C = H.int_matrix((M, N), -50, 50, "f32", 185)
    D = C.to(dev).clone()
    rc = binding.gemm_mx(D, A, B, D, sa, sb, M, N, K, K, K, N, N, sa.stride(0), sb.stride(0), 0, 1, 1.0, 1.0,
                         H.CODE["e4m3"], H.CODE["f32"], None)
    torch.cuda.synchronize()
    assert rc == 0
    ref, _ = oracle_mx(A.cpu(), B.cpu(), C, SFA, SFB, M, N, K, beta=1.0)
    H.assert_exact(D.cpu().numpy(), ref, "in place")
    D2 = torch.full((M, N), float("nan"), device=dev)
    rc = binding.gemm_mx(D2, A, B, C.to(dev), sa, sb, M, N, K, K, K, N, N, sa.stride(0), sb.stride(0), 0, 1, 0.0,
                         -2.0, H.CODE["e4m3"], H.CODE["f32"], None)
    torch.cuda.synchronize()
    assert rc == 0
    H.assert_exact(D2.cpu().numpy(), -2.0 * C.double().numpy(), "alpha = 0")


@pytest.mark.parametrize("e", [0, 1, 253])
def test_extreme_scale_exponents(e):
    """Every scale 2^(e - 127) with tiny operands: the smallest scales (2^-127,
    2^-126: the products lie far below the fp32 normal range) and a large one
    (2^126 x 2^-126 on B keeps the products representable)."""
    M, N, K = 128, 192, 128
    A = H.int_matrix((M, K), -2, 2, "e4m3", 191)
    B = H.int_matrix((N, K), -2, 2, "e4m3", 192)
    SFA = torch.full((M, K // 32), e, dtype=torch.uint8)
    SFB = torch.full((N, K // 32), 254 - e if e == 253 else 127, dtype=torch.uint8)
    D, rc = run_mx(A, B, None, SFA, SFB, M, N, K)
    assert rc == 0
    ref, bound = oracle_mx(A, B, None, SFA, SFB, M, N, K)
    H.assert_close(D.double().numpy(), ref, bound, "f32", "scale exponent %d" % e)
