"""Pins for the CPU oracle: checks against facts fixed outside the oracle.

Each ``pin_*`` function takes a loaded ``Oracle`` and raises
``AssertionError`` when the oracle disagrees with something the pages or
plain mathematics fix:

* exact decoding of every fp16 / bf16 bit pattern (numpy's IEEE binary16,
  and bfloat16 defined as the upper half of binary32) and of every E4M3 /
  E5M2 pattern (torch's float8_e4m3fn / float8_e5m2 conversions, and the
  formats' fixed points: largest finite values 448 and 57344, smallest
  subnormals 2^-9 and 2^-16, E4M3's single NaN pattern per sign, E5M2's
  infinities);
* brute force in Python integers on integer-valued inputs, with padded
  leading dimensions and all four transpose forms (exact);
* numpy's float64 matmul on random inputs (a library routine);
* identity and permutation operands, beta = 0 vs beta = 1 semantics (TIRx
  "gemm" page, "What it accepts" table, alpha / beta row: 0 -> D = A@B,
  1 -> D = A@B + C), transpose equivalence (the flags only name the
  logical orientation), linearity in alpha and beta, a closed-form sum and
  the error bound's own identities;
* MX block scaling (the OCP Microscaling reading of the TIRx gemm guide's
  "block scaling (SFA / SFB)", section 七): the UE8M0 decoder against
  torch's float8_e8m0fnu conversion, exact rational brute force with scale
  blocks of 32 along K (ragged last block, padded scale rows), unit scales
  reducing to the unscaled product, exact doubling of a row / column when
  its scales go up by one, invariance when a block's scale moves from A to
  B, a closed form at a block boundary and NaN scales;
* packed E2M1 (fp4): the format's 16 values (OCP: magnitudes 0, 0.5, 1, 1.5,
  2, 3, 4, 6), the nibble order of the packing (even elements low), and
  exact rational brute force of block-scaled fp4 products.

``tests/test_oracle_mutants.py`` runs the same pins against deliberately
broken builds of the oracle and requires each break to be caught.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle.oracle import BF16, E2M1, E4M3, E5M2, F16, F32

F16_NAN = 0x7E00
BF16_NAN = 0x7FC0
_TD = {F16: torch.float16, BF16: torch.bfloat16, E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}


def _same(a, b):
    """Bitwise-equal doubles, NaN equal to NaN."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    both_nan = np.isnan(a) & np.isnan(b)
    eq = (a == b) & (np.signbit(a) == np.signbit(b))
    return bool(np.all(both_nan | eq))


def _int_tensor(rng, shape, lo, hi, dtype):
    return torch.from_numpy(rng.integers(lo, hi + 1, size=shape).astype(np.float32)).to(_TD[dtype])


def _padded(x16: torch.Tensor, pad: int, dtype):
    """Copy of a 2-D 16-bit tensor into a buffer with `pad` extra NaN columns.

    Returns (buffer as uint16 numpy, leading dimension)."""
    bits = x16.contiguous().view(torch.int16).numpy().view(np.uint16)
    rows, cols = bits.shape
    buf = np.full((rows, cols + pad), F16_NAN if dtype == F16 else BF16_NAN, dtype=np.uint16)
    buf[:, :cols] = bits
    return buf, cols + pad


def _as_int_lists(x: torch.Tensor):
    return x.to(torch.int64).tolist()


def pin_decoders(orc):
    h = np.arange(65536, dtype=np.uint32)
    ref16 = h.astype(np.uint16).view(np.float16).astype(np.float64)
    refbf = (h << 16).view(np.float32).astype(np.float64)
    got16 = np.array([orc.decode_f16(x) for x in range(65536)])
    gotbf = np.array([orc.decode_bf16(x) for x in range(65536)])
    assert _same(got16, ref16), "fp16 decoder disagrees with IEEE binary16"
    assert _same(gotbf, refbf), "bf16 decoder disagrees with the upper half of binary32"


def pin_fp8_decoders(orc):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    for dtype, decode in ((E4M3, orc.decode_e4m3), (E5M2, orc.decode_e5m2)):
        ref = codes.view(_TD[dtype]).to(torch.float64).numpy()
        got = np.array([decode(x) for x in range(256)])
        assert _same(got, ref), "fp8 decoder %d disagrees with torch's conversion" % dtype
    # fixed points of the formats
    assert orc.decode_e4m3(0x7E) == 448.0 and orc.decode_e4m3(0xFE) == -448.0
    assert orc.decode_e4m3(0x01) == 2.0 ** -9 and orc.decode_e4m3(0x08) == 2.0 ** -6
    assert orc.decode_e4m3(0x38) == 1.0 and orc.decode_e4m3(0x78) == 256.0
    nan4 = [b for b in range(256) if np.isnan(orc.decode_e4m3(b))]
    assert nan4 == [0x7F, 0xFF], "E4M3 has exactly one NaN pattern per sign"
    assert orc.decode_e5m2(0x7B) == 57344.0 and orc.decode_e5m2(0x01) == 2.0 ** -16
    assert orc.decode_e5m2(0x3C) == 1.0 and orc.decode_e5m2(0x04) == 2.0 ** -14
    assert orc.decode_e5m2(0x7C) == np.inf and orc.decode_e5m2(0xFC) == -np.inf
    assert all(np.isnan(orc.decode_e5m2(b)) for b in (0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF))


def _padded8(x8: torch.Tensor, pad: int):
    """Copy of a 2-D fp8 tensor into a byte buffer with `pad` extra NaN columns
    (0x7F is NaN in both formats).  Returns (buffer, leading dimension)."""
    bits = x8.contiguous().view(torch.uint8).numpy()
    rows, cols = bits.shape
    buf = np.full((rows, cols + pad), 0x7F, dtype=np.uint8)
    buf[:, :cols] = bits
    return buf, cols + pad


def pin_fp8_brute_force_integers(orc):
    """Integers in [-8, 8] are exact in both formats: D is exact."""
    rng = np.random.default_rng(43)
    for dtype in (E4M3, E5M2):
        for (M, N, K) in ((16, 8, 32), (5, 3, 9), (1, 1, 1), (9, 17, 40)):
            for transA in (0, 1):
                for transB in (0, 1):
                    A = torch.from_numpy(rng.integers(-8, 9, size=(K, M) if transA else (M, K)).astype(np.float32)).to(_TD[dtype])
                    B = torch.from_numpy(rng.integers(-8, 9, size=(N, K) if transB else (K, N)).astype(np.float32)).to(_TD[dtype])
                    C = torch.from_numpy(rng.integers(-100, 101, size=(M, N)).astype(np.float32))
                    Ab, lda = _padded8(A, 5)
                    Bb, ldb = _padded8(B, 3)
                    for alpha, beta in ((1, 0), (1, 1), (-2, 1)):
                        D, _ = orc.gemm(Ab, Bb, C.numpy(), M, N, K, transA=transA, transB=transB,
                                        alpha=alpha, beta=beta, in_dtype=dtype, lda=lda, ldb=ldb)
                        ref = _brute(A.float(), B.float(), C if beta else None, transA, transB, alpha, beta)
                        assert np.array_equal(D, np.array(ref, dtype=np.float64)), \
                            "fp8 brute force mismatch %s trans=%d%d dtype=%d" % ((M, N, K), transA, transB, dtype)


def pin_fp8_numpy_float64(orc):
    rng = np.random.default_rng(47)
    M, N, K = 21, 19, 67
    for dtype in (E4M3, E5M2):
        for transA, transB in ((0, 1), (1, 0)):
            A = torch.from_numpy(rng.standard_normal((K, M) if transA else (M, K)).astype(np.float32)).to(_TD[dtype])
            B = torch.from_numpy(rng.standard_normal((N, K) if transB else (K, N)).astype(np.float32)).to(_TD[dtype])
            C = rng.standard_normal((M, N)).astype(np.float32)
            D, bound = orc.gemm(A, B, C, M, N, K, transA=transA, transB=transB, alpha=0.75, beta=-1.5,
                                in_dtype=dtype)
            ref = 0.75 * (_op(A.double().numpy(), transA) @ _op(B.double().numpy(), transB)) - 1.5 * C.astype(np.float64)
            assert np.all(np.abs(D - ref) <= 1e-12 * bound + 1e-300), "fp8 numpy float64 mismatch (dtype=%d)" % dtype


def _brute(A, B, C, transA, transB, alpha, beta):
    """Exact integer D by the definition, Python ints only."""
    a = _as_int_lists(A)
    b = _as_int_lists(B)
    c = _as_int_lists(C) if C is not None else None
    M = len(a[0]) if transA else len(a)
    K = len(a) if transA else len(a[0])
    N = len(b) if transB else len(b[0])
    D = [[0] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            s = 0
            for k in range(K):
                aik = a[k][i] if transA else a[i][k]
                bkj = b[j][k] if transB else b[k][j]
                s += aik * bkj
            D[i][j] = alpha * s + (beta * c[i][j] if beta != 0 else 0)
    return D


def pin_brute_force_integers(orc):
    rng = np.random.default_rng(7)
    shapes = [(16, 8, 16), (3, 5, 7), (1, 1, 1), (17, 9, 33), (5, 2, 40)]
    for dtype in (F16, BF16):
        for (M, N, K) in shapes:
            for transA in (0, 1):
                for transB in (0, 1):
                    for alpha, beta in ((1, 0), (1, 1), (-3, 1), (2, 0)):
                        A = _int_tensor(rng, (K, M) if transA else (M, K), -8, 8, dtype)
                        B = _int_tensor(rng, (N, K) if transB else (K, N), -8, 8, dtype)
                        C = torch.from_numpy(rng.integers(-100, 101, size=(M, N)).astype(np.float32))
                        Ab, lda = _padded(A, 3, dtype)
                        Bb, ldb = _padded(B, 5, dtype)
                        Cb = np.full((M, N + 2), np.nan, dtype=np.float32)
                        Cb[:, :N] = C.numpy()
                        D, _ = orc.gemm(Ab, Bb, Cb, M, N, K, transA=transA, transB=transB,
                                        alpha=alpha, beta=beta, in_dtype=dtype, c_dtype=F32,
                                        lda=lda, ldb=ldb, ldc=N + 2)
                        ref = _brute(A, B, C if beta else None, transA, transB, alpha, beta)
                        assert np.array_equal(D, np.array(ref, dtype=np.float64)), \
                            "brute force mismatch M,N,K=%s trans=%d%d alpha=%s beta=%s dtype=%d" % (
                                (M, N, K), transA, transB, alpha, beta, dtype)


def _op(x64, trans):
    return x64.T if trans else x64


def pin_numpy_float64(orc):
    rng = np.random.default_rng(11)
    M, N, K = 37, 29, 53
    for dtype in (F16, BF16):
        for transA in (0, 1):
            for transB in (0, 1):
                A = torch.from_numpy(rng.standard_normal((K, M) if transA else (M, K)).astype(np.float32)).to(_TD[dtype])
                B = torch.from_numpy(rng.standard_normal((N, K) if transB else (K, N)).astype(np.float32)).to(_TD[dtype])
                C = rng.standard_normal((M, N)).astype(np.float32)
                D, bound = orc.gemm(A, B, C, M, N, K, transA=transA, transB=transB,
                                    alpha=1.5, beta=0.5, in_dtype=dtype)
                a64 = _op(A.double().numpy(), transA)
                b64 = _op(B.double().numpy(), transB)
                ref = 1.5 * (a64 @ b64) + 0.5 * C.astype(np.float64)
                assert np.all(np.abs(D - ref) <= 1e-12 * bound + 1e-300), \
                    "numpy float64 matmul mismatch (trans=%d%d dtype=%d)" % (transA, transB, dtype)


def pin_identity(orc):
    rng = np.random.default_rng(13)
    K, N = 24, 19
    for dtype in (F16, BF16):
        for transB in (0, 1):
            eye = torch.eye(K, dtype=_TD[dtype])
            B = torch.from_numpy(rng.standard_normal((N, K) if transB else (K, N)).astype(np.float32)).to(_TD[dtype])
            C = rng.standard_normal((K, N)).astype(np.float32)
            D, _ = orc.gemm(eye, B, C, K, N, K, transB=transB, alpha=1.5, beta=0.5, in_dtype=dtype)
            ref = 1.5 * _op(B.double().numpy(), transB) + 0.5 * C.astype(np.float64)
            assert _same(D, ref), "identity operand: D != alpha*B + beta*C"


def pin_permutation(orc):
    rng = np.random.default_rng(17)
    K, N = 21, 13
    perm = rng.permutation(K)
    P = torch.zeros((K, K), dtype=torch.float16)
    P[torch.arange(K), torch.from_numpy(perm)] = 1.0
    B = torch.from_numpy(rng.standard_normal((K, N)).astype(np.float32)).half()
    for transA in (0, 1):
        A = P.T.contiguous() if transA else P
        D, _ = orc.gemm(A, B, None, K, N, K, transA=transA)
        assert _same(D, B.double().numpy()[perm, :]), "permutation operand: rows not permuted"


def pin_beta_semantics(orc):
    rng = np.random.default_rng(19)
    M, N, K = 9, 11, 14
    A = _int_tensor(rng, (M, K), -8, 8, F16)
    B = _int_tensor(rng, (K, N), -8, 8, F16)
    C = rng.integers(-50, 51, size=(M, N)).astype(np.float32)
    D0, _ = orc.gemm(A, B, C, M, N, K, beta=0.0)
    D1, _ = orc.gemm(A, B, C, M, N, K, beta=1.0)
    assert np.array_equal(D1 - D0, C.astype(np.float64)), "D(beta=1) - D(beta=0) != C"
    Cnan = np.full((M, N), np.nan, dtype=np.float32)
    Dn, bn = orc.gemm(A, B, Cnan, M, N, K, beta=0.0)
    assert np.all(np.isfinite(Dn)) and np.all(np.isfinite(bn)), "beta=0 read C"
    assert np.array_equal(Dn, D0)
    # K = 0: the sum is empty, D = beta * C
    Dk, bk = orc.gemm(None, None, C, M, N, 0, alpha=2.0, beta=0.5, lda=1, ldb=N)
    assert np.array_equal(Dk, 0.5 * C.astype(np.float64)) and np.array_equal(bk, np.abs(0.5 * C.astype(np.float64)))


def pin_transpose_equivalence(orc):
    rng = np.random.default_rng(23)
    M, N, K = 13, 10, 27
    for dtype in (F16, BF16):
        A = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(_TD[dtype])
        B = torch.from_numpy(rng.standard_normal((K, N)).astype(np.float32)).to(_TD[dtype])
        base, _ = orc.gemm(A, B, None, M, N, K, in_dtype=dtype)
        for transA in (0, 1):
            for transB in (0, 1):
                As = A.T.contiguous() if transA else A
                Bs = B.T.contiguous() if transB else B
                D, _ = orc.gemm(As, Bs, None, M, N, K, transA=transA, transB=transB, in_dtype=dtype)
                assert _same(D, base), "transpose forms disagree (trans=%d%d)" % (transA, transB)


def pin_linearity(orc):
    rng = np.random.default_rng(29)
    M, N, K = 12, 15, 31
    A = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).half()
    B = torch.from_numpy(rng.standard_normal((K, N)).astype(np.float32)).half()
    C = rng.standard_normal((M, N)).astype(np.float32)
    D10, b10 = orc.gemm(A, B, C, M, N, K, alpha=1.0, beta=0.0)
    for alpha, beta in ((1.5, 0.5), (-2.0, 3.0), (0.25, -1.0)):
        D, bound = orc.gemm(A, B, C, M, N, K, alpha=alpha, beta=beta)
        ref = alpha * D10 + beta * C.astype(np.float64)
        assert np.all(np.abs(D - ref) <= 1e-14 * bound), "not linear in alpha, beta"


def pin_closed_form(orc):
    """A[i][k] = i + 2k + 1, B[k][j] = 3k - j + 1:
    D[i][j] = K(i+1)(1-j) + (3(i+1) + 2(1-j)) K(K-1)/2 + 6 (K-1)K(2K-1)/6."""
    M, N, K = 7, 6, 37
    i = np.arange(M)[:, None]
    k = np.arange(K)[None, :]
    A = torch.from_numpy((i + 2 * k + 1).astype(np.float32)).half()
    kk = np.arange(K)[:, None]
    j = np.arange(N)[None, :]
    B = torch.from_numpy((3 * kk - j + 1).astype(np.float32)).half()
    s1 = K * (K - 1) // 2
    s2 = (K - 1) * K * (2 * K - 1) // 6
    ii, jj = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    ref = K * (ii + 1) * (1 - jj) + (3 * (ii + 1) + 2 * (1 - jj)) * s1 + 6 * s2
    for transA in (0, 1):
        for transB in (0, 1):
            As = A.T.contiguous() if transA else A
            Bs = B.T.contiguous() if transB else B
            D, _ = orc.gemm(As, Bs, None, M, N, K, transA=transA, transB=transB)
            assert np.array_equal(D, ref.astype(np.float64)), "closed-form sum mismatch"


def pin_bound(orc):
    rng = np.random.default_rng(31)
    M, N, K = 8, 9, 20
    # all terms non-negative: the bound equals D
    A = _int_tensor(rng, (M, K), 0, 8, F16)
    B = _int_tensor(rng, (K, N), 0, 8, F16)
    C = rng.integers(0, 40, size=(M, N)).astype(np.float32)
    D, bound = orc.gemm(A, B, C, M, N, K, alpha=2.0, beta=1.0)
    assert np.array_equal(D, bound), "bound != D for non-negative terms"
    # ones @ (-ones): D = -alpha*K, bound = |alpha|*K (+ |beta||C|)
    A = torch.ones((M, K), dtype=torch.float16)
    B = -torch.ones((K, N), dtype=torch.float16)
    D, bound = orc.gemm(A, B, C, M, N, K, alpha=-1.5, beta=-0.5)
    assert np.array_equal(D, 1.5 * K - 0.5 * C.astype(np.float64))
    assert np.array_equal(bound, 1.5 * K + 0.5 * np.abs(C.astype(np.float64)))
    # mixed signs: |D| <= bound
    A = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).half()
    B = torch.from_numpy(rng.standard_normal((K, N)).astype(np.float32)).half()
    D, bound = orc.gemm(A, B, C, M, N, K, alpha=0.7, beta=-1.3)
    assert np.all(np.abs(D) <= bound * (1 + 1e-12)), "|D| exceeds its bound"


def pin_entries_match_rows(orc):
    rng = np.random.default_rng(37)
    M, N, K = 23, 17, 29
    for transA, transB in ((0, 0), (1, 1)):
        A = torch.from_numpy(rng.standard_normal((K, M) if transA else (M, K)).astype(np.float32)).bfloat16()
        B = torch.from_numpy(rng.standard_normal((N, K) if transB else (K, N)).astype(np.float32)).bfloat16()
        C = rng.standard_normal((M, N)).astype(np.float32)
        kw = dict(transA=transA, transB=transB, alpha=1.25, beta=-0.75, in_dtype=BF16)
        D, bound = orc.gemm(A, B, C, M, N, K, **kw)
        r = rng.integers(0, M, size=50)
        c = rng.integers(0, N, size=50)
        De, be = orc.gemm_entries(A, B, C, M, N, K, r, c, **kw)
        assert _same(De, D[r, c]) and _same(be, bound[r, c]), "entry path disagrees with row path"
        # a second row-range call fills only its rows
        Dp, _ = orc.gemm(A, B, C, M, N, K, rows=(5, 9), **kw)
        assert _same(Dp[5:9], D[5:9]) and np.all(np.isnan(Dp[:5]))


def pin_16bit_c(orc):
    """C in fp16 / bf16 (16-bit outputs) is decoded like the operands."""
    rng = np.random.default_rng(41)
    M, N, K = 6, 5, 4
    A = _int_tensor(rng, (M, K), -4, 4, F16)
    B = _int_tensor(rng, (K, N), -4, 4, F16)
    for cd in (F16, BF16):
        C = _int_tensor(rng, (M, N), -30, 30, cd)
        D, _ = orc.gemm(A, B, C, M, N, K, beta=1.0, c_dtype=cd)
        ref = _brute(A, B, C, 0, 0, 1, 1)
        assert np.array_equal(D, np.array(ref, dtype=np.float64)), "16-bit C decoded wrongly"


def pin_rejects_bad_arguments(orc):
    A = torch.zeros((4, 4), dtype=torch.float16)
    bad = [
        dict(lda=3),                      # row longer than the leading dimension
        dict(ldb=2),
        dict(in_dtype=F32),               # operands must be 16- or 8-bit floating point
        dict(in_dtype=7),
    ]
    for kw in bad:
        try:
            orc.gemm(A, A, None, 4, 4, 4, **kw)
        except ValueError:
            continue
        raise AssertionError("oracle accepted malformed arguments %s" % kw)


# ---- MX block scaling ------------------------------------------------------

UE8M0_NAN = 0xFF


def pin_ue8m0_decoder(orc):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = np.array([orc.decode_ue8m0(x) for x in range(256)])
    assert _same(got, ref), "UE8M0 decoder disagrees with torch's float8_e8m0fnu"
    assert orc.decode_ue8m0(127) == 1.0 and orc.decode_ue8m0(128) == 2.0 and orc.decode_ue8m0(126) == 0.5
    assert orc.decode_ue8m0(0) == 2.0 ** -127 and orc.decode_ue8m0(254) == 2.0 ** 127
    assert np.isnan(orc.decode_ue8m0(UE8M0_NAN))


def _mx_case(rng, M, N, K, transA, transB, dtype, lo=121, hi=133):
    """Integer-valued 8-bit operands, scales in [lo, hi], scale rows padded
    with NaN scales (so a scale read from the padding shows)."""
    A = torch.from_numpy(rng.integers(-8, 9, size=(K, M) if transA else (M, K)).astype(np.float32)).to(_TD[dtype])
    B = torch.from_numpy(rng.integers(-8, 9, size=(N, K) if transB else (K, N)).astype(np.float32)).to(_TD[dtype])
    kb = (K + 31) // 32
    sfa = np.full((M, kb + 3), UE8M0_NAN, dtype=np.uint8)
    sfb = np.full((N, kb + 1), UE8M0_NAN, dtype=np.uint8)
    sfa[:, :kb] = rng.integers(lo, hi + 1, size=(M, kb))
    sfb[:, :kb] = rng.integers(lo, hi + 1, size=(N, kb))
    return A, B, sfa, sfb


def _mx_brute(A, B, sfa, sfb, C, transA, transB, alpha, beta):
    """Exact D by the definition in Python rationals."""
    from fractions import Fraction
    a = _as_int_lists(A.float())
    b = _as_int_lists(B.float())
    M = len(a[0]) if transA else len(a)
    K = len(a) if transA else len(a[0])
    N = len(b) if transB else len(b[0])
    out = []
    for i in range(M):
        row = []
        for j in range(N):
            acc = Fraction(0)
            for k in range(K):
                x = a[k][i] if transA else a[i][k]
                y = b[j][k] if transB else b[k][j]
                e = int(sfa[i, k // 32]) + int(sfb[j, k // 32]) - 254
                acc += Fraction(x * y) * (Fraction(2) ** e)
            d = Fraction(alpha) * acc
            if beta != 0:
                d += Fraction(beta) * Fraction(float(C[i, j]))
            row.append(float(d))
        out.append(row)
    return np.array(out, dtype=np.float64)


def pin_mx_brute_force(orc):
    rng = np.random.default_rng(53)
    for dtype in (E4M3, E5M2):
        for (M, N, K) in ((3, 4, 70), (2, 5, 32), (4, 3, 33), (1, 1, 1), (5, 2, 96)):
            for transA in (0, 1):
                for transB in (0, 1):
                    A, B, sfa, sfb = _mx_case(rng, M, N, K, transA, transB, dtype)
                    Ab, lda = _padded8(A, 5)
                    Bb, ldb = _padded8(B, 3)
                    C = rng.integers(-50, 51, size=(M, N)).astype(np.float32)
                    for alpha, beta in ((1, 0), (-0.5, 1)):
                        D, _ = orc.gemm(Ab, Bb, C, M, N, K, transA=transA, transB=transB, alpha=alpha,
                                        beta=beta, in_dtype=dtype, lda=lda, ldb=ldb, sfa=sfa, sfb=sfb)
                        ref = _mx_brute(A, B, sfa, sfb, C, transA, transB, alpha, beta)
                        assert np.array_equal(D, ref), "MX brute force mismatch %s trans=%d%d dtype=%d" % (
                            (M, N, K), transA, transB, dtype)


def pin_mx_unit_scales(orc):
    """Scale 127 (= 1) everywhere: the unscaled 8-bit product, bit for bit."""
    rng = np.random.default_rng(59)
    M, N, K = 7, 9, 100
    for dtype in (E4M3, E5M2):
        A = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(_TD[dtype])
        B = torch.from_numpy(rng.standard_normal((N, K)).astype(np.float32)).to(_TD[dtype])
        ones_a = np.full((M, 4), 127, dtype=np.uint8)
        ones_b = np.full((N, 4), 127, dtype=np.uint8)
        D, bound = orc.gemm(A, B, None, M, N, K, transB=1, in_dtype=dtype, sfa=ones_a, sfb=ones_b)
        D0, bound0 = orc.gemm(A, B, None, M, N, K, transB=1, in_dtype=dtype)
        assert _same(D, D0) and _same(bound, bound0), "unit scales change the product"


def pin_mx_row_column_scaling(orc):
    """One more on every scale of row i of A doubles row i of D exactly; two
    more on column j's scales of B quadruple column j; nothing else moves."""
    rng = np.random.default_rng(61)
    M, N, K = 6, 5, 80
    A, B, sfa, sfb = _mx_case(rng, M, N, K, 0, 1, E4M3)
    D, _ = orc.gemm(A, B, None, M, N, K, transB=1, in_dtype=E4M3, sfa=sfa, sfb=sfb)
    kb = 3
    sfa2 = sfa.copy()
    sfa2[2, :kb] += 1
    D2, _ = orc.gemm(A, B, None, M, N, K, transB=1, in_dtype=E4M3, sfa=sfa2, sfb=sfb)
    ref = D.copy()
    ref[2, :] *= 2
    assert _same(D2, ref), "raising one row's scales must double that row only"
    sfb2 = sfb.copy()
    sfb2[4, :kb] += 2
    D3, _ = orc.gemm(A, B, None, M, N, K, transB=1, in_dtype=E4M3, sfa=sfa, sfb=sfb2)
    ref = D.copy()
    ref[:, 4] *= 4
    assert _same(D3, ref), "raising one column's scales must quadruple that column only"


def pin_mx_block_exchange(orc):
    """Moving a factor 2^e from A's scales of block kb to B's leaves D
    unchanged; moving it into another block changes it."""
    rng = np.random.default_rng(67)
    M, N, K = 4, 6, 96
    A, B, sfa, sfb = _mx_case(rng, M, N, K, 1, 0, E5M2)
    D, _ = orc.gemm(A, B, None, M, N, K, transA=1, in_dtype=E5M2, sfa=sfa, sfb=sfb)
    sfa2, sfb2 = sfa.copy(), sfb.copy()
    sfa2[:, 1] += 3
    sfb2[:, 1] -= 3
    D2, _ = orc.gemm(A, B, None, M, N, K, transA=1, in_dtype=E5M2, sfa=sfa2, sfb=sfb2)
    assert _same(D, D2), "a factor moved between A's and B's scales of one block changed D"
    sfb3 = sfb.copy()
    sfb3[:, 2] -= 3
    D3, _ = orc.gemm(A, B, None, M, N, K, transA=1, in_dtype=E5M2, sfa=sfa2, sfb=sfb3)
    assert not _same(D, D3), "scales of different blocks must not cancel"


def pin_mx_block_boundary(orc):
    """Elements k = 31 and k = 32 fall in blocks 0 and 1: closed form."""
    K = 64
    A = torch.zeros((1, K), dtype=torch.float8_e4m3fn)
    B = torch.zeros((1, K), dtype=torch.float8_e4m3fn)
    A[0, 31] = 3.0
    A[0, 32] = 5.0
    B[0, 31] = 2.0
    B[0, 32] = 7.0
    sfa = np.array([[130, 120]], dtype=np.uint8)   # 2^3, 2^-7
    sfb = np.array([[125, 131]], dtype=np.uint8)   # 2^-2, 2^4
    D, bound = orc.gemm(A, B, None, 1, 1, K, transB=1, in_dtype=E4M3, sfa=sfa, sfb=sfb)
    want = 3 * 2 * 2.0 ** (3 - 2) + 5 * 7 * 2.0 ** (-7 + 4)
    assert D[0, 0] == want and bound[0, 0] == want, "block boundary misplaced"


def pin_mx_nan_scale(orc):
    """A NaN scale (0xFF) makes its block NaN: every D element whose sum
    takes a product from that block is NaN, the rest are finite."""
    rng = np.random.default_rng(71)
    M, N, K = 4, 3, 64
    A, B, sfa, sfb = _mx_case(rng, M, N, K, 0, 0, E4M3)
    sfa = np.ascontiguousarray(sfa[:, :2])
    sfb = np.ascontiguousarray(sfb[:, :2])
    sfa[1, 1] = UE8M0_NAN
    sfb[2, 0] = UE8M0_NAN
    D, _ = orc.gemm(A, B, None, M, N, K, in_dtype=E4M3, sfa=sfa, sfb=sfb)
    expect_nan = np.zeros((M, N), dtype=bool)
    expect_nan[1, :] = True
    expect_nan[:, 2] = True
    assert np.array_equal(np.isnan(D), expect_nan), "NaN scales propagate wrongly"


def pin_mx_numpy_float64(orc):
    rng = np.random.default_rng(73)
    M, N, K = 13, 11, 150
    kb = (K + 31) // 32
    for dtype in (E4M3, E5M2):
        A = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(_TD[dtype])
        B = torch.from_numpy(rng.standard_normal((N, K)).astype(np.float32)).to(_TD[dtype])
        sfa = rng.integers(110, 140, size=(M, kb)).astype(np.uint8)
        sfb = rng.integers(110, 140, size=(N, kb)).astype(np.uint8)
        C = rng.standard_normal((M, N)).astype(np.float32)
        D, bound = orc.gemm(A, B, C, M, N, K, transB=1, alpha=1.25, beta=0.5, in_dtype=dtype,
                            sfa=sfa, sfb=sfb)
        ea = np.repeat(sfa.astype(np.float64) - 127.0, 32, axis=1)[:, :K]
        eb = np.repeat(sfb.astype(np.float64) - 127.0, 32, axis=1)[:, :K]
        a = A.double().numpy() * np.exp2(ea)
        b = B.double().numpy() * np.exp2(eb)
        ref = 1.25 * (a @ b.T) + 0.5 * C.astype(np.float64)
        assert np.all(np.abs(D - ref) <= 1e-12 * bound), "MX numpy float64 mismatch (dtype=%d)" % dtype


E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]   # the OCP E2M1 magnitudes, codes 0..7


def pin_e2m1_decoder(orc):
    got = [orc.decode_e2m1(c) for c in range(16)]
    assert got[:8] == E2M1_VALUES, "E2M1 positive codes"
    assert got[8:] == [-v for v in E2M1_VALUES], "E2M1 sign bit"
    assert np.signbit(got[8]), "code 8 is -0"


def pin_e2m1_packing(orc):
    """Byte 0x71 holds element 0 = code 1 (0.5) in the low nibble and element
    1 = code 7 (6.0) in the high nibble."""
    A = np.array([[0x71]], dtype=np.uint8)            # [1, K = 2]
    one = np.array([[127]], dtype=np.uint8)
    for b, want in ((0x02, 0.5), (0x20, 6.0), (0x22, 6.5)):
        B = np.array([[b]], dtype=np.uint8)           # stored [N = 1, K = 2]
        D, _ = orc.gemm(A, B, None, 1, 1, 2, transB=1, in_dtype=E2M1, sfa=one, sfb=one)
        assert D[0, 0] == want, "E2M1 nibble order (byte 0x%02x)" % b
    # a row of 3 elements with ld 4: the second row starts at byte 2
    A2 = np.array([[0x21, 0x03], [0x54, 0x06]], dtype=np.uint8)   # rows (1.0, 0.5, 1.5), (2.0, 3.0, 4.0)
    B2 = np.array([[0x22, 0x02]], dtype=np.uint8)                 # (1, 1, 1)
    D2, _ = orc.gemm(A2, B2, None, 2, 1, 3, lda=4, ldb=4, transB=1, in_dtype=E2M1,
                     sfa=np.full((2, 1), 127, np.uint8), sfb=one)
    assert D2[:, 0].tolist() == [3.0, 9.0], "packed rows with a leading dimension"


def _unpack_e2m1(packed, rows, cols, ld):
    """Element values of a packed row-major fp4 array, in Python floats."""
    flat = packed.reshape(-1)
    out = []
    for r in range(rows):
        row = []
        for c in range(cols):
            e = r * ld + c
            code = (int(flat[e // 2]) >> (4 * (e % 2))) & 0xF
            v = E2M1_VALUES[code & 7]
            row.append(-v if code & 8 else v)
        out.append(row)
    return out


def pin_mx_fp4_brute_force(orc):
    from fractions import Fraction
    rng = np.random.default_rng(79)
    for (M, N, K) in ((3, 4, 70), (2, 3, 64), (5, 2, 2)):
        lda, ldb = K + 6, K + 2
        A = rng.integers(0, 256, size=(M, lda // 2), dtype=np.uint8)
        B = rng.integers(0, 256, size=(N, ldb // 2), dtype=np.uint8)
        kb = (K + 31) // 32
        sfa = rng.integers(124, 131, size=(M, kb)).astype(np.uint8)
        sfb = rng.integers(124, 131, size=(N, kb)).astype(np.uint8)
        D, _ = orc.gemm(A, B, None, M, N, K, lda=lda, ldb=ldb, transB=1, in_dtype=E2M1, sfa=sfa, sfb=sfb)
        a = _unpack_e2m1(A, M, K, lda)
        b = _unpack_e2m1(B, N, K, ldb)
        for i in range(M):
            for j in range(N):
                acc = Fraction(0)
                for k in range(K):
                    e = int(sfa[i, k // 32]) + int(sfb[j, k // 32]) - 254
                    acc += Fraction(a[i][k]) * Fraction(b[j][k]) * Fraction(2) ** e
                assert D[i, j] == float(acc), "fp4 brute force %s at (%d, %d)" % ((M, N, K), i, j)


def pin_mx_rejects_bad_arguments(orc):
    A8 = torch.zeros((4, 64), dtype=torch.float8_e4m3fn)
    A16 = torch.zeros((4, 64), dtype=torch.float16)
    s2 = np.zeros((4, 2), dtype=np.uint8)
    s1 = np.zeros((4, 1), dtype=np.uint8)
    bad = [
        (A16, dict(in_dtype=F16, sfa=s2, sfb=s2)),       # block scaling is for 8-bit operands
        (A8, dict(in_dtype=E4M3, sfa=s1, sfb=s2)),       # a scale row shorter than ceil(K/32)
        (A8, dict(in_dtype=E4M3, sfa=s2, sfb=s1)),
        (A8, dict(in_dtype=E4M3, sfa=s2, sfb=None)),     # both scale arrays or neither
    ]
    for A, kw in bad:
        try:
            orc.gemm(A, A, None, 4, 4, 64, transB=1, **kw)
        except ValueError:
            continue
        raise AssertionError("oracle accepted malformed block-scaled arguments %s" % list(kw))


ALL_PINS = [
    pin_decoders,
    pin_fp8_decoders,
    pin_fp8_brute_force_integers,
    pin_fp8_numpy_float64,
    pin_brute_force_integers,
    pin_numpy_float64,
    pin_identity,
    pin_permutation,
    pin_beta_semantics,
    pin_transpose_equivalence,
    pin_linearity,
    pin_closed_form,
    pin_bound,
    pin_entries_match_rows,
    pin_16bit_c,
    pin_rejects_bad_arguments,
    pin_ue8m0_decoder,
    pin_mx_brute_force,
    pin_mx_unit_scales,
    pin_mx_row_column_scaling,
    pin_mx_block_exchange,
    pin_mx_block_boundary,
    pin_mx_nan_scale,
    pin_mx_numpy_float64,
    pin_mx_rejects_bad_arguments,
    pin_e2m1_decoder,
    pin_e2m1_packing,
    pin_mx_fp4_brute_force,
]
