"""The CPU oracle against its pins (no GPU)."""
import pytest

import oracle.oracle as oracle
from tests import oracle_pins


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def _read_golden(name):
    import os
    import numpy as np
    path = os.path.join(os.path.dirname(__file__), "golden", name)
    mats, cur = {}, None
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = line.split()
            if parts[0].isalpha():
                cur = parts[0]
                mats[cur] = []
            else:
                mats[cur].append([int(v) for v in parts])
    return {k: np.array(v) for k, v in mats.items()}


def test_golden_single_atom(orc):
    """The stored single-atom fixture agrees with integer brute force and the oracle."""
    import numpy as np
    g = _read_golden("single_atom_int_16x8x16.txt")
    A, B, D = g["A"], g["B"], g["D"]
    brute = [[sum(int(A[i][k]) * int(B[k][j]) for k in range(16)) for j in range(8)] for i in range(16)]
    assert np.array_equal(D, np.array(brute))
    got, _ = orc.gemm(A.astype(np.float16), B.astype(np.float16), None, 16, 8, 16)
    assert np.array_equal(got, D.astype(np.float64))


@pytest.mark.parametrize("mx", [False, True], ids=["plain", "mx"])
def test_threaded_split_is_bit_identical(orc, mx):
    """The oracle's thread split (disjoint row blocks of D, or disjoint runs
    of listed entries, each computed by the same single-threaded loop) gives
    the same bits as one thread, for D and for the bound.  The row count (37)
    and entry count (101) divide evenly by none of the thread counts, so the
    last block of every split is short."""
    import numpy as np
    rng = np.random.default_rng(7)
    M, N, K = 37, 19, 70
    if mx:
        A = rng.integers(0, 256, (M, K), dtype=np.uint8)      # E4M3 bytes
        A[(A & 0x7F) == 0x7F] = 0x38                          # no NaNs: compare finite values
        B = rng.integers(0, 256, (N, K), dtype=np.uint8)
        B[(B & 0x7F) == 0x7F] = 0x38
        kb = (K + 31) // 32
        kw = dict(transB=1, in_dtype=oracle.E4M3, sfa=rng.integers(120, 135, (M, kb), dtype=np.uint8),
                  sfb=rng.integers(120, 135, (N, kb), dtype=np.uint8))
    else:
        A = rng.standard_normal((K, M)).astype(np.float16)    # stored [K, M]: transA
        B = rng.standard_normal((K, N)).astype(np.float16)
        kw = dict(transA=1)
    C = rng.standard_normal((M, N)).astype(np.float32)
    kw.update(alpha=1.25, beta=-0.5)
    rows = rng.integers(0, M, 101)
    cols = rng.integers(0, N, 101)
    D1, b1 = orc.gemm(A, B, C, M, N, K, threads=1, **kw)
    E1, eb1 = orc.gemm_entries(A, B, C, M, N, K, rows, cols, threads=1, **kw)
    assert np.isfinite(D1).all() and np.isfinite(E1).all()
    assert np.array_equal(E1, D1[rows, cols]) and np.array_equal(eb1, b1[rows, cols])
    for t in (3, 16):
        Dt, bt = orc.gemm(A, B, C, M, N, K, threads=t, **kw)
        assert np.array_equal(Dt, D1) and np.array_equal(bt, b1), t
        Et, ebt = orc.gemm_entries(A, B, C, M, N, K, rows, cols, threads=t, **kw)
        assert np.array_equal(Et, E1) and np.array_equal(ebt, eb1), t
