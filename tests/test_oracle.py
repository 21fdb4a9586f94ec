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
