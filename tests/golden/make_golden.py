"""Writes the stored expected values under tests/golden/ by calling the oracle.

Run from the repository root:  python tests/golden/make_golden.py

single_atom_int_16x8x16.txt -- the one-atom problem of the TVM TIRx "gemm"
page, section "Demonstration program": one warp computes
D[16,8] = A[16,16] @ B[16,8], fp16 operands, fp32 result, alpha = 1,
beta = 0, no transpose.  The pages print no values for it, so the operands
are small integers (seeded) and D is the oracle's; with integer operands
every partial sum is exact, so any correct implementation must reproduce
these values bit for bit.
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle.oracle as oracle  # noqa: E402


def single_atom():
    rng = np.random.default_rng(20240516)
    A = rng.integers(-8, 9, size=(16, 16)).astype(np.float16)
    B = rng.integers(-8, 9, size=(16, 8)).astype(np.float16)
    D, _ = oracle.gemm(A, B, None, 16, 8, 16)
    path = os.path.join(HERE, "single_atom_int_16x8x16.txt")
    with open(path, "w") as f:
        f.write("# TVM TIRx 'gemm' page, section 'Demonstration program': one m16n8k16 atom,\n")
        f.write("# D[16,8] = A[16,16] @ B[16,8]; fp16 A, B; fp32 D; alpha=1 beta=0; row-major.\n")
        f.write("# Integer operands (seeded); D written by tests/golden/make_golden.py from the oracle.\n")
        for name, X in (("A", A), ("B", B), ("D", D)):
            f.write("%s %d %d\n" % (name, X.shape[0], X.shape[1]))
            for row in X:
                f.write(" ".join("%d" % int(v) for v in row) + "\n")
    return path


if __name__ == "__main__":
    print(single_atom())
