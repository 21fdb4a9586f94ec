"""Extreme shapes against the oracle: a million rows, a million columns, a
K of a million (stream-K over every SM, one tile), a 16384 x 16384 output,
and block-scaled operands with a deep K.  Integer-valued inputs keep every
fp32 partial sum exact, so outputs are compared bit for bit at sampled
positions that touch every 128 x 128 output block (or, for the single deep
tile, at random positions).
"""
import numpy as np
import pytest
import torch

import oracle.oracle as oracle
from dense_tensor_core_02_gb300 import binding
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    yield
    rc, info = H.poll()
    assert rc == 0, ("device status after the module", rc, info)


@pytest.mark.parametrize("M,N,K", [(1 << 20 | 3, 24, 40), (24, 1 << 20 | 5, 40), (16384, 16384, 64)],
                         ids=["million_rows", "million_cols", "16k_square_output"])
def test_extreme_output_shapes(M, N, K):
    A = H.int_matrix((M, K), -4, 4, "f16", M % 97)
    B = H.int_matrix((K, N), -4, 4, "f16", N % 89)
    D, rc = H.run_gemm(A, B, None, M, N, K)
    assert rc == 0
    assert not torch.isnan(D).any(), "unwritten output elements"
    rows, cols = H.sample_positions(M, N, per_block=2, seed=M + N)
    ref, _ = H.oracle_at(A, B, None, M, N, K, rows, cols)
    H.assert_exact(D.numpy()[rows, cols], ref, "extreme %dx%dx%d" % (M, N, K))


def test_k_of_a_million_single_tile():
    """One output tile, K = 2^20: the whole reduction is split along K over
    every SM (stream-K), and the last contributor to arrive sums all partials."""
    M, N, K = 128, 128, 1 << 20
    A = H.int_matrix((M, K), -1, 1, "bf16", 5)
    B = H.int_matrix((N, K), -1, 1, "bf16", 6)
    D, rc = H.run_gemm(A, B, None, M, N, K, transB=1, in_dtype="bf16")
    assert rc == 0
    rng = np.random.default_rng(7)
    rows = rng.integers(0, M, size=256)
    cols = rng.integers(0, N, size=256)
    ref, _ = oracle.gemm_entries(A, B, None, M, N, K, rows, cols, transB=1, in_dtype=H.CODE["bf16"],
                                 threads=H.ORACLE_THREADS)
    H.assert_exact(D.numpy()[rows, cols], ref, "K = 2^20")


def test_block_scaled_deep_k():
    """E4M3 with MX scales, K = 2^18 (8192 scale blocks per row)."""
    from tests.test_mx_gpu import run_mx, scales
    M, N, K = 256, 384, 1 << 18
    A = H.int_matrix((M, K), -2, 2, "e4m3", 11)
    B = H.int_matrix((N, K), -2, 2, "e4m3", 12)
    SFA = scales(M, K, 126, 128, 13)
    SFB = scales(N, K, 126, 128, 14)
    D, rc = run_mx(A, B, None, SFA, SFB, M, N, K)
    assert rc == 0
    rng = np.random.default_rng(15)
    rows = rng.integers(0, M, size=192)
    cols = rng.integers(0, N, size=192)
    ref, _ = oracle.gemm_entries(A, B, None, M, N, K, rows, cols, transB=1, in_dtype=H.CODE["e4m3"],
                                 threads=H.ORACLE_THREADS, sfa=SFA.numpy(), sfb=SFB.numpy())
    H.assert_exact(D.numpy()[rows, cols], ref, "MX K = 2^18")
