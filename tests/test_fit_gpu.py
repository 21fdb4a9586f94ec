"""The 224-wide wave-fitted CTA-pair tiles (f32 D, K-major B) against the
oracle on the GPU.  GEMM_FIT_TILES=1 takes them wherever they apply, so
small shapes exercise them with ragged edges, C, general alpha/beta, 8-bit
operands and stream-K; the planner's own choice is covered by the 4096^3
workloads (sampled at full size in test_gemm_gpu.py) and by test_abi.py."""
import numpy as np
import pytest
import torch

from dense_tensor_core_02_gb300 import binding
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

FIT_N = 224


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    yield
    assert H.poll()[0] == 0


@pytest.fixture
def fit():
    with H.env(GEMM_PATH="tcgen05", GEMM_VARIANT="pair", GEMM_FIT_TILES="1"):
        yield


def _plan(M, N, K, in_dtype="f16"):
    return binding.gemm_plan_layout(M, N, K, 1, H.CODE[in_dtype], binding.F32,
                                    torch.cuda.get_device_properties(0).multi_processor_count)


SHAPES = [(1000, 1000, 1000), (600, 520, 1000), (256, 448, 4096), (1024, 768, 520), (130, 264, 2056),
          (520, 900, 1544), (2048, 2240, 640)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("beta", [0.0, 1.0])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_fit_integers_exact(fit, shape, beta, dtype):
    M, N, K = shape
    assert _plan(M, N, K, dtype)["tile_n"] == FIT_N
    A = H.int_matrix((M, K), -4, 4, dtype, M + K)
    B = H.int_matrix((N, K), -4, 4, dtype, N + K)
    C = H.int_matrix((M, N), -50, 50, "f32", M + N) if beta else None
    D, rc = H.run_gemm(A, B, C, M, N, K, transB=1, beta=beta, in_dtype=dtype)
    assert rc == 0
    assert not torch.isnan(D).any(), "unwritten output elements"
    ref, _ = H.oracle_full(A, B, C, M, N, K, transB=1, beta=beta, in_dtype=dtype)
    H.assert_exact(D.numpy(), ref, "224-wide %s beta %g %s" % (shape, beta, dtype))


@pytest.mark.parametrize("alpha,beta", [(1.5, 0.5), (-0.75, 2.0), (0.0, 1.0)])
def test_fit_general_alpha_beta(fit, alpha, beta):
    M, N, K = 777, 1111, 904
    A = H.normal_matrix((M, K), "bf16", 31)
    B = H.normal_matrix((N, K), "bf16", 32)
    C = H.normal_matrix((M, N), "f32", 33)
    kw = dict(transB=1, alpha=alpha, beta=beta, in_dtype="bf16")
    D, rc = H.run_gemm(A, B, C, M, N, K, **kw)
    assert rc == 0
    ref, bound = H.oracle_full(A, B, C, M, N, K, **kw)
    H.assert_close(D.double().numpy(), ref, bound, "f32", "224-wide alpha %g beta %g" % (alpha, beta))


@pytest.mark.parametrize("dtype", ["e4m3", "e5m2"])
@pytest.mark.parametrize("beta", [0.0, 1.0])
def test_fit_8bit_exact(fit, dtype, beta):
    M, N, K = 640, 1000, 1408
    assert _plan(M, N, K, dtype)["tile_n"] == FIT_N
    A = H.int_matrix((M, K), -4, 4, dtype, 41)
    B = H.int_matrix((N, K), -4, 4, dtype, 42)
    C = H.int_matrix((M, N), -50, 50, "f32", 43) if beta else None
    D, rc = H.run_gemm(A, B, C, M, N, K, transB=1, beta=beta, in_dtype=dtype)
    assert rc == 0
    ref, _ = H.oracle_full(A, B, C, M, N, K, transB=1, beta=beta, in_dtype=dtype)
    H.assert_exact(D.numpy(), ref, "224-wide %s beta %g" % (dtype, beta))


@pytest.mark.parametrize("dtype", ["e4m3", "e5m2"])
def test_fit_8bit_b_stored_k_by_n(fit, dtype):
    """8-bit B stored [K, N]: the call copies it K-major into a workspace
    first, then runs the 224-wide tiles on the copy."""
    M, N, K = 520, 900, 1408   # more than 4 stages of 256: the 4-warp kernel
    assert _plan(M, N, K, dtype)["tile_n"] == FIT_N   # planned K-major whatever the stored layout
    A = H.int_matrix((M, K), -4, 4, dtype, 45)
    B = H.int_matrix((K, N), -4, 4, dtype, 46)
    C = H.int_matrix((M, N), -50, 50, "f32", 47)
    D, rc = H.run_gemm(A, B, C, M, N, K, transB=0, beta=1.0, in_dtype=dtype)
    assert rc == 0
    ref, _ = H.oracle_full(A, B, C, M, N, K, transB=0, beta=1.0, in_dtype=dtype)
    H.assert_exact(D.numpy(), ref, "224-wide %s, B stored [K, N]" % dtype)


@pytest.mark.parametrize("shape", [(1000, 1000, 1000), (256, 672, 4096), (600, 520, 2000)],
                         ids=lambda s: "x".join(map(str, s)))
def test_fit_streamk_exact(fit, shape):
    """The finest stream-K split on 224-wide tiles: partial accumulators of
    224 columns in the workspace, summed by the last contributor."""
    M, N, K = shape
    with H.env(GEMM_SK_MIN_ITERS="1"):
        p = _plan(M, N, K)
        assert p["tile_n"] == FIT_N and p["sk_tiles"] > 0
        A = H.int_matrix((M, K), -4, 4, "f16", M + 3)
        B = H.int_matrix((N, K), -4, 4, "f16", N + 5)
        C = H.int_matrix((M, N), -50, 50, "f32", 7)
        D, rc = H.run_gemm(A, B, C, M, N, K, transB=1, beta=1.0)
    assert rc == 0
    ref, _ = H.oracle_full(A, B, C, M, N, K, transB=1, beta=1.0)
    H.assert_exact(D.numpy(), ref, "224-wide stream-K %s" % (shape,))


def test_fit_matches_wide_tiles_bitwise():
    """Integer inputs: the 224- and 256-wide plans give the same bits."""
    M, N, K = 1536, 1792, 1024
    A = H.int_matrix((M, K), -3, 3, "bf16", 51)
    B = H.int_matrix((N, K), -3, 3, "bf16", 52)
    with H.env(GEMM_PATH="tcgen05", GEMM_VARIANT="pair", GEMM_FIT_TILES="1"):
        assert _plan(M, N, K, "bf16")["tile_n"] == FIT_N
        D1, rc1 = H.run_gemm(A, B, None, M, N, K, transB=1, in_dtype="bf16")
    with H.env(GEMM_PATH="tcgen05", GEMM_VARIANT="pair", GEMM_FIT_TILES="0"):
        assert _plan(M, N, K, "bf16")["tile_n"] == 256
        D0, rc0 = H.run_gemm(A, B, None, M, N, K, transB=1, in_dtype="bf16")
    assert rc0 == 0 and rc1 == 0
    assert torch.equal(D0, D1)
    rows = np.arange(0, M, 97)
    ref, _ = H.oracle_at(A, B, None, M, N, K, rows[:, None].repeat(N, 1).ravel(),
                         np.tile(np.arange(N), len(rows)), transB=1, in_dtype="bf16")
    H.assert_exact(D1.numpy()[rows].ravel(), ref, "224-wide rows")


def test_fit_not_taken_for_mn_major_b_or_16bit_d(fit):
    M, N, K = 1000, 1000, 1000
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert binding.gemm_plan_layout(M, N, K, 0, binding.F16, binding.F32, sms)["tile_n"] != FIT_N
    assert binding.gemm_plan_layout(M, N, K, 1, binding.F16, binding.BF16, sms)["tile_n"] != FIT_N
    # and the calls still run (on the 256-wide tiles)
    A = H.int_matrix((M, K), -4, 4, "f16", 61)
    B = H.int_matrix((K, N), -4, 4, "f16", 62)
    D, rc = H.run_gemm(A, B, None, M, N, K)
    assert rc == 0
    ref, _ = H.oracle_full(A, B, None, M, N, K)
    H.assert_exact(D.numpy(), ref, "MN-major B under GEMM_FIT_TILES=1")
