"""Stream-K (tiles split along K, finished by the last contributor) against
the oracle on the GPU.  GEMM_SK_MIN_ITERS=1 forces the finest split, so
tiles get many contributors and every fixup path runs."""
import numpy as np
import pytest
import torch

from dense_tensor_core_02_gb300 import binding
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    yield
    assert H.poll()[0] == 0


@pytest.fixture(params=["pair", "single", "narrow"])
def variant(request):
    with H.env(GEMM_PATH="tcgen05", GEMM_VARIANT=request.param):
        yield request.param


def _plan(M, N, K):
    return binding.gemm_plan(M, N, K, torch.cuda.get_device_properties(0).multi_processor_count)


SHAPES = [(1000, 1000, 1000), (600, 520, 1000), (256, 256, 4096), (1024, 768, 520), (130, 264, 2056)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_streamk_integers_exact(variant, shape):
    M, N, K = shape
    with H.env(GEMM_SK_MIN_ITERS="1"):
        assert _plan(M, N, K)["sk_tiles"] > 0
        A = H.int_matrix((M, K), -4, 4, "f16", M + K)
        B = H.int_matrix((K, N), -4, 4, "f16", N + K)
        C = H.int_matrix((M, N), -50, 50, "f32", M + N)
        D, rc = H.run_gemm(A, B, C, M, N, K, beta=1.0)
    assert rc == 0
    ref, _ = H.oracle_full(A, B, C, M, N, K, beta=1.0)
    H.assert_exact(D.numpy(), ref, "stream-K %s %s" % (variant, shape))


@pytest.mark.parametrize("transA,transB", [(0, 0), (1, 1), (0, 1)])
@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_streamk_random(variant, transA, transB, out_dtype):
    M, N, K = 520, 392, 1544
    A = H.normal_matrix((K, M) if transA else (M, K), "bf16", 3)
    B = H.normal_matrix((N, K) if transB else (K, N), "bf16", 4)
    C = H.normal_matrix((M, N), out_dtype, 5)
    kw = dict(transA=transA, transB=transB, alpha=-1.25, beta=0.5, in_dtype="bf16", out_dtype=out_dtype)
    with H.env(GEMM_SK_MIN_ITERS="1"):
        assert _plan(M, N, K)["sk_tiles"] > 0
        D, rc = H.run_gemm(A, B, C, M, N, K, **kw)
    assert rc == 0
    ref, bound = H.oracle_full(A, B, C, M, N, K, **kw)
    H.assert_close(D.double().numpy(), ref, bound, out_dtype, "stream-K random")


def test_streamk_repeatable_and_workspace_reuse():
    """Same call twice: same bits (contributors are summed in K order, not
    arrival order); calls of other shapes in between reuse the workspace."""
    shapes = [(1000, 1000, 1000), (600, 520, 1000), (1000, 1000, 1000)]
    outs = []
    with H.env(GEMM_SK_MIN_ITERS="1"):
        for (M, N, K) in shapes:
            A = H.normal_matrix((M, K), "f16", 7)
            B = H.normal_matrix((K, N), "f16", 8)
            D, rc = H.run_gemm(A, B, None, M, N, K)
            assert rc == 0
            outs.append(D)
    assert torch.equal(outs[0], outs[2])
    M, N, K = shapes[1]
    A = H.normal_matrix((M, K), "f16", 7)
    B = H.normal_matrix((K, N), "f16", 8)
    ref, bound = H.oracle_full(A, B, None, M, N, K)
    H.assert_close(outs[1].numpy(), ref, bound, what="workspace reuse")


def test_streamk_two_streams():
    """Calls on two streams at once use separate workspaces."""
    M, N, K = 1000, 1000, 1000
    dev = torch.device("cuda", 0)
    A1 = H.int_matrix((M, K), -4, 4, "f16", 11)
    B1 = H.int_matrix((K, N), -4, 4, "f16", 12)
    A2 = H.int_matrix((M, K), -4, 4, "f16", 13)
    B2 = H.int_matrix((K, N), -4, 4, "f16", 14)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    D1 = torch.empty(M, N, device=dev)
    D2 = torch.empty(M, N, device=dev)
    a1, b1, a2, b2 = A1.to(dev), B1.to(dev), A2.to(dev), B2.to(dev)
    torch.cuda.synchronize()
    with H.env(GEMM_SK_MIN_ITERS="1"):
        for _ in range(3):
            assert binding.gemm(D1, a1, b1, None, M, N, K, K, N, N, N, 0, 0, 1.0, 0.0, 0, 2, s1) == 0
            assert binding.gemm(D2, a2, b2, None, M, N, K, K, N, N, N, 0, 0, 1.0, 0.0, 0, 2, s2) == 0
    torch.cuda.synchronize()
    r1, _ = H.oracle_full(A1, B1, None, M, N, K)
    r2, _ = H.oracle_full(A2, B2, None, M, N, K)
    H.assert_exact(D1.cpu().numpy(), r1, "stream 1")
    H.assert_exact(D2.cpu().numpy(), r2, "stream 2")


def test_default_plan_uses_streamk_on_headline_shape():
    p = _plan(8192, 8192, 8192)
    assert p["sk_tiles"] == p["num_tiles"] % (p["grid"] // 2) > 0


def test_streamk_off_matches_on_within_tolerance():
    M, N, K = 1000, 1000, 1000
    A = H.normal_matrix((M, K), "f16", 21)
    B = H.normal_matrix((K, N), "f16", 22)
    with H.env(GEMM_STREAMK="0"):
        assert _plan(M, N, K)["sk_tiles"] == 0
        D0, rc0 = H.run_gemm(A, B, None, M, N, K)
    D1, rc1 = H.run_gemm(A, B, None, M, N, K)
    assert rc0 == 0 and rc1 == 0
    ref, bound = H.oracle_full(A, B, None, M, N, K)
    H.assert_close(D0.numpy(), ref, bound, what="data-parallel")
    H.assert_close(D1.numpy(), ref, bound, what="stream-K")
    assert np.isfinite(D1.numpy()).all()
