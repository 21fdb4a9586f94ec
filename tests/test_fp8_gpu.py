"""GPU parity of 8-bit floating-point operands (E4M3, E5M2) against the
CPU oracle: the tcgen05 kernel's kind::f8f6f4 instantiations (the 8-bit
precisions the TIRx gemm guide lists for the tcgen05 path, section 七),
fp32 accumulation, the same epilogue as fp16 / bf16.

K-major operands (A stored [M, K], B stored [N, K]) are read in place; the
other transpose forms and layouts off the 16-byte grid go through the
repacking route (MN-major operands transposed into K-major workspace).
Integers in [-8, 8] are exact in both formats, so those tests are bit-exact.
"""
import pytest
import torch

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


@pytest.fixture(params=["pair", "single", "narrow"])
def variant(request):
    with H.env(GEMM_VARIANT=request.param, GEMM_PATH=None):
        yield request.param


SHAPES = [(16, 8, 32), (128, 64, 128), (296, 264, 200), (257, 130, 33), (1, 1, 1), (640, 520, 1040)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", FP8)
@pytest.mark.parametrize("beta", [0.0, 1.0])
def test_k_major_integers_exact(variant, shape, dtype, beta):
    M, N, K = shape
    seed = 3 * M + 7 * N + K + (dtype == "e5m2") + 2 * int(beta)
    A = H.int_matrix((M, K), -8, 8, dtype, seed)
    B = H.int_matrix((N, K), -8, 8, dtype, seed + 1)
    C = H.int_matrix((M, N), -100, 100, "f32", seed + 2) if beta else None
    kw = dict(transB=1, beta=beta, in_dtype=dtype)
    D, rc = H.run_gemm(A, B, C, M, N, K, **kw)
    assert rc == 0
    ref, _ = H.oracle_full(A, B, C, M, N, K, **kw)
    H.assert_exact(D.numpy(), ref, "fp8 %s %s beta=%s" % (dtype, shape, beta))


@pytest.mark.parametrize("transA", [0, 1])
@pytest.mark.parametrize("transB", [0, 1])
@pytest.mark.parametrize("dtype", FP8)
def test_transpose_forms_integers_exact(transA, transB, dtype):
    """MN-major 8-bit operands are transposed into K-major workspace."""
    M, N, K = 392, 264, 328
    seed = 11 + 4 * transA + 2 * transB + (dtype == "e5m2")
    A = H.int_matrix((K, M) if transA else (M, K), -8, 8, dtype, seed)
    B = H.int_matrix((N, K) if transB else (K, N), -8, 8, dtype, seed + 1)
    C = H.int_matrix((M, N), -50, 50, "f32", seed + 2)
    kw = dict(transA=transA, transB=transB, beta=1.0, in_dtype=dtype)
    D, rc = H.run_gemm(A, B, C, M, N, K, **kw)
    assert rc == 0
    ref, _ = H.oracle_full(A, B, C, M, N, K, **kw)
    H.assert_exact(D.numpy(), ref, "fp8 transpose %d%d %s" % (transA, transB, dtype))


@pytest.mark.parametrize("dtype", FP8)
@pytest.mark.parametrize("out_dtype", ["f32", "f16", "bf16"])
def test_random_with_alpha_beta(dtype, out_dtype):
    M, N, K = 520, 392, 776
    seed = 31 + (dtype == "e5m2") + 2 * ["f32", "f16", "bf16"].index(out_dtype)
    A = H.normal_matrix((M, K), dtype, seed)
    B = H.normal_matrix((N, K), dtype, seed + 1)
    C = H.normal_matrix((M, N), out_dtype, seed + 2)
    kw = dict(transB=1, alpha=0.125, beta=-0.5, in_dtype=dtype, out_dtype=out_dtype)
    D, rc = H.run_gemm(A, B, C, M, N, K, **kw)
    assert rc == 0
    ref, bound = H.oracle_full(A, B, C, M, N, K, **kw)
    H.assert_close(D.double().numpy(), ref, bound, out_dtype, "fp8 random %s -> %s" % (dtype, out_dtype))


@pytest.mark.parametrize("dtype", FP8)
def test_misaligned_layouts_repacked(dtype):
    """Byte offsets and row strides off the 16-byte grid, all repacked."""
    M, N, K = 200, 136, 101
    A = H.int_matrix((M, K), -8, 8, dtype, 51)
    B = H.int_matrix((N, K), -8, 8, dtype, 52)
    C = H.int_matrix((M, N), -50, 50, "f32", 53)
    kw = dict(transB=1, beta=1.0, in_dtype=dtype)
    D, Dbuf, rc = H.run_layout(A, B, C, M, N, K, offs=(1, 3, 1, 1), lds=(K + 2, K + 5, N + 1, N + 3), **kw)
    assert rc == 0
    ref, _ = H.oracle_full(A, B, C, M, N, K, **kw)
    H.assert_exact(D.numpy(), ref, "fp8 misaligned")
    H.check_canaries(Dbuf, M, N, 1, N + 3)


@pytest.mark.parametrize("dtype", FP8)
def test_streamk_split(dtype):
    M, N, K = 1024, 768, 2080
    A = H.int_matrix((M, K), -4, 4, dtype, 61)
    B = H.int_matrix((N, K), -4, 4, dtype, 62)
    with H.env(GEMM_SK_MIN_ITERS="1", GEMM_VARIANT=None):
        D, rc = H.run_gemm(A, B, None, M, N, K, transB=1, in_dtype=dtype)
    assert rc == 0
    rows, cols = H.sample_positions(M, N, per_block=8, seed=9)
    ref, _ = H.oracle_at(A, B, None, M, N, K, rows, cols, transB=1, in_dtype=dtype)
    H.assert_exact(D.numpy()[rows, cols], ref, "fp8 stream-K")


def test_k_zero_and_ragged_canaries():
    M, N = 70, 88
    C = H.int_matrix((M, N), -50, 50, "f32", 71)
    D, rc = H.run_gemm(None, None, C, M, N, 0, alpha=3.0, beta=2.0, in_dtype="e4m3")
    assert rc == 0
    H.assert_exact(D.numpy(), 2.0 * C.double().numpy(), "fp8 K = 0")
    M, N, K = 129, 257, 65
    A = H.int_matrix((M, K), -8, 8, "e4m3", 72)
    B = H.int_matrix((N, K), -8, 8, "e4m3", 73)
    D, Dbuf, rc = H.run_layout(A, B, None, M, N, K, lds=(80, 80, N, 264), transB=1, in_dtype="e4m3")
    assert rc == 0
    ref, _ = H.oracle_full(A, B, None, M, N, K, transB=1, in_dtype="e4m3")
    H.assert_exact(D.numpy(), ref, "fp8 ragged")
    H.check_canaries(Dbuf, M, N, 0, 264)


def test_noalloc_k_major_and_rejection():
    M, N, K = 264, 200, 192
    A = H.int_matrix((M, K), -8, 8, "e5m2", 81)
    B = H.int_matrix((N, K), -8, 8, "e5m2", 82)
    D, _, rc = H.run_layout(A, B, None, M, N, K, transB=1, in_dtype="e5m2", fn=binding.gemm_noalloc)
    assert rc == 0
    ref, _ = H.oracle_full(A, B, None, M, N, K, transB=1, in_dtype="e5m2")
    H.assert_exact(D.numpy(), ref, "fp8 no-alloc")
    Bt = B.t().contiguous()
    D, _, rc = H.run_layout(A, Bt, None, M, N, K, transB=0, in_dtype="e5m2", fn=binding.gemm_noalloc)
    assert rc == binding.GEMM_ERR_UNSUPPORTED_LAYOUT
    assert torch.isnan(D).all(), "a rejected call wrote D"
