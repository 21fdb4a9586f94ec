"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Every test here needs a GB300 and the built library; they are marked
``gpu``.  Inputs are seeded; expected values come only from the oracle (or
the stored golden fixture written from it).
"""
import numpy as np
import pytest
import torch

from dense_tensor_core_02_gb300 import binding
from dense_tensor_core_02_gb300.inputs import CASES, CASE_BY_NAME, make_inputs
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

# "pair" / "single" / "narrow": the tcgen05 kernel with 256 x 256 tiles on
# 2 SMs, 128 x 256 or 128 x 64 tiles on one SM (forced even where the size
# rule would pick another); "mma_sync": the warp-level kernel.
VARIANTS = ["pair", "single", "narrow", "mma_sync"]


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    yield
    rc, info = H.poll()
    assert rc == 0, ("device status after the module", rc, info)


@pytest.fixture(params=VARIANTS)
def variant(request):
    if request.param == "mma_sync":
        with H.env(GEMM_PATH="mma_sync", GEMM_VARIANT=None):
            yield request.param
    else:
        with H.env(GEMM_PATH="tcgen05", GEMM_VARIANT=request.param):
            yield request.param


@pytest.fixture(params=["tcgen05", "mma_sync"])
def path(request):
    with H.env(GEMM_PATH=request.param):
        yield request.param


def _golden():
    from tests.test_oracle import _read_golden
    return _read_golden("single_atom_int_16x8x16.txt")


def test_golden_single_atom(variant):
    """TIRx "gemm" page, "Demonstration program": one 16x8x16 atom, bit-exact."""
    g = _golden()
    A = torch.from_numpy(g["A"].astype(np.float32)).half()
    B = torch.from_numpy(g["B"].astype(np.float32)).half()
    D, rc = H.run_gemm(A, B, None, 16, 8, 16)
    assert rc == 0
    H.assert_exact(D.numpy(), g["D"].astype(np.float64), "single atom")


# The test matrix the TIRx gemm guide describes for its numeric test
# (section 六: single tile, one multi-tile dimension, every dimension
# multi-tile, M = 64, a k8 shape, K = 24), restated with concrete shapes.
PAGE_SHAPES = [(16, 8, 16), (32, 8, 16), (16, 16, 16), (16, 8, 32), (64, 8, 16), (32, 16, 48),
               (16, 8, 8), (16, 8, 24), (128, 64, 64)]


@pytest.mark.parametrize("shape", PAGE_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("beta", [0.0, 1.0])
def test_page_matrix_integers_exact(path, shape, dtype, beta):
    M, N, K = shape
    seed = M * 10007 + N * 101 + K + 7 * (dtype == "bf16") + 13 * int(beta)
    A = H.int_matrix((M, K), -8, 8, dtype, seed)
    B = H.int_matrix((K, N), -8, 8, dtype, seed + 1)
    C = H.int_matrix((M, N), -64, 64, "f32", seed + 2) if beta else None
    D, rc = H.run_gemm(A, B, C, M, N, K, beta=beta, in_dtype=dtype)
    assert rc == 0
    ref, _ = H.oracle_full(A, B, C, M, N, K, beta=beta, in_dtype=dtype)
    H.assert_exact(D.numpy(), ref, "page matrix %s %s beta=%s" % (shape, dtype, beta))


@pytest.mark.parametrize("transA", [0, 1])
@pytest.mark.parametrize("transB", [0, 1])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_transpose_forms_integers_exact(variant, transA, transB, dtype):
    M, N, K = 296, 264, 200
    seed = 17 + 4 * transA + 2 * transB + (dtype == "bf16")
    A = H.int_matrix((K, M) if transA else (M, K), -8, 8, dtype, seed)
    B = H.int_matrix((N, K) if transB else (K, N), -8, 8, dtype, seed + 100)
    C = H.int_matrix((M, N), -100, 100, "f32", seed + 200)
    D, rc = H.run_gemm(A, B, C, M, N, K, transA=transA, transB=transB, beta=1.0, in_dtype=dtype)
    assert rc == 0
    ref, _ = H.oracle_full(A, B, C, M, N, K, transA=transA, transB=transB, beta=1.0, in_dtype=dtype)
    H.assert_exact(D.numpy(), ref, "transpose %d%d %s" % (transA, transB, dtype))


@pytest.mark.parametrize("transA", [0, 1])
@pytest.mark.parametrize("transB", [0, 1])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_transpose_forms_random(transA, transB, dtype):
    M, N, K = 392, 520, 328
    seed = 41 + 4 * transA + 2 * transB + (dtype == "bf16")
    A = H.normal_matrix((K, M) if transA else (M, K), dtype, seed)
    B = H.normal_matrix((N, K) if transB else (K, N), dtype, seed + 1)
    C = H.normal_matrix((M, N), "f32", seed + 2)
    kw = dict(transA=transA, transB=transB, alpha=1.5, beta=0.5, in_dtype=dtype)
    D, rc = H.run_gemm(A, B, C, M, N, K, **kw)
    assert rc == 0
    ref, bound = H.oracle_full(A, B, C, M, N, K, **kw)
    H.assert_close(D.numpy(), ref, bound, what="random transpose %d%d %s" % (transA, transB, dtype))


SMALL_CASES = [c for c in CASES if not c.mx and c.M * c.N * c.K <= 1024 ** 3]
LARGE_CASES = [c for c in CASES if not c.mx and c.M * c.N * c.K > 1024 ** 3]


@pytest.mark.parametrize("case", SMALL_CASES, ids=lambda c: c.name)
def test_workload_full(case):
    """Every element of the small workloads against the oracle."""
    A, B, C = make_inputs(case)
    kw = dict(transA=case.transA, transB=case.transB, alpha=case.alpha, beta=case.beta,
              in_dtype=case.in_dtype, out_dtype=case.out_dtype)
    D, rc = H.run_gemm(A, B, C, case.M, case.N, case.K, **kw)
    assert rc == 0
    ref, bound = H.oracle_full(A, B, C, case.M, case.N, case.K, **kw)
    H.assert_close(D.numpy(), ref, bound, case.out_dtype, case.name)


@pytest.mark.parametrize("case", LARGE_CASES, ids=lambda c: c.name)
def test_workload_sampled(case):
    """The large workloads at full size, in the benchmark's launch
    configuration: every 128 x 128 output block sampled (corners plus random
    points) and the last row and column, against the oracle."""
    A, B, C = make_inputs(case)
    kw = dict(transA=case.transA, transB=case.transB, alpha=case.alpha, beta=case.beta,
              in_dtype=case.in_dtype, out_dtype=case.out_dtype)
    D, rc = H.run_gemm(A, B, C, case.M, case.N, case.K, **kw)
    assert rc == 0
    assert not torch.isnan(D).any(), "unwritten (NaN-filled) output elements"
    rows, cols = H.sample_positions(case.M, case.N, per_block=4, seed=case.seed)
    ref, bound = H.oracle_at(A, B, C, case.M, case.N, case.K, rows, cols, **kw)
    H.assert_close(D.numpy()[rows, cols], ref, bound, case.out_dtype, case.name)


EDGE_SHAPES = [(1, 1, 1), (255, 257, 17), (129, 513, 65), (16, 8, 24), (1000, 1000, 1000), (7, 300, 4000),
               (300, 8, 72), (257, 255, 1), (33, 40, 8)]


@pytest.mark.parametrize("out_dtype", ["f32", "f16"])
@pytest.mark.parametrize("shape", EDGE_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_ragged_edges_with_canaries(variant, shape, out_dtype):
    """D sits inside a larger NaN-filled buffer (extra rows and a padded
    leading dimension); everything outside D must stay untouched, including
    the row padding right after the last column."""
    M, N, K = shape
    dev = torch.device("cuda", 0)
    pad_rows, ldd = 3, ((N + 7) // 8) * 8 + 8
    A = H.int_matrix((M, ((K + 7) // 8) * 8), -8, 8, "f16", M + N + K)   # padded lda
    B = H.int_matrix((K, ((N + 7) // 8) * 8 + 8), -8, 8, "f16", M * N + K)  # padded ldb
    buf = torch.full((M + 2 * pad_rows, ldd), float("nan"), dtype=H.TORCH[out_dtype], device=dev)
    D = buf[pad_rows:pad_rows + M]
    Ad, Bd = A.to(dev), B.to(dev)
    rc = binding.gemm(D, Ad, Bd, None, M, N, K, Ad.stride(0), Bd.stride(0), N, ldd, 0, 0, 1.0, 0.0, 0,
                      H.CODE[out_dtype], None)
    assert rc == 0
    torch.cuda.synchronize()
    host = buf.float().cpu().numpy()
    ref, bound = H.oracle_full(A[:, :K].contiguous(), B[:, :N].contiguous(), None, M, N, K)
    if out_dtype == "f32":
        H.assert_exact(host[pad_rows:pad_rows + M, :N], ref, "ragged %s" % (shape,))
    else:
        H.assert_close(host[pad_rows:pad_rows + M, :N], ref, bound, out_dtype, "ragged %s" % (shape,))
    assert np.isnan(host[:pad_rows]).all() and np.isnan(host[pad_rows + M:]).all(), "rows outside D written"
    assert np.isnan(host[:, N:]).all(), "columns beyond N written"


def test_in_place_c_is_d(variant):
    M, N, K = 384, 320, 256
    A = H.normal_matrix((M, K), "f16", 5)
    B = H.normal_matrix((K, N), "f16", 6)
    C = H.normal_matrix((M, N), "f32", 7)
    dev = torch.device("cuda", 0)
    Ad, Bd, CD = A.to(dev), B.to(dev), C.to(dev)
    rc = binding.gemm(CD, Ad, Bd, CD, M, N, K, K, N, N, N, 0, 0, -0.5, 2.0, 0, 2, None)
    assert rc == 0
    torch.cuda.synchronize()
    ref, bound = H.oracle_full(A, B, C, M, N, K, alpha=-0.5, beta=2.0)
    H.assert_close(CD.cpu().numpy(), ref, bound, what="in place")


def test_beta_zero_never_reads_c():
    M, N, K = 256, 256, 128
    A = H.normal_matrix((M, K), "bf16", 8)
    B = H.normal_matrix((K, N), "bf16", 9)
    C = torch.full((M, N), float("nan"))
    D, rc = H.run_gemm(A, B, C, M, N, K, beta=0.0, in_dtype="bf16")
    assert rc == 0
    assert torch.isfinite(D).all()
    ref, bound = H.oracle_full(A, B, None, M, N, K, in_dtype="bf16")
    H.assert_close(D.numpy(), ref, bound, what="beta 0, NaN C")


@pytest.mark.parametrize("beta", [0.0, 1.0, -2.5])
@pytest.mark.parametrize("out_dtype", ["f32", "f16", "bf16"])
def test_k_zero(beta, out_dtype):
    M, N = 70, 88
    C = H.int_matrix((M, N), -50, 50, out_dtype, 3) if beta else None
    D, rc = H.run_gemm(None, None, C, M, N, 0, alpha=3.0, beta=beta, out_dtype=out_dtype)
    assert rc == 0
    ref = (beta * C.double().numpy()) if beta else np.zeros((M, N))
    H.assert_close(D.double().numpy(), ref, np.abs(ref), out_dtype, "K = 0")


@pytest.mark.parametrize("out_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("beta", [0.0, 0.75])
def test_16bit_outputs(variant, out_dtype, beta):
    M, N, K = 520, 392, 264
    A = H.normal_matrix((M, K), "f16", 11, std=0.25)
    B = H.normal_matrix((K, N), "f16", 12, std=0.25)
    C = H.normal_matrix((M, N), out_dtype, 13) if beta else None
    kw = dict(alpha=1.25, beta=beta, out_dtype=out_dtype)
    D, rc = H.run_gemm(A, B, C, M, N, K, **kw)
    assert rc == 0
    ref, bound = H.oracle_full(A, B, C, M, N, K, **kw)
    H.assert_close(D.double().numpy(), ref, bound, out_dtype, "out %s" % out_dtype)


@pytest.mark.parametrize("alpha,beta", [(-0.75, 2.5), (0.0, 1.0), (2.0, -1.0)])
def test_general_alpha_beta(variant, alpha, beta):
    M, N, K = 640, 768, 1040
    A = H.normal_matrix((M, K), "bf16", 21)
    B = H.normal_matrix((N, K), "bf16", 22)
    C = H.normal_matrix((M, N), "f32", 23)
    kw = dict(transB=1, alpha=alpha, beta=beta, in_dtype="bf16")
    D, rc = H.run_gemm(A, B, C, M, N, K, **kw)
    assert rc == 0
    ref, bound = H.oracle_full(A, B, C, M, N, K, **kw)
    H.assert_close(D.numpy(), ref, bound, what="alpha=%s beta=%s" % (alpha, beta))


def test_many_tiles_per_cta(variant):
    """More tiles than CTAs: each persistent CTA walks several tiles and
    both TMEM accumulators."""
    M, N, K = 2048, 4096, 192
    A = H.int_matrix((M, K), -4, 4, "f16", 31)
    B = H.int_matrix((K, N), -4, 4, "f16", 32)
    D, rc = H.run_gemm(A, B, None, M, N, K)
    assert rc == 0
    rows, cols = H.sample_positions(M, N, per_block=16, seed=3)
    ref, _ = H.oracle_at(A, B, None, M, N, K, rows, cols)
    H.assert_exact(D.numpy()[rows, cols], ref, "many tiles")


def test_non_default_stream():
    M, N, K = 512, 256, 320
    A = H.normal_matrix((M, K), "f16", 51)
    B = H.normal_matrix((K, N), "f16", 52)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        D, rc = H.run_gemm(A, B, None, M, N, K, stream=s)
    assert rc == 0
    ref, bound = H.oracle_full(A, B, None, M, N, K)
    H.assert_close(D.numpy(), ref, bound, what="side stream")


def test_default_stream_argument_is_torchs_current_stream():
    """stream=None means torch's current stream, also inside a stream context:
    the call is ordered after work queued there and before work queued later."""
    from dense_tensor_core_02_gb300.binding import _stream
    assert _stream(None) == torch.cuda.current_stream().cuda_stream
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        assert _stream(None) == s.cuda_stream != torch.cuda.default_stream().cuda_stream
        M, N, K = 384, 320, 256
        dev = torch.device("cuda", 0)
        A = H.int_matrix((M, K), -4, 4, "f16", 53).to(dev)
        B = H.int_matrix((K, N), -4, 4, "f16", 54).to(dev)
        torch.cuda._sleep(1000000)   # the call must wait for this on s
        D = torch.full((M, N), float("nan"), device=dev)
        assert binding.gemm(D, A, B, None, M, N, K, K, N, N, N, 0, 0, 1.0, 0.0, 0, 2) == 0
        out = D.clone()   # queued on s after the product
    torch.cuda.synchronize()
    ref, _ = H.oracle_full(A.cpu(), B.cpu(), None, M, N, K)
    H.assert_exact(out.cpu().numpy(), ref, "stream=None inside a stream context")
    assert _stream(None) == torch.cuda.current_stream().cuda_stream


def test_repeatable_bitwise():
    """The same call twice gives the same bits (fixed accumulation order)."""
    case = CASE_BY_NAME["gemm_512_f16_alpha1.5_beta0.5"]
    A, B, C = make_inputs(case)
    kw = dict(alpha=case.alpha, beta=case.beta)
    D1, _ = H.run_gemm(A, B, C, case.M, case.N, case.K, **kw)
    D2, _ = H.run_gemm(A, B, C, case.M, case.N, case.K, **kw)
    assert torch.equal(D1, D2)


def test_wait_bound_reports_and_recovers():
    """A pipeline stage that is never filled (test hook) makes the MMA's
    wait run out: the kernel unwinds, the status block says so, and the next
    call on the same context is clean and correct."""
    M, N, K = 256, 256, 512
    A = H.int_matrix((M, K), -4, 4, "f16", 61)
    B = H.int_matrix((K, N), -4, 4, "f16", 62)
    assert H.poll()[0] == 0
    with H.env(GEMM_TEST_SKIP_FIRST_STAGE="1", GEMM_WAIT_TIMEOUT_NS="300000000", GEMM_PATH="tcgen05"):
        _, rc = H.run_gemm(A, B, None, M, N, K)
    assert rc == 0
    status, info = H.poll()
    assert status == binding.GEMM_ERR_DEVICE_TIMEOUT, (status, info)
    assert info[0] == binding.GEMM_ERR_DEVICE_TIMEOUT and info[2] in (1, 2, 3, 4, 5, 6)
    assert H.poll()[0] == 0          # cleared by the first poll
    D, rc = H.run_gemm(A, B, None, M, N, K)
    assert rc == 0 and H.poll()[0] == 0
    ref, _ = H.oracle_full(A, B, None, M, N, K)
    H.assert_exact(D.numpy(), ref, "after recovery")


def test_rejection_leaves_d_untouched():
    dev = torch.device("cuda", 0)
    D = torch.full((64, 64), 7.0, device=dev)
    A = torch.zeros((64, 64), dtype=torch.float16, device=dev)
    rc = binding.gemm(D, A, A, None, 64, 64, 64, 63, 64, 64, 64, 0, 0, 1.0, 0.0, 0, 2, None)
    assert rc == -1
    torch.cuda.synchronize()
    assert (D == 7.0).all()


def test_arch_is_sm103():
    major, minor = torch.cuda.get_device_capability(0)
    assert (major, minor) == (10, 3)



@pytest.mark.parametrize("sms", [100, 38, 2])
def test_max_sms_limits_the_grid_and_stays_exact(sms):
    """GEMM_MAX_SMS plans the persistent grid for fewer SMs (more tiles per
    CTA, other stream-K splits); the result is the oracle's bit for bit on
    integer inputs."""
    M, N, K = 1280, 1536, 1152
    A = H.int_matrix((M, K), -4, 4, "f16", 301)
    B = H.int_matrix((K, N), -4, 4, "f16", 302)
    C = H.int_matrix((M, N), -50, 50, "f32", 303)
    with H.env(GEMM_MAX_SMS=str(sms)):
        plan = binding.gemm_plan(M, N, K, sms)
        assert plan["grid"] <= sms
        D, rc = H.run_gemm(A, B, C, M, N, K, beta=1.0)
    assert rc == 0 and H.poll()[0] == 0
    want, _ = H.oracle_full(A, B, C, M, N, K, beta=1.0)
    H.assert_exact(D.numpy(), want, "GEMM_MAX_SMS=%d" % sms)
