"""GPU parity of the warp-level mma.sync kernel against the CPU oracle.

This kernel takes any element-aligned layout as it is -- operand or output
addresses and row strides that are not 16-byte multiples, which TMA cannot
describe -- and tiny problems.  It runs every layout that gemm_noalloc()
receives off the 16-byte grid, and gemm()'s small ones (larger ones are
repacked for the tcgen05 kernel; see test_repack_gpu.py).  The tests here
force it (GEMM_PATH=mma_sync) on those layouts and on the workloads the
tcgen05 kernel is tested on.  The route has two kernels, the tiled one and,
for problems with M*N*K <= GEMM_SYNC_ATOM_MAX_WORK, the one-warp-per-16x8-
block atom kernel; the layout tests run each of them on every layout by
setting that bound to 0 or beyond the problem.  The shared parity cases (golden atom, page
test matrix, transposes, ragged canaries, in place, 16-bit outputs,
alpha/beta) run on it through the "mma_sync" variant of the main GPU test
module.
"""
import numpy as np
import pytest
import torch

from dense_tensor_core_02_gb300 import binding
from dense_tensor_core_02_gb300.inputs import CASES, make_inputs
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


# (M, N, K, element offsets of A, B, C, D, strides lda, ldb, ldc, ldd or None)
ODD_LAYOUTS = [
    (300, 200, 1001, (0, 0, 0, 0), None),                  # K = 1001: lda = 1001 (2002 bytes)
    (129, 77, 65, (1, 3, 1, 1), None),                     # every base off the 16-byte grid
    (64, 64, 64, (0, 0, 0, 0), (65, 67, 66, 69)),          # odd strides, aligned bases
    (257, 130, 33, (5, 0, 2, 3), (41, 133, 131, 135)),
    (1, 1, 7, (1, 1, 1, 1), None),
    (17, 9, 3, (0, 1, 0, 1), None),
    (520, 392, 264, (2, 0, 0, 0), None),                   # only A off the grid
]


# GEMM_SYNC_ATOM_MAX_WORK for each of the route's two kernels
SYNC_KERNELS = {"tiled": "0", "atom": str(1 << 62)}


@pytest.mark.parametrize("kernel", list(SYNC_KERNELS))
@pytest.mark.parametrize("transA", [0, 1])
@pytest.mark.parametrize("transB", [0, 1])
@pytest.mark.parametrize("layout", ODD_LAYOUTS, ids=lambda l: "%dx%dx%d_o%s" % (l[0], l[1], l[2],
                                                                               "".join(map(str, l[3]))))
def test_odd_layouts_integers_exact(layout, transA, transB, kernel):
    """Layouts TMA cannot take; integer-valued inputs, so the fp32 result is
    exact."""
    M, N, K, offs, lds = layout
    if lds is not None:
        ra, ca = (K, M) if transA else (M, K)
        rb, cb = (N, K) if transB else (K, N)
        lds = (max(lds[0], ca), max(lds[1], cb), lds[2], lds[3])
    seed = M * 31 + N * 7 + K + 2 * transA + transB
    A = H.int_matrix((K, M) if transA else (M, K), -8, 8, "f16", seed)
    B = H.int_matrix((N, K) if transB else (K, N), -8, 8, "f16", seed + 1)
    C = H.int_matrix((M, N), -100, 100, "f32", seed + 2)
    with H.env(GEMM_PATH="mma_sync", GEMM_SYNC_ATOM_MAX_WORK=SYNC_KERNELS[kernel]):
        D, Dbuf, rc = H.run_layout(A, B, C, M, N, K, offs=offs, lds=lds, transA=transA, transB=transB, beta=1.0)
    assert rc == 0
    ref, _ = H.oracle_full(A, B, C, M, N, K, transA=transA, transB=transB, beta=1.0)
    H.assert_exact(D.numpy(), ref, "odd layout %s" % (layout,))
    ldd = lds[3] if lds else N
    H.check_canaries(Dbuf, M, N, offs[3], ldd)


@pytest.mark.parametrize("kernel", list(SYNC_KERNELS))
@pytest.mark.parametrize("in_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("out_dtype", ["f32", "f16", "bf16"])
def test_odd_layouts_random(in_dtype, out_dtype, kernel):
    M, N, K = 333, 250, 517
    seed = 7 + 3 * (in_dtype == "bf16") + ["f32", "f16", "bf16"].index(out_dtype)
    A = H.normal_matrix((K, M), in_dtype, seed)
    B = H.normal_matrix((K, N), in_dtype, seed + 1)
    C = H.normal_matrix((M, N), out_dtype, seed + 2)
    kw = dict(transA=1, alpha=-1.25, beta=0.5, in_dtype=in_dtype, out_dtype=out_dtype)
    with H.env(GEMM_PATH="mma_sync", GEMM_SYNC_ATOM_MAX_WORK=SYNC_KERNELS[kernel]):
        D, Dbuf, rc = H.run_layout(A, B, C, M, N, K, offs=(1, 1, 1, 1), lds=(M + 1, N + 3, N + 1, N + 5), **kw)
    assert rc == 0
    ref, bound = H.oracle_full(A, B, C, M, N, K, **kw)
    H.assert_close(D.double().numpy(), ref, bound, out_dtype, "odd random %s->%s" % (in_dtype, out_dtype))
    H.check_canaries(Dbuf, M, N, 1, N + 5)


def test_in_place_odd_layout():
    """C == D (same pointer, same stride) off the 16-byte grid."""
    M, N, K = 130, 90, 77
    A = H.normal_matrix((M, K), "bf16", 91)
    B = H.normal_matrix((N, K), "bf16", 92)
    C = H.normal_matrix((M, N), "f32", 93)
    dev = torch.device("cuda", 0)
    _, Av = H.strided(A, 1, K, "bf16")
    _, Bv = H.strided(B, 1, K, "bf16")
    _, CD = H.strided(C, 3, N + 1, "f32")
    with H.env(GEMM_PATH="mma_sync"):
        rc = binding.gemm(CD, Av, Bv, CD, M, N, K, K, K, N + 1, N + 1, 0, 1, 0.75, -1.5, 1, 2, None)
    assert rc == 0
    torch.cuda.synchronize()
    ref, bound = H.oracle_full(A, B, C, M, N, K, transB=1, alpha=0.75, beta=-1.5, in_dtype="bf16")
    H.assert_close(CD.cpu().numpy(), ref, bound, what="in place, odd layout")


def test_beta_zero_never_reads_c_odd_layout():
    M, N, K = 40, 24, 9
    A = H.normal_matrix((M, K), "f16", 94)
    B = H.normal_matrix((K, N), "f16", 95)
    C = torch.full((M, N), float("nan"))
    with H.env(GEMM_PATH="mma_sync"):
        D, _, rc = H.run_layout(A, B, C, M, N, K, offs=(1, 1, 1, 1), beta=0.0)
    assert rc == 0 and torch.isfinite(D).all()
    ref, bound = H.oracle_full(A, B, None, M, N, K)
    H.assert_close(D.numpy(), ref, bound, what="beta 0, NaN C, odd layout")


TINY = [(1, 1, 1), (16, 8, 16), (8, 16, 8), (63, 65, 17), (64, 64, 64), (5, 300, 3), (100, 7, 250)]


@pytest.mark.parametrize("shape", TINY, ids=lambda s: "x".join(map(str, s)))
def test_tiny_problems_default_routing(shape):
    """Tiny problems through the default routing (those with K <= 32 take
    the mma.sync route's atom kernel, the rest the tcgen05 kernel): exact on
    integers."""
    M, N, K = shape
    A = H.int_matrix((M, K), -8, 8, "bf16", M + N + K)
    B = H.int_matrix((N, K), -8, 8, "bf16", M * N + K)
    with H.env(GEMM_PATH=None, GEMM_SYNC_MAX_WORK=None):
        D, rc = H.run_gemm(A, B, None, M, N, K, transB=1, in_dtype="bf16", alpha=2.0)
    assert rc == 0
    ref, _ = H.oracle_full(A, B, None, M, N, K, transB=1, in_dtype="bf16", alpha=2.0)
    H.assert_exact(D.numpy(), ref, "tiny %s" % (shape,))


# (M, N, K, transA, transB, in_dtype, out_dtype, beta): tiny problems, each
# kernel of the route forced; K remainders of 0, 1..8 (the k8 atom) and 9..15
TINY_FORCED = [(16, 8, 16, 0, 0, "f16", "f32", 0.0), (1, 1, 1, 1, 1, "bf16", "f16", 1.0),
               (15, 9, 8, 1, 0, "f16", "bf16", -0.5), (33, 17, 24, 0, 1, "bf16", "f32", 2.0),
               (7, 40, 41, 1, 1, "f16", "f32", 1.0), (48, 24, 9, 0, 0, "bf16", "bf16", 0.0)]


@pytest.mark.parametrize("kernel", list(SYNC_KERNELS))
@pytest.mark.parametrize("shape", TINY_FORCED, ids=lambda s: "%dx%dx%d_t%d%d_%s_%s_b%g" % s)
def test_tiny_problems_each_sync_kernel(shape, kernel):
    """Both kernels of the mma.sync route on tiny problems, every transpose
    pair, 16-bit and fp32 outputs, with and without C: exact on integers."""
    M, N, K, transA, transB, in_dtype, out_dtype, beta = shape
    seed = 1000 + M * 7 + N * 3 + K
    A = H.int_matrix((K, M) if transA else (M, K), -8, 8, in_dtype, seed)
    B = H.int_matrix((N, K) if transB else (K, N), -8, 8, in_dtype, seed + 1)
    C = H.int_matrix((M, N), -50, 50, out_dtype, seed + 2) if beta else None
    kw = dict(transA=transA, transB=transB, alpha=1.0, beta=beta, in_dtype=in_dtype, out_dtype=out_dtype)
    with H.env(GEMM_PATH="mma_sync", GEMM_SYNC_ATOM_MAX_WORK=SYNC_KERNELS[kernel]):
        D, rc = H.run_gemm(A, B, C, M, N, K, **kw)
    assert rc == 0
    ref, bound = H.oracle_full(A, B, C, M, N, K, **kw)
    if out_dtype == "f32":
        H.assert_exact(D.numpy(), ref, "tiny %s on the %s kernel" % (shape, kernel))
    else:
        H.assert_close(D.double().numpy(), ref, bound, out_dtype, "tiny %s on the %s kernel" % (shape, kernel))


SMALL_CASES = [c for c in CASES if not c.mx and c.M * c.N * c.K <= 1024 ** 3]


@pytest.mark.parametrize("case", SMALL_CASES, ids=lambda c: c.name)
def test_workloads_forced_mma_sync(case):
    """The small workloads, every element, on the mma.sync kernel."""
    A, B, C = make_inputs(case)
    kw = dict(transA=case.transA, transB=case.transB, alpha=case.alpha, beta=case.beta,
              in_dtype=case.in_dtype, out_dtype=case.out_dtype)
    with H.env(GEMM_PATH="mma_sync"):
        D, rc = H.run_gemm(A, B, C, case.M, case.N, case.K, **kw)
    assert rc == 0
    ref, bound = H.oracle_full(A, B, C, case.M, case.N, case.K, **kw)
    H.assert_close(D.numpy(), ref, bound, case.out_dtype, case.name)


def test_large_odd_stride_sampled():
    """A large problem whose K (4097) keeps it off TMA, on this kernel:
    sampled positions in every 128 x 128 block against the oracle."""
    M, N, K = 2048, 1536, 4097
    A = H.normal_matrix((M, K), "f16", 101)
    B = H.normal_matrix((N, K), "f16", 102)
    with H.env(GEMM_PATH="mma_sync"):
        D, rc = H.run_gemm(A, B, None, M, N, K, transB=1)
    assert rc == 0
    assert not torch.isnan(D).any()
    rows, cols = H.sample_positions(M, N, per_block=4, seed=5)
    ref, bound = H.oracle_at(A, B, None, M, N, K, rows, cols, transB=1)
    H.assert_close(D.numpy()[rows, cols], ref, bound, what="large odd stride")


def test_paths_agree_on_integers():
    """On integer-valued inputs both kernels are exact, so they agree bit for bit."""
    M, N, K = 264, 200, 136
    A = H.int_matrix((M, K), -8, 8, "f16", 111)
    B = H.int_matrix((K, N), -8, 8, "f16", 112)
    C = H.int_matrix((M, N), -50, 50, "f32", 113)
    out = []
    for path in ("tcgen05", "mma_sync"):
        with H.env(GEMM_PATH=path):
            D, rc = H.run_gemm(A, B, C, M, N, K, beta=-1.0)
        assert rc == 0
        out.append(D)
    assert torch.equal(out[0], out[1])
