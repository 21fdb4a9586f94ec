"""GPU parity of gemm() on layouts TMA cannot describe, through the repacking
route: operands whose address or row stride is off the 16-byte grid are
copied into aligned workspace rows, a misaligned D is computed in workspace
and copied back, a misaligned C is copied into the D the tcgen05 kernel then
updates in place.  GEMM_REPACK_MIN_WORK=0 sends every such call that way, so
small shapes exercise it too; one large shape takes it through the default
routing.  Canary bands check that nothing outside D is written.
"""
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
    rc, info = H.poll()
    assert rc == 0, ("device status after the module", rc, info)


# (M, N, K, element offsets of A, B, C, D, strides lda, ldb, ldc, ldd or None)
LAYOUTS = [
    (300, 200, 1001, (0, 0, 0, 0), None),                  # K = 1001: A (and B^T) rows off the grid
    (264, 136, 128, (1, 0, 0, 0), None),                   # only A's base
    (264, 136, 128, (0, 3, 0, 0), None),                   # only B's base
    (264, 136, 128, (0, 0, 2, 0), None),                   # only C's base: copied into D
    (264, 136, 128, (0, 0, 0, 1), None),                   # only D's base: computed in workspace
    (257, 130, 33, (5, 0, 2, 3), (41, 133, 131, 135)),     # everything off the grid
    (64, 64, 64, (0, 0, 0, 0), (65, 67, 66, 69)),          # odd strides, aligned bases
    (520, 392, 264, (2, 1, 1, 3), None),
]


def _lds(layout, transA, transB):
    M, N, K, _, lds = layout
    if lds is None:
        return None
    ca = M if transA else K
    cb = K if transB else N
    return (max(lds[0], ca), max(lds[1], cb), lds[2], lds[3])


@pytest.mark.parametrize("transA", [0, 1])
@pytest.mark.parametrize("transB", [0, 1])
@pytest.mark.parametrize("layout", LAYOUTS, ids=lambda l: "%dx%dx%d_o%s%s" % (
    l[0], l[1], l[2], "".join(map(str, l[3])), "_ld" if l[4] else ""))
def test_repacked_integers_exact(layout, transA, transB):
    M, N, K, offs, _ = layout
    lds = _lds(layout, transA, transB)
    seed = 3 * M + 5 * N + K + 2 * transA + transB
    A = H.int_matrix((K, M) if transA else (M, K), -8, 8, "bf16", seed)
    B = H.int_matrix((N, K) if transB else (K, N), -8, 8, "bf16", seed + 1)
    C = H.int_matrix((M, N), -100, 100, "f32", seed + 2)
    kw = dict(transA=transA, transB=transB, beta=1.0, in_dtype="bf16")
    with H.env(GEMM_PATH=None, GEMM_REPACK_MIN_WORK="0"):
        D, Dbuf, rc = H.run_layout(A, B, C, M, N, K, offs=offs, lds=lds, **kw)
    assert rc == 0
    ref, _ = H.oracle_full(A, B, C, M, N, K, **kw)
    H.assert_exact(D.numpy(), ref, "repacked %s" % (layout,))
    H.check_canaries(Dbuf, M, N, offs[3], lds[3] if lds else N)


@pytest.mark.parametrize("out_dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("beta", [0.0, -0.5])
def test_repacked_random(out_dtype, beta):
    M, N, K = 333, 250, 517
    seed = 71 + ["f32", "f16", "bf16"].index(out_dtype) + 3 * int(beta != 0)
    A = H.normal_matrix((M, K), "f16", seed)
    B = H.normal_matrix((K, N), "f16", seed + 1)
    C = H.normal_matrix((M, N), out_dtype, seed + 2) if beta else None
    kw = dict(alpha=1.25, beta=beta, out_dtype=out_dtype)
    with H.env(GEMM_PATH=None, GEMM_REPACK_MIN_WORK="0"):
        D, Dbuf, rc = H.run_layout(A, B, C, M, N, K, offs=(1, 1, 1, 1), lds=(K + 1, N + 3, N + 1, N + 5), **kw)
    assert rc == 0
    ref, bound = H.oracle_full(A, B, C, M, N, K, **kw)
    H.assert_close(D.double().numpy(), ref, bound, out_dtype, "repacked random %s" % out_dtype)
    H.check_canaries(Dbuf, M, N, 1, N + 5)


@pytest.mark.parametrize("d_off", [0, 1])
def test_repacked_in_place(d_off):
    """C == D (same pointer and stride): aligned D with odd operands, and a
    misaligned D computed in workspace from its own old values."""
    M, N, K = 130, 90, 77
    A = H.normal_matrix((M, K), "bf16", 91)
    B = H.normal_matrix((N, K), "bf16", 92)
    C = H.normal_matrix((M, N), "f32", 93)
    _, Av = H.strided(A, 1, K, "bf16")
    _, Bv = H.strided(B, 1, K, "bf16")
    ldd = 96 if d_off == 0 else N + 1
    _, CD = H.strided(C, d_off, ldd, "f32")
    with H.env(GEMM_PATH=None, GEMM_REPACK_MIN_WORK="0"):
        rc = binding.gemm(CD, Av, Bv, CD, M, N, K, K, K, ldd, ldd, 0, 1, 0.75, -1.5, 1, 2, None)
    assert rc == 0
    torch.cuda.synchronize()
    ref, bound = H.oracle_full(A, B, C, M, N, K, transB=1, alpha=0.75, beta=-1.5, in_dtype="bf16")
    H.assert_close(CD.cpu().numpy(), ref, bound, what="repacked in place")


def test_repacked_matches_mma_sync_bitwise_on_integers():
    M, N, K = 200, 136, 101
    A = H.int_matrix((M, K), -8, 8, "f16", 121)
    B = H.int_matrix((N, K), -8, 8, "f16", 122)
    C = H.int_matrix((M, N), -50, 50, "f32", 123)
    out = []
    for path, work in (("mma_sync", None), (None, "0")):
        with H.env(GEMM_PATH=path, GEMM_REPACK_MIN_WORK=work):
            D, _, rc = H.run_layout(A, B, C, M, N, K, offs=(1, 1, 1, 1), transB=1, beta=1.0)
        assert rc == 0
        out.append(D)
    assert torch.equal(out[0], out[1])


def test_large_odd_stride_default_routing():
    """4096 x 2048 x 4095 with every row stride odd: repacked by default;
    sampled positions in every 128 x 128 block against the oracle."""
    M, N, K = 4096, 2048, 4095
    A = H.normal_matrix((M, K), "f16", 131)
    B = H.normal_matrix((K, N), "f16", 132)
    C = H.normal_matrix((M, N), "f32", 133)
    kw = dict(alpha=1.0, beta=1.0)
    with H.env(GEMM_PATH=None, GEMM_REPACK_MIN_WORK=None):
        D, _, rc = H.run_layout(A, B, C, M, N, K, offs=(1, 1, 1, 1), lds=(K, N + 1, N + 1, N + 3), **kw)
    assert rc == 0
    assert not torch.isnan(D).any()
    rows, cols = H.sample_positions(M, N, per_block=4, seed=7)
    ref, bound = H.oracle_at(A, B, C, M, N, K, rows, cols, **kw)
    H.assert_close(D.numpy()[rows, cols], ref, bound, what="large repacked")
