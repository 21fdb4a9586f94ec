"""GPU parity of the whole-stage operand boxes.

The CTA-pair kernel with four epilogue warps, and the narrow one, stage two
64-wide K sub-blocks per pipeline stage.  Their producer fetches each
complete stage of an operand with one TMA box: a 3-D box for a K-major
operand, a 4-D box for an MN-major one.  A partial last stage (K not a
multiple of the stage), and for an MN-major operand whose extent is not a
multiple of 64 the last stage, take one 2-D box per sub-block and per 64-wide
MN chunk, as every stage does with GEMM_STAGE_BOXES=0.  Both forms fill
shared memory with the same image, so on integer inputs both are exact
against the oracle and equal to each other bit for bit.  The shapes below
take each form for A and for B: ragged M, N and K, an odd number of
sub-blocks (the last stage's second sub-block lies past K and reads zeros),
MN extents below and above 64 that are not multiples of 64 (whose last chunk
reads past the row, into values that reach only unstored rows or columns of
D), K shorter than one stage, 8-bit operands, and the block-scaled kernel's
operands.
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


# (M, N, K, transA, transB, in_dtype, out_dtype, integer range), on the pair
# kernel (forced: the size rule would give these small problems narrow
# one-SM tiles) with four epilogue warps: 16-bit D, or f32 D with more than
# four stages (K > 512; > 1024 for 8-bit operands).  Those with K-major B and
# f32 D run on the 224-wide tiles (112 B rows per CTA).
SHAPES = [
    (520, 392, 704, 0, 1, "f16", "f32", 8),     # A, B K-major: 3-D boxes; 11 sub-blocks
    (520, 384, 640, 1, 0, "bf16", "f32", 8),    # A MN-major, M % 64 != 0: 4-D but the last stage; B 4-D
    (512, 448, 576, 1, 0, "f16", "f32", 8),     # A, B MN-major: 4-D boxes; 9 sub-blocks
    (300, 256, 128, 0, 0, "f16", "f16", 2),     # A K-major 3-D, B MN-major 4-D, one stage, f16 D
    (384, 320, 1000, 0, 1, "f16", "f32", 8),    # K % 64 != 0: 3-D boxes, the partial last stage 2-D
    (520, 392, 1000, 0, 0, "f16", "f32", 8),    # ragged K, B MN-major with N % 64 != 0
    (264, 40, 704, 1, 0, "bf16", "f32", 8),     # B MN-major with N < 64: 2-D boxes only
    (300, 200, 100, 0, 1, "f16", "f32", 8),     # K shorter than one stage: 2-D boxes only
    (520, 392, 1152, 0, 1, "e4m3", "f32", 8),   # 8-bit, K-major: 3-D boxes of 128-byte K rows; 9 sub-blocks
    (264, 200, 704, 1, 1, "bf16", "bf16", 2),   # A MN-major 4-D but the last stage (M % 64 != 0), B 3-D
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "%dx%dx%d_t%d%d_%s_%s" % s[:7])
def test_stage_boxes_match_2d_boxes_and_oracle(shape):
    M, N, K, transA, transB, in_dtype, out_dtype, lim = shape
    seed = 7 * M + 3 * N + K + transA + 2 * transB
    A = H.int_matrix((K, M) if transA else (M, K), -lim, lim, in_dtype, seed)
    B = H.int_matrix((N, K) if transB else (K, N), -lim, lim, in_dtype, seed + 1)
    C = H.int_matrix((M, N), -20, 20, out_dtype, seed + 2)
    kw = dict(transA=transA, transB=transB, alpha=1.0, beta=1.0, in_dtype=in_dtype, out_dtype=out_dtype)
    out = []
    for boxes in (None, "0"):
        with H.env(GEMM_PATH="tcgen05", GEMM_VARIANT="pair", GEMM_STAGE_BOXES=boxes):
            D, rc = H.run_gemm(A, B, C, M, N, K, **kw)
        assert rc == 0, boxes
        out.append(D)
    assert torch.equal(out[0], out[1]), "whole-stage boxes and 2-D boxes disagree"
    ref, bound = H.oracle_full(A, B, C, M, N, K, **kw)
    if out_dtype == "f32":
        H.assert_exact(out[0].numpy(), ref, "stage boxes %s" % (shape,))
    else:   # one rounding to the 16-bit D
        H.assert_close(out[0].double().numpy(), ref, bound, out_dtype, "stage boxes %s" % (shape,))


# block-scaled operands (gemm_mx): the same whole-stage operand boxes (packed
# E2M1 through its 16U4_ALIGN16B maps; K = 1000 has a partial last stage),
# scales per sub-block as before
MX_SHAPES = [(640, 520, 1024, "e4m3", 0.0), (264, 448, 640, "e5m2", 1.0), (520, 392, 1000, "e4m3", 1.0),
             (384, 392, 1152, "e2m1", 1.0), (264, 448, 1000, "e5m2", 0.0)]


@pytest.mark.parametrize("shape", MX_SHAPES, ids=lambda s: "%dx%dx%d_%s_b%g" % s)
def test_mx_stage_boxes_match_2d_boxes_and_oracle(shape):
    from tests.test_mx_gpu import fp4_matrix, oracle_mx, run_mx, scales
    M, N, K, dtype, beta = shape
    seed = 11 * M + N + K
    if dtype == "e2m1":   # packed codes, two per byte
        A, B = fp4_matrix(M, K, seed), fp4_matrix(N, K, seed + 1)
    else:
        A = H.int_matrix((M, K), -8, 8, dtype, seed)
        B = H.int_matrix((N, K), -8, 8, dtype, seed + 1)
    C = H.int_matrix((M, N), -100, 100, "f32", seed + 2) if beta else None
    SFA = scales(M, K, 126, 128, seed + 3)
    SFB = scales(N, K, 126, 128, seed + 4)
    kw = dict(beta=beta, in_dtype=dtype)
    out = []
    for boxes in (None, "0"):
        with H.env(GEMM_PATH=None, GEMM_VARIANT="pair", GEMM_STAGE_BOXES=boxes):
            D, rc = run_mx(A, B, C, SFA, SFB, M, N, K, **kw)
        assert rc == 0, boxes
        out.append(D)
    assert torch.equal(out[0], out[1]), "whole-stage boxes and 2-D boxes disagree"
    ref, _ = oracle_mx(A, B, C, SFA, SFB, M, N, K, **kw)
    H.assert_exact(out[0].numpy(), ref, "mx stage boxes %s" % (shape,))
