"""GPU parity of gemm_host(): A, B, C and D in host memory, staged and
pipelined over row panels of D by the library, against the CPU oracle.
Pinned and pageable host buffers, all transposes, beta = 0 / 1 / general,
16-bit and 8-bit operands, padded host strides, several panels, and
back-to-back calls on one stream with different inputs.
"""
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
    rc, info = H.poll()
    assert rc == 0, ("device status after the module", rc, info)


def _host(x, pinned, pad=0):
    """A host copy of x with `pad` extra columns; returns (tensor view, ld)."""
    rows, cols = x.shape
    buf = torch.empty((rows, cols + pad), dtype=x.dtype)
    if pinned:
        buf = buf.pin_memory()
    buf[:, :cols] = x
    return buf[:, :cols], cols + pad


def _run_host(A, B, C, M, N, K, *, pinned=True, pad=0, transA=0, transB=0, alpha=1.0, beta=0.0,
              in_dtype="f16", out_dtype="f32", stream=None):
    hA, lda = _host(A, pinned, pad) if A is not None else (None, 0)
    hB, ldb = _host(B, pinned, pad) if B is not None else (None, 0)
    hC, ldc = _host(C, pinned, pad) if C is not None else (None, N)
    hD, ldd = _host(torch.full((M, N), float("nan"), dtype=H.TORCH[out_dtype]), pinned, pad)
    rc = binding.gemm_host(hD, hA, hB, hC, M, N, K, lda, ldb, ldc, ldd, transA, transB, alpha, beta,
                           H.CODE[in_dtype], H.CODE[out_dtype], stream)
    torch.cuda.synchronize()
    return hD.clone(), rc


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("transA", [0, 1])
@pytest.mark.parametrize("transB", [0, 1])
def test_integers_exact(pinned, transA, transB):
    M, N, K = 2600, 520, 328     # 3 row panels, the last one ragged
    seed = 5 + 2 * transA + transB + 4 * pinned
    A = H.int_matrix((K, M) if transA else (M, K), -8, 8, "f16", seed)
    B = H.int_matrix((N, K) if transB else (K, N), -8, 8, "f16", seed + 1)
    C = H.int_matrix((M, N), -50, 50, "f32", seed + 2)
    kw = dict(transA=transA, transB=transB, beta=1.0)
    D, rc = _run_host(A, B, C, M, N, K, pinned=pinned, pad=3, **kw)
    assert rc == 0
    ref, _ = H.oracle_full(A, B, C, M, N, K, **kw)
    H.assert_exact(D.numpy(), ref, "gemm_host trans=%d%d pinned=%s" % (transA, transB, pinned))


@pytest.mark.parametrize("in_dtype,out_dtype", [("bf16", "f32"), ("f16", "bf16"), ("e4m3", "f32"),
                                                ("e5m2", "f16")])
def test_random_general_alpha_beta(in_dtype, out_dtype):
    M, N, K = 1500, 392, 520
    seed = 21 + ["bf16", "f16", "e4m3", "e5m2"].index(in_dtype)
    transB = 1 if in_dtype in ("e4m3", "e5m2") else 0
    A = H.normal_matrix((M, K), in_dtype, seed)
    B = H.normal_matrix((N, K) if transB else (K, N), in_dtype, seed + 1)
    C = H.normal_matrix((M, N), out_dtype, seed + 2)
    kw = dict(transB=transB, alpha=-0.75, beta=1.5, in_dtype=in_dtype, out_dtype=out_dtype)
    D, rc = _run_host(A, B, C, M, N, K, **kw)
    assert rc == 0
    ref, bound = H.oracle_full(A, B, C, M, N, K, **kw)
    H.assert_close(D.double().numpy(), ref, bound, out_dtype, "gemm_host %s->%s" % (in_dtype, out_dtype))


def test_small_and_k_zero():
    M, N, K = 16, 8, 16
    A = H.int_matrix((M, K), -8, 8, "f16", 31)
    B = H.int_matrix((K, N), -8, 8, "f16", 32)
    D, rc = _run_host(A, B, None, M, N, K)
    assert rc == 0
    ref, _ = H.oracle_full(A, B, None, M, N, K)
    H.assert_exact(D.numpy(), ref, "gemm_host single atom")
    C = H.int_matrix((70, 88), -50, 50, "f32", 33)
    D, rc = _run_host(None, None, C, 70, 88, 0, alpha=2.0, beta=-1.0)
    assert rc == 0
    H.assert_exact(D.numpy(), -C.double().numpy(), "gemm_host K = 0")


def test_back_to_back_calls_on_one_stream():
    """Consecutive calls reuse the staging buffers; each result must be its own."""
    M, N, K = 2048, 256, 192
    s = torch.cuda.Stream()
    outs, refs, keep = [], [], []
    for i in range(4):
        A = H.int_matrix((M, K), -8, 8, "bf16", 40 + i)
        B = H.int_matrix((K, N), -8, 8, "bf16", 50 + i)
        hA, _ = _host(A, True)
        hB, _ = _host(B, True)
        hD, _ = _host(torch.full((M, N), float("nan")), True)
        keep += [hA, hB]
        rc = binding.gemm_host(hD, hA, hB, None, M, N, K, K, N, N, N, 0, 0, 1.0, 0.0, 1, 2, s)
        assert rc == 0
        outs.append(hD)
        refs.append(H.oracle_full(A, B, None, M, N, K, in_dtype="bf16")[0])
    s.synchronize()
    for i in range(4):
        H.assert_exact(outs[i].numpy(), refs[i], "call %d" % i)


def test_host_alias_rejected():
    buf = torch.zeros((64, 64), dtype=torch.float32).pin_memory()
    A = torch.zeros((64, 64), dtype=torch.float16).pin_memory()
    # D overlapping B (same host buffer viewed twice)
    rc = binding.gemm_host(buf, A, buf, None, 64, 64, 64, 64, 128, 64, 64, 0, 0, 1.0, 0.0, 0, 2, None)
    assert rc == -4


@pytest.mark.parametrize("transB", [0, 1])
@pytest.mark.parametrize("in_dtype", ["f16", "e4m3"])
def test_first_panel_in_column_blocks(transB, in_dtype):
    """N >= 1024: the first row panel is computed and copied out in column
    blocks (a ragged last one here) while the rest of B is still arriving."""
    M, N, K = 2300, 1100, 200
    seed = 61 + transB + 2 * (in_dtype == "e4m3")
    A = H.int_matrix((M, K), -8, 8, in_dtype, seed)
    B = H.int_matrix((N, K) if transB else (K, N), -8, 8, in_dtype, seed + 1)
    C = H.int_matrix((M, N), -50, 50, "f32", seed + 2)
    kw = dict(transB=transB, beta=1.0, in_dtype=in_dtype)
    D, rc = _run_host(A, B, C, M, N, K, pad=5, **kw)
    assert rc == 0
    ref, _ = H.oracle_full(A, B, C, M, N, K, **kw)
    H.assert_exact(D.numpy(), ref, "column blocks transB=%d %s" % (transB, in_dtype))
