"""gemm_noalloc(): the allocation-free entry point, against gemm().

Some callers cannot let a library allocate device memory (they own the
device's memory through their own pool, or run where allocation calls are
not allowed).  gemm_noalloc() keeps its kernel's scratch in a fixed static
array instead.  Here it is called through the C ABI twice in a row for each
problem and both results are compared with gemm()'s on the same inputs,
within the parity tolerance the other tests use.  gemm_noalloc() is called
first, so that in a fresh process its one-time per-device set-up runs too.

The file name makes pytest collect it last.
"""
import numpy as np
import pytest
import torch

from dense_tensor_core_02_gb300 import binding
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

PROBLEMS = [
    # (M, N, K, in, out, transA, transB, alpha, beta)
    (512, 512, 512, "f16", "f32", 0, 0, 1.5, 0.5),
    (1000, 1000, 1000, "f16", "f32", 0, 0, 1.0, 0.0),
    (768, 520, 392, "bf16", "f32", 1, 1, -0.75, 1.0),
    (264, 392, 200, "f16", "bf16", 0, 1, 1.0, 0.0),
    (96, 64, 0, "f16", "f32", 0, 0, 2.0, 0.5),
    (200, 136, 101, "f16", "f32", 0, 1, 1.0, 0.5),   # lda = ldb = 101: the mma.sync kernel
    (24, 16, 40, "bf16", "f16", 1, 0, 0.5, 0.0),      # tiny: the mma.sync kernel
]


def _call(fn, D, Ad, Bd, Cd, M, N, K, it, ot, ta, tb, alpha, beta):
    lda = Ad.stride(0) if Ad is not None else 0
    ldb = Bd.stride(0) if Bd is not None else 0
    ldc = Cd.stride(0) if Cd is not None else N
    return fn(D, Ad, Bd, Cd, M, N, K, lda, ldb, ldc, D.stride(0), ta, tb, alpha, beta, H.CODE[it], H.CODE[ot],
              None)


@pytest.mark.parametrize("prob", PROBLEMS, ids=lambda p: "%dx%dx%d_%s_%s_t%d%d" % p[:7])
def test_noalloc_matches_gemm_twice(prob):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    M, N, K, it, ot, ta, tb, alpha, beta = prob
    dev = torch.device("cuda", 0)
    seed = M + 3 * N + 7 * K
    A = H.normal_matrix((K, M) if ta else (M, K), it, seed) if K else None
    B = H.normal_matrix((N, K) if tb else (K, N), it, seed + 1) if K else None
    C = H.normal_matrix((M, N), ot, seed + 2) if beta else None
    Ad = A.to(dev) if A is not None else None
    Bd = B.to(dev) if B is not None else None
    Cd = C.to(dev) if C is not None else None

    outs = []
    for _ in range(2):                      # two calls in a row
        D = torch.full((M, N), float("nan"), dtype=H.TORCH[ot], device=dev)
        assert _call(binding.gemm_noalloc, D, Ad, Bd, Cd, M, N, K, it, ot, ta, tb, alpha, beta) == 0
        outs.append(D)
    ref = torch.full((M, N), float("nan"), dtype=H.TORCH[ot], device=dev)
    assert _call(binding.gemm, ref, Ad, Bd, Cd, M, N, K, it, ot, ta, tb, alpha, beta) == 0
    torch.cuda.synchronize()
    assert binding.gemm_poll_device_error()[0] == 0

    if K:
        _, bound = H.oracle_full(A, B, C, M, N, K, transA=ta, transB=tb, alpha=alpha, beta=beta,
                                 in_dtype=it, out_dtype=ot)
    else:
        bound = np.abs(beta * C.double().numpy())
    want = ref.double().cpu().numpy()
    assert np.isfinite(want).all()
    for i, D in enumerate(outs):
        got = D.double().cpu().numpy()
        H.assert_close(got, want, bound, ot, "gemm_noalloc call %d vs gemm" % (i + 1))


def test_noalloc_wave_fitted_tiles():
    """gemm_noalloc() on the 224-wide tiles (taken by force on this shape) gives
    the same bits as gemm() on integer inputs, and the oracle's."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    M, N, K = 1024, 1120, 1408
    dev = torch.device("cuda", 0)
    A = H.int_matrix((M, K), -4, 4, "bf16", 71)
    B = H.int_matrix((N, K), -4, 4, "bf16", 72)
    C = H.int_matrix((M, N), -50, 50, "f32", 73)
    Ad, Bd, Cd = A.to(dev), B.to(dev), C.to(dev)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    with H.env(GEMM_FIT_TILES="1", GEMM_VARIANT="pair", GEMM_PATH="tcgen05"):
        assert binding.gemm_plan_layout(M, N, K, 1, binding.BF16, binding.F32, sms)["tile_n"] == 224
        D = torch.full((M, N), float("nan"), device=dev)
        ref = torch.full((M, N), float("nan"), device=dev)
        assert _call(binding.gemm_noalloc, D, Ad, Bd, Cd, M, N, K, "bf16", "f32", 0, 1, 1.0, 1.0) == 0
        assert _call(binding.gemm, ref, Ad, Bd, Cd, M, N, K, "bf16", "f32", 0, 1, 1.0, 1.0) == 0
    torch.cuda.synchronize()
    assert binding.gemm_poll_device_error()[0] == 0
    assert torch.equal(D, ref)
    want, _ = H.oracle_full(A, B, C, M, N, K, transB=1, beta=1.0, in_dtype="bf16")
    H.assert_exact(D.cpu().numpy(), want, "gemm_noalloc on 224-wide tiles")
