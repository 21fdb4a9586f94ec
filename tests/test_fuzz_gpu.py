"""Seeded random sweep over the whole argument space, against the oracle:
sizes (including 1 and ragged edges), operand and output types, transpose
forms, alpha / beta, element offsets and padded or odd row strides, and the
three entry points (gemm, gemm_noalloc, gemm_host).  Every case takes
whichever kernel route the library chooses for it; integer-valued inputs
are compared bit for bit, random ones within the tolerance.  Cases that
gemm_noalloc() cannot take (8-bit operands that are not K-major or off the
16-byte grid) must be refused with GEMM_ERR_UNSUPPORTED_LAYOUT.
"""
import numpy as np
import pytest
import torch

from dense_tensor_core_02_gb300 import binding
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

IN = ["f16", "bf16", "e4m3", "e5m2"]
OUT = ["f32", "f16", "bf16"]
ISZ = {"f16": 2, "bf16": 2, "e4m3": 1, "e5m2": 1}
OSZ = {"f32": 4, "f16": 2, "bf16": 2}


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    yield
    rc, info = H.poll()
    assert rc == 0, ("device status after the module", rc, info)


def _case(seed):
    rng = np.random.default_rng(seed)
    pick = lambda xs: xs[int(rng.integers(len(xs)))]
    dims = [1, 7, 16, 33, 64, 100, 128, 129, 255, 256, 300, 513, 640]
    M, N, K = pick(dims), pick(dims), pick(dims + [0])
    ind, outd = pick(IN), pick(OUT)
    transA, transB = int(rng.integers(2)), int(rng.integers(2))
    beta = pick([0.0, 1.0, -0.5])
    alpha = pick([1.0, 1.0, 2.0, -0.75])
    exact = bool(rng.integers(2)) and alpha in (1.0, 2.0) and beta in (0.0, 1.0)
    layout = pick(["dense", "padded", "odd"])
    api = pick(["gemm", "gemm", "noalloc", "host"])
    return dict(M=M, N=N, K=K, ind=ind, outd=outd, transA=transA, transB=transB, alpha=alpha, beta=beta,
                exact=exact, layout=layout, api=api, seed=seed)


def _lds_offs(c, rng):
    M, N, K = c["M"], c["N"], c["K"]
    ca = M if c["transA"] else K
    cb = K if c["transB"] else N
    if c["layout"] == "dense":
        return (ca, cb, N, N), (0, 0, 0, 0)
    if c["layout"] == "padded":   # 16-byte multiples, aligned bases
        r = lambda x, e: -(-max(x, 1) // (16 // e)) * (16 // e) + 16 // e
        isz, osz = ISZ[c["ind"]], OSZ[c["outd"]]
        return (r(ca, isz), r(cb, isz), r(N, osz), r(N, osz)), (0, 0, 0, 0)
    odd = lambda x: x + 1 + int(rng.integers(3))
    return (odd(ca), odd(cb), odd(N), odd(N)), tuple(int(rng.integers(1, 4)) for _ in range(4))


def _run_host(A, B, C, c, lds):
    M, N, K = c["M"], c["N"], c["K"]

    def host(x, ld, dt):
        rows, cols = x.shape
        buf = torch.empty((rows, ld), dtype=H.TORCH[dt]).pin_memory()
        buf[:, :cols] = x
        return buf
    hA = host(A, lds[0], c["ind"]) if K else None
    hB = host(B, lds[1], c["ind"]) if K else None
    hC = host(C, lds[2], c["outd"]) if C is not None else None
    hD = host(torch.full((M, N), float("nan")).to(H.TORCH[c["outd"]]), lds[3], c["outd"])
    rc = binding.gemm_host(hD, hA, hB, hC, M, N, K, lds[0], lds[1], lds[2], lds[3], c["transA"], c["transB"],
                           c["alpha"], c["beta"], H.CODE[c["ind"]], H.CODE[c["outd"]], None)
    torch.cuda.synchronize()
    return hD[:, :N].clone(), rc


@pytest.mark.parametrize("seed", range(240))
def test_random_case(seed):
    c = _case(seed)
    rng = np.random.default_rng(1000 + seed)
    M, N, K = c["M"], c["N"], c["K"]
    a_shape = (K, M) if c["transA"] else (M, K)
    b_shape = (N, K) if c["transB"] else (K, N)
    if c["exact"]:
        A = H.int_matrix(a_shape, -8, 8, c["ind"], seed)
        B = H.int_matrix(b_shape, -8, 8, c["ind"], seed + 1)
        C = H.int_matrix((M, N), -50, 50, c["outd"], seed + 2) if c["beta"] else None
    else:
        A = H.normal_matrix(a_shape, c["ind"], seed)
        B = H.normal_matrix(b_shape, c["ind"], seed + 1)
        C = H.normal_matrix((M, N), c["outd"], seed + 2) if c["beta"] else None
    lds, offs = _lds_offs(c, rng)
    kw = dict(transA=c["transA"], transB=c["transB"], alpha=c["alpha"], beta=c["beta"], in_dtype=c["ind"],
              out_dtype=c["outd"])
    if c["api"] == "host":
        D, rc = _run_host(A, B, C, c, lds)
    else:
        fn = binding.gemm_noalloc if c["api"] == "noalloc" else binding.gemm
        D, _, rc = H.run_layout(A, B, C, M, N, K, offs=offs, lds=lds, fn=fn, **kw)
    f8 = c["ind"] in ("e4m3", "e5m2")
    if c["api"] == "noalloc" and f8 and K > 0:
        isz, osz = ISZ[c["ind"]], OSZ[c["outd"]]
        aligned = all((o * s) % 16 == 0 for o, s in zip(offs, (isz, isz, osz, osz))) and \
            (lds[0] * isz) % 16 == 0 and (lds[1] * isz) % 16 == 0 and (lds[3] * osz) % 16 == 0 and \
            (C is None or (lds[2] * osz) % 16 == 0)
        if c["transA"] or not c["transB"] or not aligned:
            assert rc == binding.GEMM_ERR_UNSUPPORTED_LAYOUT, (c, rc)
            return
    assert rc == 0, (c, rc)
    ref, bound = H.oracle_full(A if K else None, B if K else None, C, M, N, K, **kw)
    if c["exact"]:
        got = D.double().numpy()
        if c["outd"] == "f32":
            H.assert_exact(got, ref, str(c))
        else:   # integers up to |D| <= 2048 are exact in fp16; bf16 rounds above 256
            H.assert_close(got, ref, bound, c["outd"], str(c))
    else:
        H.assert_close(D.double().numpy(), ref, bound, c["outd"], str(c))
