"""Back-to-back dependent calls with no synchronisation between them: each
product's D is the next product's A.  Every kernel is launched with
programmatic stream serialisation and must wait for its predecessor before
reading its operands; a torch kernel writing A just before the first call
checks the same against a foreign predecessor.  Integer-valued data, exact.
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


def _two_per_column(K, N, rng):
    """K x N with two entries of +-1 per column: each link at most doubles
    the magnitudes, so the whole chain stays exact in fp16."""
    b = np.zeros((K, N), dtype=np.float32)
    for j in range(N):
        rows = rng.choice(K, size=2, replace=False)
        b[rows, j] = rng.choice([-1.0, 1.0], size=2)
    return torch.from_numpy(b).half()


# (rows M, then the K -> N widths of each link); the shapes take the pair,
# narrow and mma.sync routes in turn
CHAINS = [
    (1024, [64, 256, 512, 128, 64]),
    (300, [32, 16, 48, 24, 40]),
    (2048, [128, 1024, 64, 256, 128]),
]


@pytest.mark.parametrize("chain", CHAINS, ids=lambda c: "M%d" % c[0])
def test_chained_products_exact(chain):
    M, widths = chain
    dev = torch.device("cuda", 0)
    s = torch.cuda.Stream()
    rng = np.random.default_rng(M)
    Bs = [_two_per_column(widths[i], widths[i + 1], rng) for i in range(len(widths) - 1)]
    A0 = torch.from_numpy(rng.integers(-2, 3, size=(M, widths[0])).astype(np.float32)).half()
    Bd = [b.to(dev) for b in Bs]
    Ds = [torch.empty((M, w), dtype=torch.float16, device=dev) for w in widths[1:]]
    A0d = torch.zeros((M, widths[0]), dtype=torch.float16, device=dev)
    with torch.cuda.stream(s):
        A0d.copy_(A0.to(dev, non_blocking=False))   # a torch kernel just before the first product
        A0d.mul_(1.0)
        cur = A0d
        for b, D in zip(Bd, Ds):
            K, N = b.shape
            rc = binding.gemm(D, cur, b, None, M, N, K, K, N, N, N, 0, 0, 1.0, 0.0, 0, 0, s)   # f16 in, f16 out
            assert rc == 0
            cur = D
    s.synchronize()
    ref = A0.double().numpy()
    for b in Bs:
        ref = ref @ b.double().numpy()
    assert np.abs(ref).max() <= 2048, "the chain must stay exact in fp16"
    assert np.abs(ref).max() >= 8, "the chain must carry nontrivial values"
    H.assert_exact(cur.double().cpu().numpy(), ref, "chain M=%d" % M)
