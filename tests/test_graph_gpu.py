"""gemm(), gemm_noalloc() and gemm_host() captured into CUDA graphs and
replayed, against the CPU oracle.  Inside a capture the library allocates
nothing: stream-K and the repacking route use only workspaces that earlier
calls on the stream created, else the call falls back to whole tiles /
the mma.sync kernel.  Replays read the buffers' current contents, so new
inputs copied into the same buffers give new, correct results.
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


def _problem(M, N, K, seed, dev):
    A = H.int_matrix((M, K), -8, 8, "f16", seed)
    B = H.int_matrix((K, N), -8, 8, "f16", seed + 1)
    return A, B, A.to(dev), B.to(dev), torch.empty((M, N), device=dev)


@pytest.mark.parametrize("warm", [True, False])
def test_captured_gemm_replays(warm):
    """A stream-K shape (forced fine split) and a narrow-tile shape in one
    graph.  Without a warm-up call on this stream the stream-K workspace does
    not exist yet, so the captured call plans whole tiles instead."""
    dev = torch.device("cuda", 0)
    s = torch.cuda.Stream()
    shapes = [(1024, 768, 2080), (300, 200, 136)]
    probs = [_problem(M, N, K, 10 * i + 1, dev) for i, (M, N, K) in enumerate(shapes)]
    binding.gemm(probs[0][4], probs[0][2], probs[0][3], None, 16, 8, 16, 2080, 768, 768, 768, 0, 0, 1.0, 0.0, 0,
                 2, s)   # the device's one-time set-up happens outside the capture
    s.synchronize()

    def calls():
        for (A, B, Ad, Bd, Dd), (M, N, K) in zip(probs, shapes):
            rc = binding.gemm(Dd, Ad, Bd, None, M, N, K, K, N, N, N, 0, 0, 1.0, 0.0, 0, 2, s)
            assert rc == 0

    with H.env(GEMM_SK_MIN_ITERS="1"):
        if warm:
            with torch.cuda.stream(s):
                calls()
            s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            calls()
    for rep in range(2):
        if rep == 1:   # new inputs in the same buffers
            for i, (A, B, Ad, Bd, Dd) in enumerate(probs):
                A2 = H.int_matrix(tuple(A.shape), -8, 8, "f16", 100 + i)
                Ad.copy_(A2)
                probs[i] = (A2, B, Ad, Bd, Dd)
        for (_, _, _, _, Dd) in probs:
            Dd.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for (A, B, _, _, Dd), (M, N, K) in zip(probs, shapes):
            ref, _ = H.oracle_full(A, B, None, M, N, K)
            H.assert_exact(Dd.cpu().numpy(), ref, "replay %d %s" % (rep, (M, N, K)))


def test_replay_after_the_workspace_grew():
    """A graph captured with the stream-K workspace of one size, then an
    eager call on the same stream that needs a larger one: the library keeps
    the captured buffer (it does not free what a graph refers to), so later
    replays still compute into valid memory and give exact results."""
    dev = torch.device("cuda", 0)
    s = torch.cuda.Stream()
    small, large = (256, 256, 1024), (1024, 1024, 2048)   # stream-K workspaces of 34 and 101 MB
    A, B, Ad, Bd, Dd = _problem(*small, 31, dev)
    A2, B2, Ad2, Bd2, Dd2 = _problem(*large, 41, dev)
    sms = torch.cuda.get_device_properties(0).multi_processor_count

    def call(prob, shape):
        M, N, K = shape
        assert binding.gemm(prob[2], prob[0], prob[1], None, M, N, K, K, N, N, N, 0, 0, 1.0, 0.0, 0, 2, s) == 0

    with H.env(GEMM_SK_MIN_ITERS="1"):
        p_small, p_large = binding.gemm_plan(*small, sms), binding.gemm_plan(*large, sms)
        assert 0 < p_small["workspace_bytes"] < p_large["workspace_bytes"]
        with torch.cuda.stream(s):
            call((Ad, Bd, Dd), small)   # creates the workspace at the small size
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            call((Ad, Bd, Dd), small)
        with torch.cuda.stream(s):
            call((Ad2, Bd2, Dd2), large)   # grows the workspace
        s.synchronize()
        for _ in range(2):
            Dd.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            ref, _ = H.oracle_full(A, B, None, *small)
            H.assert_exact(Dd.cpu().numpy(), ref, "replay after growth")
    rows = list(range(0, large[0], 61))
    ref2, _ = H.oracle_at(A2, B2, None, *large, [r for r in rows for _ in range(large[1])],
                          [c for _ in rows for c in range(large[1])])
    H.assert_exact(Dd2.cpu().numpy()[rows].ravel(), ref2, "the eager call that grew the workspace")


def test_captured_misaligned_call_without_workspace():
    """A layout off the 16-byte grid, large enough for the repacking route,
    captured on a fresh stream: no repack workspace exists, so the captured
    call runs the mma.sync kernel instead."""
    dev = torch.device("cuda", 0)
    s = torch.cuda.Stream()
    M, N, K = 520, 392, 1001
    A = H.int_matrix((M, K), -8, 8, "bf16", 41)
    B = H.int_matrix((K, N), -8, 8, "bf16", 42)
    Ad, Bd, Dd = A.to(dev), B.to(dev), torch.empty((M, N), device=dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        assert binding.gemm(Dd, Ad, Bd, None, M, N, K, K, N, N, N, 0, 0, 1.0, 0.0, 1, 2, s) == 0
    Dd.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    ref, _ = H.oracle_full(A, B, None, M, N, K, in_dtype="bf16")
    H.assert_exact(Dd.cpu().numpy(), ref, "captured misaligned")


def test_captured_noalloc_and_host():
    dev = torch.device("cuda", 0)
    s = torch.cuda.Stream()
    M, N, K = 2048, 256, 192
    A = H.int_matrix((M, K), -8, 8, "f16", 51)
    B = H.int_matrix((K, N), -8, 8, "f16", 52)
    Ad, Bd, Dd = A.to(dev), B.to(dev), torch.empty((M, N), device=dev)
    hA, hB = A.pin_memory(), B.pin_memory()
    hD = torch.empty((M, N)).pin_memory()
    # warm-up outside the capture: one-time set-up and gemm_host staging
    assert binding.gemm_noalloc(Dd, Ad, Bd, None, M, N, K, K, N, N, N, 0, 0, 1.0, 0.0, 0, 2, s) == 0
    assert binding.gemm_host(hD, hA, hB, None, M, N, K, K, N, N, N, 0, 0, 1.0, 0.0, 0, 2, s) == 0
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        assert binding.gemm_noalloc(Dd, Ad, Bd, None, M, N, K, K, N, N, N, 0, 0, 2.0, 0.0, 0, 2, s) == 0
        assert binding.gemm_host(hD, hA, hB, None, M, N, K, K, N, N, N, 0, 0, -1.0, 0.0, 0, 2, s) == 0
    Dd.fill_(float("nan"))
    hD.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    ref, _ = H.oracle_full(A, B, None, M, N, K)
    H.assert_exact(Dd.cpu().numpy(), 2.0 * ref, "captured no-alloc")
    H.assert_exact(hD.numpy(), -ref, "captured gemm_host")


@pytest.mark.parametrize("dtype", ["e4m3", "e2m1"])
def test_captured_gemm_mx_replays(dtype):
    """gemm_mx in a graph, after a call of the same size on the stream made
    its workspaces (rearranged scales; for 4-bit rows off TMA's grid, the
    padded operand copies, whose memset and copies are captured too).
    Replays with new operands and new scales in the same buffers."""
    import oracle.oracle as oracle
    from tests.test_mx_gpu import fp4_matrix, scales
    dev = torch.device("cuda", 0)
    s = torch.cuda.Stream()
    M, N, K = 512, 384, (1000 if dtype == "e2m1" else 1024)
    epu = 2 if dtype == "e2m1" else 1

    def operands(seed):
        if dtype == "e2m1":
            return fp4_matrix(M, K, seed), fp4_matrix(N, K, seed + 1)
        return H.int_matrix((M, K), -8, 8, dtype, seed), H.int_matrix((N, K), -8, 8, dtype, seed + 1)

    A, B = operands(201)
    SFA, SFB = scales(M, K, 126, 128, 203), scales(N, K, 126, 128, 204)
    Ad, Bd, sa, sb = A.to(dev), B.to(dev), SFA.to(dev), SFB.to(dev)
    Dd = torch.empty((M, N), device=dev)

    def call():
        rc = binding.gemm_mx(Dd, Ad, Bd, None, sa, sb, M, N, K, Ad.stride(0) * epu, Bd.stride(0) * epu, N, N,
                             sa.stride(0), sb.stride(0), 0, 1, 1.0, 0.0, H.CODE[dtype], H.CODE["f32"], s)
        assert rc == 0

    with torch.cuda.stream(s):
        call()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    for rep in range(2):
        if rep == 1:
            A, B = operands(301)
            SFA = scales(M, K, 126, 128, 303)
            Ad.copy_(A)
            Bd.copy_(B)
            sa.copy_(SFA)
        Dd.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ref, _ = oracle.gemm(A, B, None, M, N, K, transB=1, in_dtype=H.CODE[dtype], threads=H.ORACLE_THREADS,
                             sfa=SFA.numpy(), sfb=SFB.numpy())
        H.assert_exact(Dd.cpu().numpy(), ref, "gemm_mx replay %d (%s)" % (rep, dtype))


def test_captured_gemm_mx_without_workspace_is_refused():
    """On a stream with no earlier gemm_mx call the scale workspace does not
    exist, and a capture may not allocate it: the call is refused before it
    enqueues anything (GEMM_ERR_CUDA) and the capture stays valid."""
    dev = torch.device("cuda", 0)
    s = torch.cuda.Stream()
    M, N, K = 256, 192, 256
    A = H.int_matrix((M, K), -8, 8, "e4m3", 211).to(dev)
    B = H.int_matrix((N, K), -8, 8, "e4m3", 212).to(dev)
    sa = torch.full((M, K // 32), 127, dtype=torch.uint8, device=dev)
    sb = torch.full((N, K // 32), 127, dtype=torch.uint8, device=dev)
    Dd = torch.full((M, N), 3.0, device=dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        rc = binding.gemm_mx(Dd, A, B, None, sa, sb, M, N, K, K, K, N, N, K // 32, K // 32, 0, 1, 1.0, 0.0,
                             H.CODE["e4m3"], H.CODE["f32"], s)
        Dd.add_(1.0)
    assert rc == -7
    g.replay()
    torch.cuda.synchronize()
    assert bool((Dd == 4.0).all()), "the refused call must not have written D"
