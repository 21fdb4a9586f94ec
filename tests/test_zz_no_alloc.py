"""gemm_noalloc(): the allocation-free entry point, against gemm().

Some callers cannot let a library allocate device memory: they own the
device's memory through their own pool or budget, or they run where CUDA
allocation calls are not allowed.  gemm_noalloc() keeps its kernel's only
scratch, the 16-byte status record, in a fixed static array instead of a
cudaMalloc'd block.  The tests here:

- call it through the C ABI twice in a row for each problem and compare
  both results with gemm()'s on the same inputs, within the parity
  tolerance the other tests use (in this pytest process, after the other
  test files, so gemm() has set the device up long before);
- run it in a fresh interpreter before any gemm() call, so that its own
  one-time set-up is what runs, check the result against the oracle, and
  count with a CUPTI callback every allocation call that reaches the CUDA
  driver while it runs: none (gemm()'s first call, made afterwards as a
  control, is seen allocating its status record);
- make a pipeline wait run out inside a gemm_noalloc() launch (a host-set
  test hook that leaves one stage unfilled: no fault) and check that
  gemm_poll_device_error() reports it, clears it, and that the next call
  is bit-exact.

The file name makes pytest collect it last.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from dense_tensor_core_02_gb300 import binding
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROBLEMS = [
    # (M, N, K, in, out, transA, transB, alpha, beta)
    (512, 512, 512, "f16", "f32", 0, 0, 1.5, 0.5),
    (1000, 1000, 1000, "f16", "f32", 0, 0, 1.0, 0.0),
    (768, 520, 392, "bf16", "f32", 1, 1, -0.75, 1.0),
    (264, 392, 200, "f16", "bf16", 0, 1, 1.0, 0.0),
    (96, 64, 0, "f16", "f32", 0, 0, 2.0, 0.5),
    (200, 136, 101, "f16", "f32", 0, 1, 1.0, 0.5),   # lda = ldb = 101: the mma.sync kernel
    (24, 16, 24, "bf16", "f16", 1, 0, 0.5, 0.0),      # tiny: the mma.sync route's atom kernel
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


# ---------------------------------------------------------------------------
# A fresh process: gemm_noalloc() before any gemm().  The child holds its
# buffers through the CUDA runtime's shared library (not torch), and counts
# every device-memory allocation call that reaches the CUDA driver with a
# CUPTI callback (tests/alloc_counter.c, loaded before any CUDA call), so
# that the library's statically linked runtime is seen too.  gemm()'s first
# call, which allocates its status record, is the control that shows the
# counter sees the library's allocations.

_CHILD = r"""
import ctypes, json, os, sys
import numpy as np
sys.path.insert(0, os.environ["REPO_ROOT"])
out = {}
counter = None
if os.environ.get("ALLOC_COUNTER"):
    counter = ctypes.CDLL(os.environ["ALLOC_COUNTER"])
    counter.alloc_counter_allocs.restype = ctypes.c_long
    counter.alloc_counter_frees.restype = ctypes.c_long
    out["counter_rc"] = counter.alloc_counter_start()
from dense_tensor_core_02_gb300 import binding

def counts():
    if counter is None or out.get("counter_rc"):
        return None
    return [counter.alloc_counter_allocs(), counter.alloc_counter_frees()]

def cudart():
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    for name in (os.path.join(home, "lib64", "libcudart.so"), "libcudart.so.13", "libcudart.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            pass
    raise RuntimeError("the CUDA runtime library was not found")

rt = cudart()
rt.cudaMalloc.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t]
rt.cudaMemcpy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int]
H2D, D2H = 1, 2

def check(rc, what):
    if rc != 0:
        raise RuntimeError("%s: CUDA error %d" % (what, rc))

def device_copy(host):
    p = ctypes.c_void_p()
    check(rt.cudaMalloc(ctypes.byref(p), host.nbytes), "cudaMalloc")
    check(rt.cudaMemcpy(p, host.ctypes.data, host.nbytes, H2D), "cudaMemcpy H2D")
    return p.value

check(rt.cudaSetDevice(0), "cudaSetDevice")
args = json.loads(sys.argv[1])
M, N, K = args["M"], args["N"], args["K"]
A = np.load(args["A"]); B = np.load(args["B"]); C = np.load(args["C"])
dA, dB, dC = device_copy(A), device_copy(B), device_copy(C)
D_init = np.full((M, N), np.nan, dtype=np.float32)
dDs = [device_copy(D_init) for _ in range(4)]
check(rt.cudaDeviceSynchronize(), "cudaDeviceSynchronize")

# three gemm_noalloc() calls and a poll, before any gemm(); allocation
# calls counted from just before the first to just after the poll
out["counts_before"] = counts()
out["rc"] = []
for dD in dDs[:3]:
    out["rc"].append(binding.gemm_noalloc(
        dD, dA, dB, dC, M, N, K, K, N, N, N, 0, 0, 1.0, 1.0, binding.F16, binding.F32, 0))
out["poll"] = binding.gemm_poll_device_error(0)[0]
out["counts_after"] = counts()
for i, dD in enumerate(dDs[:3]):
    D = np.empty((M, N), dtype=np.float32)
    check(rt.cudaMemcpy(D.ctypes.data, dD, D.nbytes, D2H), "cudaMemcpy D2H")
    np.save(os.path.join(args["out"], "D%d.npy" % i), D)
# the control: gemm()'s first call on the device allocates its status record
out["gemm_rc"] = binding.gemm(dDs[3], dA, dB, dC, M, N, K, K, N, N, N, 0, 0, 1.0, 1.0, binding.F16,
                              binding.F32, 0)
check(rt.cudaDeviceSynchronize(), "cudaDeviceSynchronize")
out["counts_after_gemm"] = counts()
print(json.dumps(out))
"""

_FRESH_SHAPE = (384, 520, 264)


@pytest.fixture(scope="module")
def fresh_process(tmp_path_factory):
    """Runs the child once: gemm_noalloc() three times in a fresh
    interpreter, then the gemm() control.  Returns (report, integer inputs,
    output directory)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tmp = tmp_path_factory.mktemp("noalloc_fresh")
    M, N, K = _FRESH_SHAPE
    A = H.int_matrix((M, K), -4, 4, "f16", 81)
    B = H.int_matrix((K, N), -4, 4, "f16", 82)
    C = H.int_matrix((M, N), -50, 50, "f32", 83)
    paths = {}
    for name, x in (("A", A.view(torch.int16)), ("B", B.view(torch.int16)), ("C", C)):
        paths[name] = str(tmp / ("%s.npy" % name))
        np.save(paths[name], x.numpy())
    env = dict(os.environ, REPO_ROOT=ROOT)
    for k in ("GEMM_TEST_SKIP_FIRST_STAGE", "GEMM_PATH", "GEMM_VARIANT", "ALLOC_COUNTER"):
        env.pop(k, None)
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    counter = str(tmp / "liballoc_counter.so")
    build = subprocess.run(["gcc", "-shared", "-fPIC", "-O2", "-std=c99", "-I" + os.path.join(cuda, "include"),
                            "-o", counter, os.path.join(ROOT, "tests", "alloc_counter.c"),
                            "-L" + os.path.join(cuda, "lib64"), "-lcupti",
                            "-Wl,-rpath," + os.path.join(cuda, "lib64")], capture_output=True, text=True)
    if build.returncode == 0:
        env["ALLOC_COUNTER"] = counter
    proc = subprocess.run([sys.executable, "-c", _CHILD, json.dumps(dict(M=M, N=N, K=K, out=str(tmp), **paths))],
                          env=env, capture_output=True, text=True, timeout=300)
    assert proc.returncode == 0, proc.stderr[-3000:]
    report = json.loads(proc.stdout.strip().splitlines()[-1])
    report["counter_build"] = build.returncode == 0 or build.stderr[-500:]
    return report, (A, B, C), tmp


def test_noalloc_first_in_fresh_process(fresh_process):
    """In a fresh interpreter, gemm_noalloc() runs before any gemm(): its own
    one-time set-up runs, the poll reads its record without creating
    gemm()'s, and the three results are the oracle's bit for bit (integer
    inputs)."""
    report, (A, B, C), tmp = fresh_process
    assert report["rc"] == [0, 0, 0], report
    assert report["poll"] == 0 and report["gemm_rc"] == 0, report
    M, N, K = _FRESH_SHAPE
    want, _ = H.oracle_full(A, B, C, M, N, K, beta=1.0)
    for i in range(3):
        H.assert_exact(np.load(str(tmp / ("D%d.npy" % i))), want, "fresh-process gemm_noalloc call %d" % i)


def test_noalloc_makes_no_allocation_call(fresh_process):
    """CUPTI sees no device-memory allocation or release call from the first
    gemm_noalloc() call (with its set-up) through the third and the poll,
    and does see the one gemm()'s first call makes."""
    report, _, _ = fresh_process
    if report["counter_build"] is not True:
        pytest.skip("the CUPTI allocation counter did not build: %s" % report["counter_build"])
    if report.get("counter_rc"):
        pytest.skip("CUPTI refused the subscription (CUptiResult %d)" % report["counter_rc"])
    before, after, control = report["counts_before"], report["counts_after"], report["counts_after_gemm"]
    assert after == before, "gemm_noalloc() made allocation / release calls: %s -> %s" % (before, after)
    assert control[0] > after[0], "the counter did not see gemm()'s first allocation: %s" % report


def test_noalloc_wait_bound_reported_and_cleared():
    """A stage that is never filled (test hook) makes a wait inside a
    gemm_noalloc() launch run out: gemm_poll_device_error() reports the
    timeout from the static record and clears it, and the next call is
    bit-exact."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    M, N, K = 256, 256, 512
    dev = torch.device("cuda", 0)
    A = H.int_matrix((M, K), -4, 4, "f16", 91)
    B = H.int_matrix((K, N), -4, 4, "f16", 92)
    Ad, Bd = A.to(dev), B.to(dev)
    assert H.poll()[0] == 0
    D = torch.full((M, N), float("nan"), device=dev)
    with H.env(GEMM_TEST_SKIP_FIRST_STAGE="1", GEMM_WAIT_TIMEOUT_NS="300000000", GEMM_PATH="tcgen05"):
        assert _call(binding.gemm_noalloc, D, Ad, Bd, None, M, N, K, "f16", "f32", 0, 0, 1.0, 0.0) == 0
    status, info = H.poll()
    assert status == binding.GEMM_ERR_DEVICE_TIMEOUT, (status, info)
    assert info[0] == binding.GEMM_ERR_DEVICE_TIMEOUT and info[2] in (1, 2, 3, 4, 5, 6), info
    assert H.poll() == (0, [0, 0, 0, 0])      # cleared by the first poll
    want, _ = H.oracle_full(A, B, None, M, N, K)
    for i in range(2):
        D = torch.full((M, N), float("nan"), device=dev)
        assert _call(binding.gemm_noalloc, D, Ad, Bd, None, M, N, K, "f16", "f32", 0, 0, 1.0, 0.0) == 0
        assert H.poll()[0] == 0
        H.assert_exact(D.cpu().numpy(), want, "gemm_noalloc after the timeout, call %d" % (i + 1))


def test_both_records_reported_one_per_poll():
    """A timeout in gemm() and one in gemm_noalloc(), both unpolled: the
    first poll reports one, the second the other, the third finds none."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    M, N, K = 256, 256, 512
    dev = torch.device("cuda", 0)
    Ad = H.int_matrix((M, K), -4, 4, "f16", 93).to(dev)
    Bd = H.int_matrix((K, N), -4, 4, "f16", 94).to(dev)
    assert H.poll()[0] == 0
    D = torch.empty((M, N), device=dev)
    with H.env(GEMM_TEST_SKIP_FIRST_STAGE="1", GEMM_WAIT_TIMEOUT_NS="300000000", GEMM_PATH="tcgen05"):
        assert _call(binding.gemm, D, Ad, Bd, None, M, N, K, "f16", "f32", 0, 0, 1.0, 0.0) == 0
        assert _call(binding.gemm_noalloc, D, Ad, Bd, None, M, N, K, "f16", "f32", 0, 0, 1.0, 0.0) == 0
    assert H.poll()[0] == binding.GEMM_ERR_DEVICE_TIMEOUT
    assert H.poll()[0] == binding.GEMM_ERR_DEVICE_TIMEOUT
    assert H.poll()[0] == 0


_CHILD_RETRY = r"""
import json, os, sys
sys.path.insert(0, os.environ["REPO_ROOT"])
import torch
from dense_tensor_core_02_gb300 import binding
M, N, K = 256, 264, 192
g = torch.Generator().manual_seed(5)
A = torch.randint(-4, 5, (M, K), generator=g).half().cuda()
B = torch.randint(-4, 5, (K, N), generator=g).half().cuda()
out = {}
def run(fn):
    D = torch.full((M, N), float("nan"), device="cuda")
    rc = fn(D, A, B, None, M, N, K, K, N, N, N, 0, 0, 1.0, 0.0, binding.F16, binding.F32, None)
    torch.cuda.synchronize()
    return rc, D
want = (A.float().cpu() @ B.float().cpu())
for name, fn in (("noalloc", binding.gemm_noalloc), ("gemm", binding.gemm)):
    os.environ["GEMM_TEST_FAIL_SETUP"] = "1"
    out[name + "_failed"] = run(fn)[0]
    del os.environ["GEMM_TEST_FAIL_SETUP"]
    rc, D = run(fn)
    out[name + "_retried"] = rc
    out[name + "_exact"] = bool(torch.equal(D.cpu(), want))
out["poll"] = binding.gemm_poll_device_error()[0]
print(json.dumps(out))
"""


def test_failed_setup_is_retried():
    """A device set-up that fails (host test hook, before any CUDA call) is
    reported by that call and not remembered: the next call on the device
    sets up and computes the exact result.  For gemm_noalloc() and gemm(),
    in a fresh interpreter where neither has set the device up."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, REPO_ROOT=ROOT)
    env.pop("GEMM_TEST_FAIL_SETUP", None)
    proc = subprocess.run([sys.executable, "-c", _CHILD_RETRY], env=env, capture_output=True, text=True,
                          timeout=300)
    assert proc.returncode == 0, proc.stderr[-3000:]
    out = json.loads(proc.stdout.strip().splitlines()[-1])
    for name in ("noalloc", "gemm"):
        assert out[name + "_failed"] == -7, out            # GEMM_ERR_CUDA, nothing enqueued
        assert out[name + "_retried"] == 0 and out[name + "_exact"], out
    assert out["poll"] == 0, out
