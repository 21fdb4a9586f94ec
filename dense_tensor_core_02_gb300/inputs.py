"""Seeded synthetic inputs for the GEMM workloads.

This module only draws random numbers and lays them out; it holds none of
the product's arithmetic, so both the CUDA path (tests, benchmark) and the
CPU oracle can be fed from it.

Operand rounding follows the Phobos "@tensorcore" page, section "The
forms" (operands are rounded to f16 before the tensor cores see them):
values are drawn in fp32 and rounded once, round-to-nearest-even, by
``Tensor.half()`` / ``Tensor.bfloat16()`` (``Tensor.to(torch.float8_*)``,
saturating to the largest finite value, for the 8-bit operands).  Storage is row-major; A is
stored [M, K] (or [K, M] when transposed), B [K, N] (or [N, K]), C and D
[M, N].
"""
from __future__ import annotations

import dataclasses
import math

import torch

_TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32,
                "e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
_ELEM_BYTES = {"f16": 2, "bf16": 2, "f32": 4, "e4m3": 1, "e5m2": 1, "e2m1": 0.5}


@dataclasses.dataclass(frozen=True)
class GemmCase:
    """One synthetic GEMM workload: shapes, value distributions, scalars."""
    name: str
    M: int
    N: int
    K: int
    in_dtype: str = "f16"          # dtype of A and B ("e2m1": packed fp4, uniform random codes)
    out_dtype: str = "f32"         # dtype of C and D
    dist: str = "normal"           # "normal" (mean 0, std) or "uniform" on [-1, 1]
    std: float = 1.0
    transA: int = 0
    transB: int = 0
    alpha: float = 1.0
    beta: float = 0.0
    c_dist: str = "normal"         # distribution of C when beta != 0
    seed: int = 0
    mx: bool = False               # MX block-scaled operands (UE8M0 scale per 32 K elements)
    sf_lo: int = 120               # scale bytes uniform on [sf_lo, sf_hi] (2^(e - 127))
    sf_hi: int = 134

    @property
    def a_shape(self):
        return (self.K, self.M) if self.transA else (self.M, self.K)

    @property
    def b_shape(self):
        return (self.N, self.K) if self.transB else (self.K, self.N)

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def algorithmic_bytes(self) -> int:
        """Each operand read once, C read once when beta != 0, D written once."""
        isz = _ELEM_BYTES[self.in_dtype]
        osz = _ELEM_BYTES[self.out_dtype]
        scale_bytes = (self.M + self.N) * ((self.K + 31) // 32) if self.mx else 0
        return int(isz * (self.M * self.K + self.K * self.N) + osz * self.M * self.N * (1 + (self.beta != 0)) +
                   scale_bytes)


def _draw(gen, shape, dist, std):
    if dist == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    if dist == "normal":
        x = torch.randn(shape, generator=gen, dtype=torch.float32)
        return x * std if std != 1.0 else x
    raise ValueError(dist)


def packed_fp4(gen, shape):
    """Uniform random E2M1 codes for a row-major [rows, cols] operand (cols
    even), packed two to a byte, even columns in the low nibble: uint8
    [rows, cols / 2]."""
    rows, cols = shape
    codes = torch.randint(0, 16, (rows, cols), generator=gen, dtype=torch.int32)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).to(torch.uint8)


def make_inputs(case: GemmCase):
    """CPU tensors (A, B, C) for ``case``; C is None when beta == 0.

    The generator is ``torch.Generator().manual_seed(case.seed)``; A, B
    and C are drawn from it in that order.  Packed E2M1 operands are uint8
    tensors of uniform random codes (``packed_fp4``).
    """
    gen = torch.Generator().manual_seed(case.seed)
    if case.in_dtype == "e2m1":
        A = packed_fp4(gen, case.a_shape)
        B = packed_fp4(gen, case.b_shape)
    else:
        dt = _TORCH_DTYPE[case.in_dtype]
        A = _draw(gen, case.a_shape, case.dist, case.std).to(dt)
        B = _draw(gen, case.b_shape, case.dist, case.std).to(dt)
    C = None
    if case.beta != 0.0:
        C = _draw(gen, (case.M, case.N), case.c_dist, 1.0).to(_TORCH_DTYPE[case.out_dtype])
    return A, B, C


def make_scales(case: GemmCase):
    """CPU uint8 tensors (SFA [M, ceil(K/32)], SFB [N, ceil(K/32)]) of MX
    scale bytes for ``case``, uniform on [sf_lo, sf_hi], drawn in that order
    from ``torch.Generator().manual_seed(case.seed + 1000000)``."""
    gen = torch.Generator().manual_seed(case.seed + 1000000)
    kb = (case.K + 31) // 32
    SFA = torch.randint(case.sf_lo, case.sf_hi + 1, (case.M, kb), generator=gen, dtype=torch.int32)
    SFB = torch.randint(case.sf_lo, case.sf_hi + 1, (case.N, kb), generator=gen, dtype=torch.int32)
    return SFA.to(torch.uint8), SFB.to(torch.uint8)


def integer_matrix(shape, lo, hi, seed, dtype="f16"):
    """Integer-valued matrix with entries uniform on [lo, hi], seeded."""
    gen = torch.Generator().manual_seed(seed)
    x = torch.randint(lo, hi + 1, shape, generator=gen, dtype=torch.int32)
    return x.float().to(_TORCH_DTYPE[dtype])


# The workloads the benchmark and the parity tests run, in a fixed order; the
# seed of the i-th entry (1-based) is 1000 + i.
def _cases():
    k8192 = 8192
    rows = [
        # single m16n8k16 atom: TIRx "gemm" page, "Demonstration program"
        GemmCase("single_atom_16x8x16_f16", 16, 8, 16, "f16", dist="uniform"),
        GemmCase("gemm_512_f16_alpha1.5_beta0.5", 512, 512, 512, "f16", dist="normal",
                 alpha=1.5, beta=0.5, c_dist="normal"),
        GemmCase("gemm_4096_bf16_transB_beta1", 4096, 4096, 4096, "bf16", dist="uniform",
                 transB=1, alpha=1.0, beta=1.0, c_dist="uniform"),
        GemmCase("gemm_8192_f16", k8192, k8192, k8192, "f16", dist="normal",
                 std=1.0 / math.sqrt(k8192)),
        GemmCase("sweep_8192x8192_K256_f16", 8192, 8192, 256, "f16"),
        GemmCase("sweep_8192x8192_K1024_f16", 8192, 8192, 1024, "f16"),
        GemmCase("sweep_8192x8192_K4096_f16", 8192, 8192, 4096, "f16"),
        GemmCase("sweep_8192x8192_K16384_f16", 8192, 8192, 16384, "f16"),
        GemmCase("tall_skinny_32768x256x4096_f16", 32768, 256, 4096, "f16"),
        GemmCase("unaligned_1000_f16", 1000, 1000, 1000, "f16"),
        # 8-bit operands (the tcgen05 path's fp8 precisions, TIRx gemm guide
        # section 七), K-major as the kind::f8f6f4 kernel reads them in place
        GemmCase("gemm_8192_e4m3_transB", k8192, k8192, k8192, "e4m3", transB=1),
        GemmCase("gemm_4096_e5m2_transB_beta1", 4096, 4096, 4096, "e5m2", dist="uniform",
                 transB=1, alpha=1.0, beta=1.0, c_dist="uniform"),
        # MX block-scaled 8-bit operands (the SFA / SFB block scaling of the
        # same section), scales 2^-7 .. 2^7
        GemmCase("gemm_8192_mxe4m3_transB", k8192, k8192, k8192, "e4m3", transB=1, mx=True),
        GemmCase("gemm_4096_mxe5m2_transB_beta1", 4096, 4096, 4096, "e5m2", dist="uniform",
                 transB=1, alpha=1.0, beta=1.0, c_dist="uniform", mx=True),
        # packed fp4 (E2M1, the guide's other gemm_async precision), block-scaled
        GemmCase("gemm_8192_mxe2m1_transB", k8192, k8192, k8192, "e2m1", transB=1, mx=True),
    ]
    return [dataclasses.replace(c, seed=1000 + i + 1) for i, c in enumerate(rows)]


CASES = _cases()
CASE_BY_NAME = {c.name: c for c in CASES}
HEADLINE = CASE_BY_NAME["gemm_8192_f16"]
